"""The allocation-free decode entry point (pa_decode_attention_noalloc).

It serves callers that cannot give the library device memory: a host program
that reaches the GPU only through the C ABI, or a serving process whose
allocator already holds all device memory.  Instead of a caller workspace it
uses a fixed 32 MiB array inside the library, shared by every call.  These
tests check, through the C ABI, that two calls in a row give the same output
as the workspace-taking entry point (within the attention tolerance of the
other GPU tests), and that a problem too large for the array is refused.
The file is named to be collected last, and passes alone or after the rest.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_265_gb300 import pa
from paged_kv_cache_265_gb300 import workload as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from paged_kv_cache_265_gb300 import build

    build.build()
    import gpu_helpers

    pa.get_device_error(clear=True)
    return gpu_helpers


def test_noalloc_matches_workspace_entry_point_twice(gpu):
    G = gpu
    w = W.gqa_batch128()                       # long sequences: the scratch holds split-K partials
    need = pa.workspace_size(w.num_seqs, w.q_len, w.num_heads, w.head_dim, w.max_context_len)
    assert 0 < need <= pa.NOALLOC_WORKSPACE_BYTES
    step = G.GpuStep(w)
    step.append()
    ref = G.to_bits(step.attend().clone())
    outs = [torch.full_like(step.query, float("nan")) for _ in range(2)]
    torch.cuda.synchronize()
    for call in range(2):
        free_before = torch.cuda.mem_get_info()[0]
        pa.decode_attention_noalloc(outs[call], step.query, step.key_cache, step.value_cache, step.block_tables,
                                    step.context_lens, w.scale, w.max_context_len)
        torch.cuda.synchronize()
        if call == 1:   # the first call may load the library's kernels; the second allocates nothing
            assert torch.cuda.mem_get_info()[0] == free_before, "device memory changed during the call"
        got = G.to_bits(outs[call])
        G.compare(got, G.bits_to_f64(ref, w.dtype), w.dtype, f"noalloc call {call}")
        assert np.array_equal(got, ref), f"call {call} differs from the workspace entry point"
    assert pa.get_device_error(clear=True) == 0


def test_noalloc_multiquery_and_small_partitions(gpu):
    G = gpu
    w = W.shared_prefix_verify()               # 5 query rows per sequence, causal inside the chunk
    step = G.GpuStep(w, partition_size=256)
    step.append()
    ref = G.to_bits(step.attend().clone())
    for _ in range(2):
        out = torch.empty_like(step.query)
        pa.decode_attention_noalloc(out, step.query, step.key_cache, step.value_cache, step.block_tables,
                                    step.context_lens, w.scale, w.max_context_len, partition_size=256)
        torch.cuda.synchronize()
        got = G.to_bits(out)
        G.compare(got, G.bits_to_f64(ref, w.dtype), w.dtype, "noalloc multi-query")
        assert np.array_equal(got, ref)
    assert pa.get_device_error(clear=True) == 0


def test_noalloc_prefill_chunk_needs_no_scratch(gpu):
    """A chunk with >= 128 query rows per kv head runs on the tcgen05 kernel, which uses no
    scratch: the call is accepted even where a split of the same shape would not fit the array,
    and it matches the oracle."""
    G = gpu
    w = W.make_workload("noalloc_chunk", [600, 1400], num_heads=32, num_kv_heads=8, head_dim=128, q_len=64,
                        num_blocks=140, seed=43)
    step = G.GpuStep(w)
    step.append()
    torch.cuda.synchronize()
    for call in range(2):
        out = torch.full_like(step.query, float("nan"))
        pa.decode_attention_noalloc(out, step.query, step.key_cache, step.value_cache, step.block_tables,
                                    step.context_lens, w.scale, w.max_context_len)
        torch.cuda.synchronize()
        assert pa.last_partition_size() == 0          # the tcgen05 kernel, no split
        _, _, ref = G.oracle_step(w)
        G.compare(G.to_bits(out), ref, w.dtype, f"noalloc chunk call {call}")
    # a 512-row chunk per kv head over a 131072-token bound: a split layout of 256 partitions would
    # need far more than the array holds, the tcgen05 kernel needs none of it
    big = W.make_workload("noalloc_big_bound", [700], num_heads=32, num_kv_heads=8, head_dim=128, q_len=128,
                          num_blocks=60, seed=44, max_blocks_per_seq=8192)
    assert pa.workspace_size(1, 128, 32, 128, 131072) > pa.NOALLOC_WORKSPACE_BYTES
    bstep = G.GpuStep(big)
    bstep.append()
    out = torch.empty_like(bstep.query)
    pa.decode_attention_noalloc(out, bstep.query, bstep.key_cache, bstep.value_cache, bstep.block_tables,
                                bstep.context_lens, big.scale, 131072)
    torch.cuda.synchronize()
    _, _, ref = G.oracle_step(big)
    G.compare(G.to_bits(out), ref, big.dtype, "noalloc chunk with a large length bound")
    assert pa.get_device_error(clear=True) == 0


def test_noalloc_refuses_problems_beyond_its_scratch(gpu):
    # 256 sequences of up to 32768 tokens, 64 heads: about 0.5 GB of partials
    n, hq, hkv, d, max_len = 256, 64, 8, 128, 32768
    assert pa.workspace_size(n, 1, hq, d, max_len) > pa.NOALLOC_WORKSPACE_BYTES
    q = torch.empty((n, hq, d), dtype=torch.bfloat16, device="cuda")
    kc = torch.empty((4, 16, hkv, d), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((n, max_len // 16), dtype=torch.int32, device="cuda")
    cl = torch.ones((n,), dtype=torch.int32, device="cuda")
    with pytest.raises(pa.PaError) as e:
        pa.decode_attention_noalloc(torch.empty_like(q), q, kc, kc, bt, cl, 0.088, max_len)
    assert e.value.status == 3
