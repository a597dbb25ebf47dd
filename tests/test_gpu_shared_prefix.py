"""GPU parity of pa_decode_attention_shared_prefix against the oracle.

Sequences that share prefix blocks ("每生成一个字都要把全部权重读一遍：从 vLLM 看 LLM 推理提速",
section "KV Cache 又大又碎，为何不用操作系统分页的思路管它？": one physical block mapped by many
sequences under a reference count) are computed with the prefix attended once per kv head for
all of a group's query rows on the tcgen05 kernel, the rest split-K, and the pieces merged.  The
result is still dense attention over each sequence's own positions, so the oracle is the
ordinary multi-query decode oracle on the same inputs.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_265_gb300 import pa
from paged_kv_cache_265_gb300 import workload as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import gpu_helpers as G


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from paged_kv_cache_265_gb300 import build

    build.build()
    pa.get_device_error(clear=True)
    yield
    assert pa.get_device_error(clear=True) == 0


def run_prefix(w, starts, lens, partition=0):
    step = G.GpuStep(w)
    step.append()
    ws = pa.alloc_workspace_shared_prefix(w.num_seqs, w.q_len, w.num_heads, w.head_dim, w.max_context_len, partition)
    out = torch.full_like(step.query, float("nan"))
    pa.decode_attention_shared_prefix(out, step.query, step.key_cache, step.value_cache, step.block_tables,
                                      step.context_lens, w.scale, w.max_context_len, ws, starts, lens,
                                      partition_size=partition)
    torch.cuda.synchronize()
    return step, G.to_bits(out)


@pytest.mark.parametrize("partition", [0, 512])
def test_shared_prefix_workload(partition):
    """The named shared-prefix workload: 64 sequences, one 1024-token prefix, q = 5."""
    w = W.shared_prefix_verify()
    step, got = run_prefix(w, [0, w.num_seqs], [w.shared_prefix_blocks * 16], partition)
    # 20 query rows per kv head: the one-CTA kernel that orders the suffix units longest first,
    # then the suffix kernel and the prefix kernel, both on tcgen05 (the prefix kernel merges
    # every grouped sequence's pieces)
    assert pa.last_launch_count() == 3
    _, _, ref = G.oracle_step(w)
    G.compare(got, ref, w.dtype, f"shared prefix, partition {partition}")
    assert G.ulps_from_rounded_oracle(got, ref, w.dtype) <= 1
    assert pa.get_device_error(clear=True) == 0


@pytest.mark.parametrize("partition", [0, 16, 128])
def test_shared_prefix_single_token_decode(partition):
    """One query token per sequence (4 rows per kv head): the split-K partition pass takes the
    positions after the prefix, the prefix kernel merges."""
    w = W.make_workload("sp_q1", 1024 + np.arange(5, 400, 13), num_heads=32, num_kv_heads=8, head_dim=128,
                        q_len=1, seed=560, shared_prefix_blocks=64)
    _, got = run_prefix(w, [0, w.num_seqs], [1024], partition)
    assert pa.last_launch_count() == 3           # plan, partition pass, prefix kernel
    _, _, ref = G.oracle_step(w)
    G.compare(got, ref, w.dtype, f"single-token shared prefix, partition {partition}")
    assert G.ulps_from_rounded_oracle(got, ref, w.dtype) <= 1


def _groups_batch(seed, dtype, hq, hkv, d, q_len, sizes, prefix_blocks, suffix):
    """Groups of sequences, group k with sizes[k] sequences sharing prefix_blocks[k] blocks
    (0: a plain group), each sequence with a private suffix of U[suffix] positions."""
    g = np.random.Generator(np.random.PCG64(seed))
    parts = []
    for k, (n, pb) in enumerate(zip(sizes, prefix_blocks)):
        lens = 16 * pb + g.integers(suffix[0], suffix[1] + 1, size=n)
        parts.append(W.make_workload(f"g{k}", lens, num_heads=hq, num_kv_heads=hkv, head_dim=d, dtype=dtype,
                                     q_len=q_len, seed=seed * 100 + k, shared_prefix_blocks=pb))
    w = W.concat_workloads("groups", parts)
    starts = np.concatenate([[0], np.cumsum(sizes)]).tolist()
    return w, starts, [16 * pb for pb in prefix_blocks]


CASES = [
    # (dtype, Hq, Hkv, d, q_len, group sizes, prefix blocks, suffix range)
    ("bf16", 32, 8, 128, 5, [7, 1, 30], [64, 3, 10], (5, 300)),       # rows per group not multiples of 128
    ("fp16", 16, 2, 128, 1, [40, 3], [20, 0], (1, 600)),               # single-token decode; a plain group
    ("bf16", 8, 8, 64, 4, [5, 9], [9, 33], (4, 70)),                   # MHA, d = 64
    ("bf16", 64, 8, 128, 2, [3], [200], (2, 2000)),                    # 3200-position prefix, long suffixes
    ("fp16", 8, 1, 64, 3, [2, 2, 2], [1, 2, 8], (3, 16)),              # one-block prefixes, short suffixes
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_prefix_groups(case):
    dt, hq, hkv, d, q_len, sizes, pblocks, suffix = CASES[case]
    w, starts, lens = _groups_batch(500 + case, dt, hq, hkv, d, q_len, sizes, pblocks, suffix)
    _, _, ref = G.oracle_step(w)
    for partition in (0, 32):
        _, got = run_prefix(w, starts, lens, partition)
        G.compare(got, ref, w.dtype, f"case {case} partition {partition}")
        assert G.ulps_from_rounded_oracle(got, ref, w.dtype) <= 1
    assert pa.get_device_error(clear=True) == 0


def test_ungrouped_sequences_around_groups():
    """Sequences before the first group and after the last share nothing and come out right."""
    dt, hq, hkv, d, q_len = "bf16", 16, 4, 128, 5
    w, starts, lens = _groups_batch(520, dt, hq, hkv, d, q_len, [4, 6, 5], [0, 12, 0], (5, 400))
    # only the middle group is declared, as group [4, 10)
    _, got = run_prefix(w, [4, 10], [lens[1]])
    _, _, ref = G.oracle_step(w)
    G.compare(got, ref, w.dtype, "ungrouped around a group")
    assert G.ulps_from_rounded_oracle(got, ref, w.dtype) <= 1


def test_no_groups_equals_multiquery():
    """With no groups the call is the multi-query call with a finer split: same oracle result."""
    w = W.make_workload("nogroups", [5, 40, 700, 1500], num_heads=32, num_kv_heads=8, head_dim=128, q_len=5,
                        seed=530)
    _, got = run_prefix(w, [], [])
    _, _, ref = G.oracle_step(w)
    G.compare(got, ref, w.dtype, "no groups")


def test_block_permutation_is_bit_identical():
    w = W.shared_prefix_verify()
    _, a = run_prefix(w, [0, w.num_seqs], [1024])
    perm = np.random.Generator(np.random.PCG64(9)).permutation(w.num_blocks)
    kc = np.empty_like(w.key_cache)
    vc = np.empty_like(w.value_cache)
    kc[perm] = w.key_cache
    vc[perm] = w.value_cache
    bt = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    moved = W.Workload(**{**w.__dict__, "key_cache": kc, "value_cache": vc, "block_tables": bt,
                          "slot_mapping": (perm[w.slot_mapping // 16] * 16 + w.slot_mapping % 16).astype(np.int64)})
    _, b = run_prefix(moved, [0, w.num_seqs], [1024])
    assert np.array_equal(a, b)


def test_length_breaking_the_prefix_rule_is_flagged():
    """A grouped sequence whose chunk would start inside the prefix is refused on the device:
    PA_DEVERR_CONTEXT, its rows untouched, the others right."""
    w, starts, lens = _groups_batch(540, "bf16", 8, 2, 128, 5, [6], [8], (5, 100))
    step = G.GpuStep(w)
    step.append()
    torch.cuda.synchronize()
    _, _, ref = G.oracle_step(w)
    step.context_lens[2] = lens[0] + 2          # L - q_len < prefix
    ws = pa.alloc_workspace_shared_prefix(w.num_seqs, w.q_len, w.num_heads, w.head_dim, w.max_context_len)
    out = torch.full_like(step.query, 7.0)
    pa.decode_attention_shared_prefix(out, step.query, step.key_cache, step.value_cache, step.block_tables,
                                      step.context_lens, w.scale, w.max_context_len, ws, starts, lens)
    torch.cuda.synchronize()
    assert pa.get_device_error(clear=True) & pa.PA_DEVERR_CONTEXT
    assert torch.all(out[2] == 7.0)
    keep = [i for i in range(w.num_seqs) if i != 2]
    G.compare(G.to_bits(out)[keep], ref[keep], w.dtype, "the other sequences")


def test_host_validation_of_groups():
    w = W.tiny_mha()
    step = G.GpuStep(w)
    ws = pa.alloc_workspace_shared_prefix(w.num_seqs, w.q_len, w.num_heads, w.head_dim, w.max_context_len)
    args = (torch.empty_like(step.query), step.query, step.key_cache, step.value_cache, step.block_tables,
            step.context_lens, w.scale, w.max_context_len, ws)
    for starts, lens in [([0, 5], [16]),          # past the batch
                         ([2, 1], [16]),          # decreasing
                         ([0, 2], [8]),           # not whole blocks
                         ([0, 2], [-16]),
                         ([0, 2], [112])]:        # more than max_context_len - q_len
        with pytest.raises(pa.PaError) as e:
            pa.decode_attention_shared_prefix(*args, starts, lens)
        assert e.value.status == 1
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(pa.PaError) as e:
        pa.decode_attention_shared_prefix(*args[:-1], small, [0, 2], [16])
    assert e.value.status == 3
