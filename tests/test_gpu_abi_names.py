"""The boundary calls by their own names, on the GPU through the C ABI.

pa_decode_attention (one query token per sequence) and pa_decode_attention_multiquery (q_len
rows per sequence, causal inside the chunk) are the two attention calls the library exports
for the paged decode step ("现代 LLM 推理引擎剖析", section 1.6: the forward pass runs the
paged attention kernel; "每生成一个字都要把全部权重读一遍：从 vLLM 看 LLM 推理提速", section
"对症下药": the large model checks gamma + 1 positions in one forward).  Each is checked
element by element against the oracle and bit for bit against the general call
(pa_decode_attention_ex) with the library-chosen split.
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


def _ex_bits(step):
    step.attend()                           # pa_decode_attention_ex, partition 0
    torch.cuda.synchronize()
    return G.to_bits(step.out)


@pytest.mark.parametrize("make", [W.tiny_mha, W.gqa_batch32], ids=["tiny_mha", "gqa_batch32"])
def test_pa_decode_attention(make):
    w = make()
    step = G.GpuStep(w)
    step.append()
    q = step.query.view(w.num_seqs, w.num_heads, w.head_dim)       # one query token: [N, Hq, d]
    out = torch.full_like(q, float("nan"))
    pa.decode_attention_single(out, q, step.key_cache, step.value_cache, step.block_tables, step.context_lens,
                               w.scale, w.max_context_len, step.workspace)
    torch.cuda.synchronize()
    got = G.to_bits(out)
    _, _, ref = G.oracle_step(w)
    G.compare(got, ref.reshape(w.num_seqs, w.num_heads, w.head_dim), w.dtype, f"pa_decode_attention {w.name}")
    assert np.array_equal(got.reshape(-1), _ex_bits(step).reshape(-1))
    assert pa.get_device_error(clear=True) == 0


@pytest.mark.parametrize("make", [W.shared_prefix_verify, W.chunked_prefill], ids=["shared_prefix_q5", "chunk_q256"])
def test_pa_decode_attention_multiquery(make):
    w = make()
    step = G.GpuStep(w)
    step.append()
    out = torch.full_like(step.query, float("nan"))
    pa.decode_attention_multiquery(out, step.query, step.key_cache, step.value_cache, step.block_tables,
                                   step.context_lens, w.scale, w.max_context_len, step.workspace)
    torch.cuda.synchronize()
    got = G.to_bits(out)
    _, _, ref = G.oracle_step(w)
    G.compare(got, ref, w.dtype, f"pa_decode_attention_multiquery {w.name}")
    assert G.ulps_from_rounded_oracle(got, ref, w.dtype) <= 1
    assert np.array_equal(got, _ex_bits(step))
    assert pa.get_device_error(clear=True) == 0


def test_names_refuse_bad_shapes_before_launch():
    w = W.tiny_mha()
    step = G.GpuStep(w)
    q = step.query.view(w.num_seqs, w.num_heads, w.head_dim)
    small = torch.empty(4, dtype=torch.uint8, device="cuda")        # workspace far too small
    with pytest.raises(pa.PaError) as e:
        pa.decode_attention_single(torch.empty_like(q), q, step.key_cache, step.value_cache, step.block_tables,
                                   step.context_lens, w.scale, w.max_context_len, small)
    assert e.value.status == 3
    assert pa.last_launch_count() == 0
