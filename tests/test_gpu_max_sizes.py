"""GPU parity at the largest sizes the suite reaches.

* Decode over one 131,072-token sequence (8,192 pool blocks) among short ones: 64 query heads
  on 8 kv heads, every output compared with the oracle. It runs with the library's partition
  choice and with 512-token partitions (256 partials of the long sequence merged).
* A 512-token prefill chunk of 64 query heads over that sequence: 4,096 query rows per kv head,
  32 tcgen05 tiles each. The oracle checks sampled rows. Row j of a chunk attends to positions
  0 .. L - q_len + j, so the oracle computes it as a one-row decode over the first
  L - q_len + j + 1 positions of the same appended pool. The oracle pins check that this
  identity holds.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_265_gb300 import pa
from paged_kv_cache_265_gb300 import workload as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import gpu_helpers as G

LONG = 131072


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from paged_kv_cache_265_gb300 import build

    build.build()
    pa.get_device_error(clear=True)
    yield
    assert pa.get_device_error(clear=True) == 0


def _pool_blocks(lens):
    return sum((l + 15) // 16 for l in lens) + 7


@pytest.fixture(scope="module")
def long_decode():
    lens = [LONG, 1, 17, 4095]
    w = W.make_workload("max_decode", lens, num_heads=64, num_kv_heads=8, head_dim=128, dtype="bf16", q_len=1,
                        num_blocks=_pool_blocks(lens), seed=9001)
    return w, G.oracle_step(w)


@pytest.mark.parametrize("partition", [0, 512])
def test_decode_131072_tokens(long_decode, partition):
    w, (kc, vc, ref) = long_decode
    step = G.GpuStep(w, partition_size=partition)
    got = step.run()
    assert np.array_equal(G.to_bits(step.key_cache), kc)
    assert np.array_equal(G.to_bits(step.value_cache), vc)
    G.compare(got, ref, w.dtype, f"max decode partition {partition}")
    assert G.ulps_from_rounded_oracle(got, ref, w.dtype) <= 1
    assert pa.get_device_error(clear=True) == 0


def test_prefill_chunk_512_over_131072_tokens():
    q_len = 512
    lens = [LONG, 600]
    w = W.make_workload("max_chunk", lens, num_heads=64, num_kv_heads=8, head_dim=128, dtype="bf16", q_len=q_len,
                        num_blocks=_pool_blocks(lens), seed=9002)
    step = G.GpuStep(w)
    got = step.run()   # 4096 rows per kv head: the tcgen05 kernel, one launch
    assert pa.last_launch_count() == 1
    assert pa.get_device_error(clear=True) == 0

    orc = oracle.load()
    kc, vc = w.key_cache.copy(), w.value_cache.copy()
    assert orc.reshape_and_cache(w.new_key, w.new_value, kc, vc, w.slot_mapping) == 0
    assert np.array_equal(G.to_bits(step.key_cache), kc)
    # (sequence, chunk row): tile edges (128 rows = 16 chunk tokens at g = 8), both ends, the middle
    sample = [(0, 0), (0, 15), (0, 16), (0, 255), (0, 511), (1, 0), (1, 1), (1, 300), (1, 511)]
    seqs = np.array([s for s, _ in sample])
    rows = np.array([j for _, j in sample])
    query = w.query[seqs, rows][:, None]                       # [S, 1, Hq, d]
    tables = w.block_tables[seqs]
    ctx = (w.context_lens[seqs] - q_len + rows + 1).astype(np.int32)
    ref, bad = orc.decode_attention(query, kc, vc, tables, ctx, w.scale, w.dtype)
    assert bad == 0
    got_rows = got[seqs, rows][:, None]
    G.compare(got_rows, ref, w.dtype, "max chunk sampled rows")
    assert G.ulps_from_rounded_oracle(got_rows, ref, w.dtype) <= 1
