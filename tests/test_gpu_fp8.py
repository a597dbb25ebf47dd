"""GPU parity of the FP8 (E4M3) KV cache against the oracle: the quantising append
bit-exact over the whole pool, attention within the attention tolerance."""
import dataclasses

import numpy as np
import pytest
import torch

from paged_kv_cache_265_gb300 import pa
from paged_kv_cache_265_gb300 import workload as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import gpu_helpers as G
    import oracle

K_SCALE, V_SCALE = 0.05, 0.03   # not powers of two: real rescaling on both sides


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from paged_kv_cache_265_gb300 import build

    build.build()
    pa.get_device_error(clear=True)
    yield
    assert pa.get_device_error(clear=True) == 0


def fp8_pools(w: W.Workload):
    """History quantised on the host by the oracle (NaN sentinels stay NaN bytes)."""
    orc = oracle.load()
    k = G.bits_to_f64(w.key_cache.ravel(), w.dtype).astype(np.float32)
    v = G.bits_to_f64(w.value_cache.ravel(), w.dtype).astype(np.float32)
    kc = orc.e4m3_encode(k / np.float32(K_SCALE)).reshape(w.key_cache.shape)
    vc = orc.e4m3_encode(v / np.float32(V_SCALE)).reshape(w.value_cache.shape)
    return kc, vc


def run_fp8(w: W.Workload, partition: int = 0):
    kc, vc = fp8_pools(w)
    dk, dv = torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda()
    pa.reshape_and_cache_fp8(G.to_dev(w.new_key, w.dtype), G.to_dev(w.new_value, w.dtype), dk, dv,
                             torch.from_numpy(w.slot_mapping).cuda(), K_SCALE, V_SCALE)
    q = G.to_dev(w.query, w.dtype)
    out = torch.empty_like(q)
    ws = pa.alloc_workspace(w.num_seqs, w.q_len, w.num_heads, w.head_dim, w.max_context_len, partition)
    pa.decode_attention_fp8kv(out, q, dk, dv, torch.from_numpy(w.block_tables).cuda(),
                              torch.from_numpy(w.context_lens).cuda(), w.scale, w.max_context_len, ws, K_SCALE,
                              V_SCALE, partition_size=partition)
    torch.cuda.synchronize()
    orc = oracle.load()
    assert orc.reshape_and_cache_fp8(w.new_key, w.new_value, kc, vc, w.slot_mapping, w.dtype, K_SCALE, V_SCALE) == 0
    assert np.array_equal(dk.cpu().numpy(), kc) and np.array_equal(dv.cpu().numpy(), vc)
    ref, bad = orc.decode_attention_fp8(w.query, kc, vc, w.block_tables, w.context_lens, w.scale, w.dtype,
                                        K_SCALE, V_SCALE)
    assert bad == 0
    return G.to_bits(out), ref


@pytest.mark.parametrize("cfg", [3, 2, 4])
def test_fp8_named_workloads(cfg):
    w = W.WORKLOADS[cfg]()
    got, ref = run_fp8(w)
    if cfg == 3:
        assert pa.last_partition_size() == 1024   # the automatic rule's choice for this batch
    mabs, mrel = G.compare(got, ref, w.dtype, f"{w.name} fp8")
    print(f"{w.name} fp8: max abs {mabs:.3e}, ulp vs rounded oracle {G.ulps_from_rounded_oracle(got, ref, w.dtype)}")


@pytest.mark.parametrize("partition", [16, 1 << 20])
def test_fp8_partitions_and_edges(partition):
    w = W.make_workload("fp8edge", [1, 16, 17, 513, 1500], num_heads=16, num_kv_heads=4, head_dim=128,
                        dtype="fp16", q_len=1, num_blocks=160, seed=41)
    got, ref = run_fp8(w, partition)
    G.compare(got, ref, w.dtype, f"fp8 partition {partition}")


@pytest.mark.parametrize("partition", [0, 32])
def test_fp8_rising_falling_and_jumping_scores(partition):
    """Scores that keep passing the running max, fall, or jump inside a block, over an FP8 cache
    (keys up to about 10, within E4M3's range at the test's k_scale)."""
    w = G.rising_scores_workload("bf16")
    got, ref = run_fp8(w, partition)
    G.compare(got, ref, w.dtype, f"{w.name} fp8 partition {partition}")
    assert pa.get_device_error(clear=True) == 0


def test_fp8_head_dim_64_is_unsupported():
    q = torch.empty((2, 4, 64), dtype=torch.bfloat16, device="cuda")
    kc = torch.empty((4, 16, 4, 64), dtype=torch.uint8, device="cuda")
    bt = torch.zeros((2, 4), dtype=torch.int32, device="cuda")
    cl = torch.ones(2, dtype=torch.int32, device="cuda")
    ws = pa.alloc_workspace(2, 1, 4, 64, 64)
    with pytest.raises(pa.PaError) as e:
        pa.decode_attention_fp8kv(torch.empty_like(q), q, kc, kc, bt, cl, 0.125, 64, ws, 1.0, 1.0)
    assert e.value.status == 2


def test_fp8_chunk_row_groups():
    """A 64-token chunk over FP8 caches: 256 query rows per kv head run as eight 32-row groups."""
    w = W.make_workload("fp8chunk", [64, 300, 1100], num_heads=16, num_kv_heads=4, head_dim=128, dtype="bf16",
                        q_len=64, num_blocks=110, seed=42)
    got, ref = run_fp8(w)
    G.compare(got, ref, w.dtype, "fp8 chunk")


def _query_row_scaled(w: W.Workload, row: int, log2_factor: int) -> W.Workload:
    """The workload with query row `row` (a (sequence, token, head) row of the flattened query)
    times 2^log2_factor, exact in bf16."""
    q = G.bits_to_f64(w.query.ravel(), w.dtype).reshape(-1, w.head_dim)
    q[row] *= 2.0 ** log2_factor
    bits = torch.from_numpy(q.ravel()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(G.bits_to_f64(bits, "bf16"), q.ravel())
    return dataclasses.replace(w, query=bits.reshape(w.query.shape))


def test_fp8_bf16_query_beyond_fp16_is_refused():
    """A bf16 query element beyond fp16's range (here a row scaled by 2^17, |q| up to ~5e5) has no
    value in the fp16 score products: the call raises PA_DEVERR_QUERY_RANGE, and every other row
    (another column of the products) still matches the oracle and the in-range call bit for bit."""
    w = W.make_workload("fp8range", [1, 40, 700, 2100], num_heads=32, num_kv_heads=4, head_dim=128,
                        dtype="bf16", q_len=1, num_blocks=190, seed=43)
    base, _ = run_fp8(w)
    assert pa.get_device_error(clear=True) == 0
    bad_row = 2 * w.num_heads + 5  # sequence 2, head 5
    wb = _query_row_scaled(w, bad_row, 17)
    assert np.abs(G.bits_to_f64(wb.query.ravel(), "bf16")).max() >= 65520.0
    got, ref = run_fp8(wb)
    assert pa.get_device_error(clear=True) & pa.PA_DEVERR_QUERY_RANGE
    keep = np.ones(got.reshape(-1, w.head_dim).shape[0], dtype=bool)
    keep[bad_row] = False
    g2, r2 = got.reshape(-1, w.head_dim)[keep], ref.reshape(-1, w.head_dim)[keep]
    G.compare(g2, r2, w.dtype, "fp8 rows beside the refused one")
    assert np.array_equal(g2, base.reshape(-1, w.head_dim)[keep])


def test_fp8_bf16_query_at_fp16_edges():
    """bf16 query rows at the edges of what fp16 holds exactly: a row scaled so its largest element
    is just under 65504 and a row scaled down to about 2^-16: no flag, oracle tolerance."""
    w = W.make_workload("fp8edge16", [33, 600], num_heads=16, num_kv_heads=4, head_dim=128, dtype="bf16",
                        q_len=1, num_blocks=60, seed=44)
    q = G.bits_to_f64(w.query.ravel(), "bf16").reshape(-1, w.head_dim)
    big = int(np.floor(np.log2(65504.0 / np.abs(q[3]).max())))
    wb = _query_row_scaled(_query_row_scaled(w, 3, big), 7, -14)
    got, ref = run_fp8(wb)
    assert pa.get_device_error(clear=True) == 0
    G.compare(got, ref, w.dtype, "fp8 query rows at the fp16 edges")


def test_fp8_kernel_wait_runs_out_and_recovers():
    """The FP8 decode kernel (whose warps release each stage right after loading it) stops on a
    pipeline wait that runs out (pa_set_wait_limit_ns(1)): the call reports PA_DEVERR_TIMEOUT and
    nothing else, and the next call with the default limit matches the oracle."""
    w = W.make_workload("fp8_timeout", [40, 700, 1900, 3000], num_heads=32, num_kv_heads=8, head_dim=128,
                        q_len=1, num_blocks=400, seed=43)
    kc, vc = fp8_pools(w)
    dk, dv = torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda()
    pa.reshape_and_cache_fp8(G.to_dev(w.new_key, w.dtype), G.to_dev(w.new_value, w.dtype), dk, dv,
                             torch.from_numpy(w.slot_mapping).cuda(), K_SCALE, V_SCALE)
    q = G.to_dev(w.query, w.dtype)
    out = torch.empty_like(q)
    ws = pa.alloc_workspace(w.num_seqs, w.q_len, w.num_heads, w.head_dim, w.max_context_len, 0)
    bt, cl = torch.from_numpy(w.block_tables).cuda(), torch.from_numpy(w.context_lens).cuda()

    def call():
        pa.decode_attention_fp8kv(out, q, dk, dv, bt, cl, w.scale, w.max_context_len, ws, K_SCALE, V_SCALE)
        torch.cuda.synchronize()

    torch.cuda.synchronize()
    pa.get_device_error(clear=True)
    try:
        pa.set_wait_limit_ns(1)
        call()
        pa.set_wait_limit_ns(0)
        flags = pa.get_device_error(clear=True)
        assert flags & pa.PA_DEVERR_TIMEOUT, f"no wait ran out (flags {flags:#x})"
        assert flags & ~pa.PA_DEVERR_TIMEOUT == 0, f"unexpected flags {flags:#x}"
        out.fill_(float("nan"))
        call()
        got = G.to_bits(out)
    finally:
        pa.set_wait_limit_ns(0)
    assert pa.get_device_error(clear=True) == 0
    orc = oracle.load()
    assert orc.reshape_and_cache_fp8(w.new_key, w.new_value, kc, vc, w.slot_mapping, w.dtype, K_SCALE, V_SCALE) == 0
    ref, bad = orc.decode_attention_fp8(w.query, kc, vc, w.block_tables, w.context_lens, w.scale, w.dtype,
                                        K_SCALE, V_SCALE)
    assert bad == 0
    G.compare(got, ref, w.dtype, "fp8 after a timed-out call")
