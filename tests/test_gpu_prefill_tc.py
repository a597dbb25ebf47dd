"""GPU parity of the tcgen05 prefill kernel (128-row query tiles, S and O in tensor memory)
through the C ABI against the fp64 oracle.

Like the other paths it is held to the attention tolerance (|gpu - oracle| <= 2e-3 or
<= 1e-2 |oracle|) element by element, and to one unit in the last place of the oracle rounded
once to the output type (the softmax weights reach the P.V product as a hi + lo pair of 16-bit
values, about 16 significant bits).
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_265_gb300 import pa
from paged_kv_cache_265_gb300 import workload as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import gpu_helpers as G

# Largest distance from the oracle rounded once to the output type, in units in the last place,
# over outputs with |o| >= 2^-6.
TC_ULP_BOUND = 1


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from paged_kv_cache_265_gb300 import build

    build.build()
    pa.get_device_error(clear=True)
    yield
    pa.set_decode_math("auto")
    assert pa.get_device_error(clear=True) == 0


def run_tc(w, partition_size=0):
    pa.set_decode_math("tcgen05")
    try:
        return G.GpuStep(w, partition_size=partition_size).run()
    finally:
        pa.set_decode_math("auto")


def test_chunked_prefill_workload():
    """The chunked-prefill workload (16 sequences, 256-token chunks over up to 4096 positions of
    history) on its default path, which is the tcgen05 kernel."""
    w = W.chunked_prefill()
    step = G.GpuStep(w)
    got = step.run()
    assert pa.last_launch_count() == 1
    kc, vc, ref = G.oracle_step(w)
    assert np.array_equal(G.to_bits(step.key_cache), kc)
    mabs, mrel = G.compare(got, ref, w.dtype, w.name)
    ulps = G.ulps_from_rounded_oracle(got, ref, w.dtype)
    print(f"{w.name} (tcgen05): max abs {mabs:.3e}, max rel {mrel:.3e}, max ulp {ulps}")
    assert ulps <= TC_ULP_BOUND


TC_SHAPES = [
    # (lens, Hq, Hkv, d, q_len, dtype)
    ([64, 300, 700, 1500], 32, 8, 128, 64, "bf16"),   # 256 rows: two tiles per kv head
    ([200, 513, 1100], 8, 8, 128, 200, "fp16"),       # 200 rows: a full and a ragged tile
    ([128, 129, 255, 1000], 4, 1, 64, 128, "bf16"),   # d = 64, 512 rows, L == q_len
    ([33, 257, 1030], 12, 4, 128, 33, "bf16"),        # g = 3: tiles straddle chunk tokens
    ([130, 2049], 2, 2, 128, 130, "fp16"),            # MHA rows, 2 tiles, short last blocks
    ([1, 16, 17, 512, 513, 1025], 8, 8, 128, 1, "bf16"),   # one row per kv head (padded tile)
    ([5, 5, 6, 21, 512, 517], 32, 8, 128, 5, "bf16"),      # 20 rows (speculative chunk)
    ([1, 2, 15, 31, 33, 700], 4, 4, 64, 1, "fp16"),
]


@pytest.mark.parametrize("case", range(len(TC_SHAPES)))
def test_tc_shapes(case):
    lens, hq, hkv, d, q_len, dt = TC_SHAPES[case]
    w = W.make_workload(f"tc{case}", lens, num_heads=hq, num_kv_heads=hkv, head_dim=d, dtype=dt, q_len=q_len,
                        num_blocks=sum((l + 15) // 16 for l in lens) + 7, seed=700 + case)
    got = run_tc(w)
    _, _, ref = G.oracle_step(w)
    mabs, mrel = G.compare(got, ref, w.dtype, f"tc{case}")
    ulps = G.ulps_from_rounded_oracle(got, ref, w.dtype)
    print(f"tc{case}: max abs {mabs:.3e}, max ulp {ulps}")
    assert ulps <= TC_ULP_BOUND


@pytest.mark.parametrize("cfg", [1, 3, 4])
def test_tc_named_workloads(cfg):
    """The named decode workloads forced onto the tcgen05 kernel (mostly padding rows there)."""
    w = W.WORKLOADS[cfg]()
    got = run_tc(w)
    _, _, ref = G.oracle_step(w)
    G.compare(got, ref, w.dtype, f"{w.name} (tcgen05)")
    assert G.ulps_from_rounded_oracle(got, ref, w.dtype) <= TC_ULP_BOUND


def _small_chunk(seed=41):
    return W.make_workload("chunk", [300, 777, 1290], num_heads=16, num_kv_heads=4, head_dim=128, q_len=96,
                           num_blocks=160, seed=seed)


def test_tc_repeat_and_block_permutation_bit_identical():
    w = _small_chunk()
    a = run_tc(w)
    b = run_tc(w)
    assert np.array_equal(a, b)
    perm = np.random.Generator(np.random.PCG64(6)).permutation(w.num_blocks)
    kc = np.empty_like(w.key_cache)
    vc = np.empty_like(w.value_cache)
    kc[perm] = w.key_cache
    vc[perm] = w.value_cache
    bt = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    moved = W.Workload(**{**w.__dict__, "key_cache": kc, "value_cache": vc, "block_tables": bt,
                          "slot_mapping": (perm[w.slot_mapping // 16] * 16 + w.slot_mapping % 16).astype(np.int64)})
    assert np.array_equal(a, run_tc(moved))


def test_tc_chunk_rows_equal_shorter_chunks():
    """Row j of a q-row chunk is bit-identical to the last row of the (j+1)-row chunk over the same
    cache with the later q-1-j tokens cut off (causality inside the chunk, on the GPU alone)."""
    w = _small_chunk(seed=43)
    step = G.GpuStep(w)
    pa.set_decode_math("tcgen05")
    try:
        step.run()
        full = step.out.clone()
        for j in (0, 1, 31, 32, w.q_len // 2, w.q_len - 1):
            q2 = step.query[:, : j + 1].contiguous()
            out2 = torch.empty_like(q2)
            lens2 = (step.context_lens - (w.q_len - 1 - j)).contiguous()
            ws = pa.alloc_workspace(w.num_seqs, j + 1, w.num_heads, w.head_dim, w.max_context_len)
            pa.decode_attention(out2, q2, step.key_cache, step.value_cache, step.block_tables, lens2, w.scale,
                                w.max_context_len, ws)
            torch.cuda.synchronize()
            assert torch.equal(out2[:, j].view(torch.int16), full[:, j].view(torch.int16)), f"row {j}"
    finally:
        pa.set_decode_math("auto")


def test_tc_bad_context_len_sets_flag_and_leaves_row():
    w = _small_chunk(seed=44)
    step = G.GpuStep(w)
    step.append()
    step.context_lens[1] = 10 ** 6
    step.out.fill_(7.0)
    pa.set_decode_math("tcgen05")
    try:
        step.attend()
    finally:
        pa.set_decode_math("auto")
    torch.cuda.synchronize()
    assert pa.get_device_error(clear=True) & pa.PA_DEVERR_CONTEXT
    assert torch.all(step.out[1] == 7.0)
    _, _, ref = G.oracle_step(w)
    got = G.to_bits(step.out).reshape(ref.shape)
    G.compare(got[0], ref[0], w.dtype, "unaffected sequence 0")
    G.compare(got[2], ref[2], w.dtype, "unaffected sequence 2")


def test_tc_bad_block_id_sets_flag_without_fault():
    w = _small_chunk(seed=45)
    bt = w.block_tables.copy()
    bt[2, 3] = w.num_blocks + 1000
    step = G.GpuStep(W.Workload(**{**w.__dict__, "block_tables": bt}))
    step.append()
    pa.set_decode_math("tcgen05")
    try:
        step.attend()
    finally:
        pa.set_decode_math("auto")
    torch.cuda.synchronize()
    assert pa.get_device_error(clear=True) & pa.PA_DEVERR_BLOCK_ID
    _, _, ref = G.oracle_step(w)
    got = G.to_bits(step.out).reshape(ref.shape)
    G.compare(got[:2], ref[:2], w.dtype, "sequences with valid blocks")
