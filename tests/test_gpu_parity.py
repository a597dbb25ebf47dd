"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Append: bit-exact over the WHOLE pool (stray writes would show).
Attention: |gpu - oracle| <= 2e-3 or <= 1e-2 * |oracle|, element by element.
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


_CACHE = {}


def named(k):
    if k not in _CACHE:
        _CACHE.clear()
        _CACHE[k] = W.WORKLOADS[k]()
    return _CACHE[k]


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_named_workload_step(cfg):
    """Append + attention on each named workload, full size, whole outputs compared."""
    w = named(cfg)
    step = G.GpuStep(w)
    got = step.run()
    kc, vc, ref = G.oracle_step(w)
    assert np.array_equal(G.to_bits(step.key_cache), kc)
    assert np.array_equal(G.to_bits(step.value_cache), vc)
    mabs, mrel = G.compare(got, ref, w.dtype, w.name)
    ulps = G.ulps_from_rounded_oracle(got, ref, w.dtype)
    print(f"{w.name}: max abs {mabs:.3e}, max rel (past abs tol) {mrel:.3e}, max ulp vs rounded oracle {ulps}")
    # fp32 accumulation keeps the result within one rounding step of the exact answer
    assert ulps <= 1
    assert pa.get_device_error(clear=True) == 0


@pytest.mark.parametrize("partition", [16, 48, 512, 1 << 20])
@pytest.mark.parametrize("cfg", [1, 4])
def test_partition_sizes_agree(cfg, partition):
    """Forced split (down to one block per partition) and forced no-split give the oracle's result."""
    w = named(cfg)
    step = G.GpuStep(w, partition_size=partition)
    got = step.run()
    _, _, ref = G.oracle_step(w)
    G.compare(got, ref, w.dtype, f"{w.name} partition {partition}")


EDGE = [
    # (lens, Hq, Hkv, d, q_len, dtype)
    ([1, 16, 17, 512, 513, 1025], 8, 8, 128, 1, "bf16"),
    ([1, 2, 15, 31, 33, 700], 4, 4, 64, 1, "fp16"),
    ([5, 5, 6, 21, 512, 517], 32, 8, 128, 5, "bf16"),      # L == q_len, chunk across a partition edge
    ([8, 100, 600], 16, 2, 64, 1, "bf16"),                  # 8 rows per kv head
    ([16, 40, 1200], 16, 1, 128, 1, "fp16"),                # 16 rows: one full row tile
    ([9, 64, 999], 32, 4, 128, 3, "bf16"),                  # 24 rows: two row tiles
    ([12, 300, 1600], 8, 1, 64, 8, "bf16"),                 # 64 rows: four row tiles
    ([5, 77, 1300], 16, 2, 128, 5, "bf16"),                 # 40 rows: three row tiles (+1 padding tile)
    ([64, 300, 700, 1500], 32, 8, 128, 64, "bf16"),         # prefill chunk: 256 rows, four 64-row groups
    ([200, 513, 1100], 8, 8, 128, 200, "fp16"),             # 200 rows: groups of 64, 64, 64, 8
]


@pytest.mark.parametrize("partition", [0, 32])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_rising_falling_and_jumping_scores(dtype, partition):
    """Scores that keep passing the running max every few blocks, that fall from the first block
    on, or that jump inside a block: the online softmax's rescaling paths, held to the same bar
    as the named workloads (with and without a split into 32-token partitions)."""
    w = G.rising_scores_workload(dtype)
    step = G.GpuStep(w, partition_size=partition)
    got = step.run()
    kc, _, ref = G.oracle_step(w)
    assert np.array_equal(G.to_bits(step.key_cache), kc)
    G.compare(got, ref, dtype, f"{w.name} partition {partition}")
    assert G.ulps_from_rounded_oracle(got, ref, dtype) <= 1
    assert pa.get_device_error(clear=True) == 0


@pytest.mark.parametrize("case", range(len(EDGE)))
def test_edge_shapes(case):
    lens, hq, hkv, d, q_len, dt = EDGE[case]
    w = W.make_workload(f"edge{case}", lens, num_heads=hq, num_kv_heads=hkv, head_dim=d, dtype=dt, q_len=q_len,
                        num_blocks=sum((l + 15) // 16 for l in lens) + 7, seed=300 + case)
    for partition in (0, 32):
        step = G.GpuStep(w, partition_size=partition)
        got = step.run()
        _, _, ref = G.oracle_step(w)
        G.compare(got, ref, w.dtype, f"edge{case} partition {partition}")


def test_block_permutation_is_bit_identical():
    """Moving every physical block (and fixing the tables) leaves the GPU output bit-identical."""
    w = named(3)
    a = G.GpuStep(w).run()
    perm = np.random.Generator(np.random.PCG64(5)).permutation(w.num_blocks)
    kc = np.empty_like(w.key_cache)
    vc = np.empty_like(w.value_cache)
    kc[perm] = w.key_cache
    vc[perm] = w.value_cache
    bt = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    moved = W.Workload(**{**w.__dict__, "key_cache": kc, "value_cache": vc, "block_tables": bt,
                          "slot_mapping": (perm[w.slot_mapping // 16] * 16 + w.slot_mapping % 16).astype(np.int64)})
    b = G.GpuStep(moved).run()
    assert np.array_equal(a, b)


def test_repeat_is_bit_identical():
    w = named(3)
    step = G.GpuStep(w)
    a = step.run()
    b = step.run()
    assert np.array_equal(a, b)


def test_shared_prefix_equals_private_copies():
    """The shared-prefix workload gives the same bits when every sequence owns a copy of the prefix."""
    w = named(4)
    a = G.GpuStep(w).run()
    nb = w.num_blocks + (w.num_seqs - 1) * w.shared_prefix_blocks
    kc = np.concatenate([w.key_cache, np.zeros((nb - w.num_blocks,) + w.key_cache.shape[1:], np.uint16)])
    vc = np.concatenate([w.value_cache, np.zeros_like(kc[w.num_blocks:])])
    bt = w.block_tables.copy()
    nxt = w.num_blocks
    for i in range(1, w.num_seqs):
        for j in range(w.shared_prefix_blocks):
            kc[nxt] = w.key_cache[w.block_tables[i, j]]
            vc[nxt] = w.value_cache[w.block_tables[i, j]]
            bt[i, j] = nxt
            nxt += 1
    dup = W.Workload(**{**w.__dict__, "key_cache": kc, "value_cache": vc, "block_tables": bt, "num_blocks": nb})
    b = G.GpuStep(dup).run()
    assert np.array_equal(a, b)


@pytest.mark.parametrize("math", ["tensor", "fma", "tcgen05"])
def test_gqa_equals_replicated_mha(math):
    """GQA (4 query heads per kv head) equals MHA over kv heads repeated 4 times, bit for bit,
    with either consumer arithmetic (each row's sums do not depend on the other rows)."""
    w = W.make_workload("gqa", [40, 333, 1000], num_heads=8, num_kv_heads=2, head_dim=128, num_blocks=120,
                        seed=21)
    mha = W.Workload(**{**w.__dict__, "num_kv_heads": 8,
                        "key_cache": np.ascontiguousarray(np.repeat(w.key_cache, 4, axis=2)),
                        "value_cache": np.ascontiguousarray(np.repeat(w.value_cache, 4, axis=2)),
                        "new_key": np.ascontiguousarray(np.repeat(w.new_key, 4, axis=1)),
                        "new_value": np.ascontiguousarray(np.repeat(w.new_value, 4, axis=1))})
    pa.set_decode_math(math)
    try:
        a = G.GpuStep(w).run()
        b = G.GpuStep(mha).run()
    finally:
        pa.set_decode_math("auto")
    assert np.array_equal(a, b)


def test_bad_block_id_sets_flag_without_fault():
    w = W.make_workload("bad", [40, 70], num_heads=4, num_kv_heads=4, head_dim=64, num_blocks=12, seed=22)
    bt = w.block_tables.copy()
    bt[1, 2] = w.num_blocks + 1000
    step = G.GpuStep(W.Workload(**{**w.__dict__, "block_tables": bt}))
    step.append()
    step.attend()
    torch.cuda.synchronize()
    assert pa.get_device_error(clear=True) & pa.PA_DEVERR_BLOCK_ID
    # the sequence with valid blocks is still right
    _, _, ref = G.oracle_step(w)
    G.compare(G.to_bits(step.out)[:1], ref[:1], w.dtype, "unaffected sequence")


def test_bad_context_len_sets_flag_and_leaves_row():
    w = W.make_workload("badlen", [40, 70], num_heads=4, num_kv_heads=4, head_dim=64, num_blocks=12, seed=23)
    step = G.GpuStep(w)
    step.append()
    step.context_lens[1] = 10 ** 6           # beyond max_context_len
    step.out.fill_(7.0)
    step.attend()
    torch.cuda.synchronize()
    assert pa.get_device_error(clear=True) & pa.PA_DEVERR_CONTEXT
    assert torch.all(step.out[1] == 7.0)


def test_bad_slot_sets_flag_and_writes_nothing():
    w = W.make_workload("badslot", [5, 9], num_heads=4, num_kv_heads=2, head_dim=64, num_blocks=4, seed=24)
    step = G.GpuStep(w)
    before_k = G.to_bits(step.key_cache)
    step.slot_mapping[0] = w.num_blocks * 16 + 3
    step.slot_mapping[1] = -1
    step.append()
    torch.cuda.synchronize()
    assert pa.get_device_error(clear=True) & pa.PA_DEVERR_SLOT
    assert np.array_equal(G.to_bits(step.key_cache), before_k)


def test_launch_counts():
    """Append = 1 kernel; attention = plan + partition kernels, + the merge kernel when a sequence
    can span more than one partition."""
    w = named(1)                                  # longest context 100 < one 512-token partition
    step = G.GpuStep(w)
    step.append()
    assert pa.last_launch_count() == 1
    step.attend()
    assert pa.last_launch_count() == 2
    step16 = G.GpuStep(w, partition_size=16)
    step16.attend()
    assert pa.last_launch_count() == 3
    # a prefill chunk with >= 128 query rows per kv head: one tcgen05 kernel
    chunk = W.make_workload("chunk", [200, 300], num_heads=8, num_kv_heads=2, head_dim=128, q_len=32,
                            num_blocks=40, seed=31)
    G.GpuStep(chunk).attend()
    assert pa.last_launch_count() == 1
    assert pa.last_partition_size() == 0          # no split on the tcgen05 kernel


def test_partition_choice():
    """A forced partition is used as given; partition 0 lets the library pick 512, 1024 or 2048
    tokens (more units per resident CTA -> larger partitions); every choice reaches the oracle."""
    w = named(3)                                  # 128 sequences up to 4096 positions
    step = G.GpuStep(w, partition_size=256)
    step.attend()
    assert pa.last_partition_size() == 256
    auto = G.GpuStep(w)
    got = auto.run()
    assert pa.last_partition_size() in (512, 1024, 2048)
    _, _, ref = G.oracle_step(w)
    G.compare(got, ref, w.dtype, f"{w.name} auto partition {pa.last_partition_size()}")
    assert G.ulps_from_rounded_oracle(got, ref, w.dtype) <= 1


@pytest.mark.parametrize("cfg", [1, 2, 3, 5])
def test_cuda_core_path_matches_oracle(cfg):
    """The CUDA-core FMA consumers, forced on grouped heads too, reach the same results as the
    tensor-core tiles: within tolerance of the oracle and within one ulp of its rounding."""
    w = named(cfg)
    pa.set_decode_math("fma")
    try:
        got = G.GpuStep(w).run()
    finally:
        pa.set_decode_math("auto")
    _, _, ref = G.oracle_step(w)
    G.compare(got, ref, w.dtype, f"{w.name} (CUDA-core path)")
    assert G.ulps_from_rounded_oracle(got, ref, w.dtype) <= 1


@pytest.mark.parametrize("case", [1, 3])
def test_cuda_core_path_edge_shapes(case):
    lens, hq, hkv, d, q_len, dt = EDGE[case]
    w = W.make_workload(f"edge{case}", lens, num_heads=hq, num_kv_heads=hkv, head_dim=d, dtype=dt, q_len=q_len,
                        num_blocks=sum((l + 15) // 16 for l in lens) + 7, seed=300 + case)
    pa.set_decode_math("fma")
    try:
        got = G.GpuStep(w, partition_size=32).run()
    finally:
        pa.set_decode_math("auto")
    _, _, ref = G.oracle_step(w)
    G.compare(got, ref, w.dtype, f"edge{case} (CUDA-core path)")


@pytest.mark.parametrize("cfg", [1, 2])
def test_tensor_path_on_single_row_heads(cfg):
    """MHA workloads run on CUDA cores by default; the tensor-core tiles stay correct there too."""
    w = named(cfg)
    pa.set_decode_math("tensor")
    try:
        got = G.GpuStep(w).run()
    finally:
        pa.set_decode_math("auto")
    _, _, ref = G.oracle_step(w)
    G.compare(got, ref, w.dtype, f"{w.name} (tensor-core path)")
    assert G.ulps_from_rounded_oracle(got, ref, w.dtype) <= 1


def test_chunked_prefill_workload_mma_sync():
    """Chunked prefill on the mma.sync row-group path: 16 sequences, a 256-token chunk each over up
    to 4096 tokens of history."""
    w = W.chunked_prefill()
    pa.set_decode_math("tensor")
    try:
        got = G.GpuStep(w).run()
    finally:
        pa.set_decode_math("auto")
    kc, vc, ref = G.oracle_step(w)
    G.compare(got, ref, w.dtype, w.name)
    assert G.ulps_from_rounded_oracle(got, ref, w.dtype) <= 1
