"""The seeded input generator, the one module both the oracle and the CUDA path take inputs from:
its block tables, slot mapping and pool agree with one another and with the recipe."""
import numpy as np

from paged_kv_cache_265_gb300 import workload as W


def _gather(w, cache, i, upto):
    """Rows 0 .. upto-1 of sequence i read from the pool through its block table."""
    p = np.arange(upto)
    return cache[w.block_tables[i, p // w.block_size], p % w.block_size]


def test_tables_slots_and_pool_agree():
    lens = [3, 16, 17, 40, 300]
    w = W.make_workload("gen", lens, num_heads=4, num_kv_heads=2, head_dim=64, q_len=3, append_len=3,
                        num_blocks=40, seed=5, keep_logical=True)
    nblk = [(l + 15) // 16 for l in lens]
    used = np.concatenate([w.block_tables[i, :nblk[i]] for i in range(len(lens))])
    assert len(set(used.tolist())) == used.size and used.min() >= 0 and used.max() < w.num_blocks
    for i, n in enumerate(nblk):
        assert np.all(w.block_tables[i, n:] == -1)          # entries past the sequence are unused
    # the append's rows: each sequence's last 3 positions, in sequence order
    want = []
    for i, L in enumerate(lens):
        for p in range(max(0, L - 3), L):
            want.append(int(w.block_tables[i, p // 16]) * 16 + p % 16)
    assert w.slot_mapping.tolist() == want
    # before the append those slots hold the sentinel; after it the pool is each sequence's
    # logical K/V, read through its table
    kc = w.key_cache.reshape(-1, w.num_kv_heads, w.head_dim).copy()
    vc = w.value_cache.reshape(-1, w.num_kv_heads, w.head_dim).copy()
    assert np.all(kc[w.slot_mapping] == W.NAN_BITS[w.dtype])
    kc[w.slot_mapping] = w.new_key
    vc[w.slot_mapping] = w.new_value
    kc = kc.reshape(w.key_cache.shape)
    vc = vc.reshape(w.value_cache.shape)
    for i, L in enumerate(lens):
        assert np.array_equal(_gather(w, kc, i, L), w.logical_key[i])
        assert np.array_equal(_gather(w, vc, i, L), w.logical_value[i])
        # the tail of the last block stays the sentinel
        last = int(w.block_tables[i, nblk[i] - 1])
        assert np.all(kc[last, L - 16 * (nblk[i] - 1):] == W.NAN_BITS[w.dtype])


def test_shared_prefix_tables():
    w = W.make_workload("sp", [40, 50, 70], num_heads=4, num_kv_heads=1, head_dim=64, q_len=2,
                        num_blocks=20, seed=6, shared_prefix_blocks=2, keep_logical=True)
    assert np.all(w.block_tables[:, :2] == w.block_tables[0, :2])
    private = np.concatenate([w.block_tables[i, 2:(l + 15) // 16] for i, l in enumerate([40, 50, 70])])
    assert len(set(private.tolist())) == private.size
    assert not set(private.tolist()) & set(w.block_tables[0, :2].tolist())
    for i in range(3):  # the first 32 logical rows are the same tokens in every sequence
        assert np.array_equal(w.logical_key[i][:32], w.logical_key[0][:32])


def test_length_recipe_bounds_and_seed():
    a = W._uniform_lens(2653, 128, 1, 4096)
    assert a.min() >= 1 and a.max() <= 4096 and 1500 < a.mean() < 2600
    assert np.array_equal(a, W._uniform_lens(2653, 128, 1, 4096))
    assert not np.array_equal(a, W._uniform_lens(2654, 128, 1, 4096))
    q = W.make_workload("q", [3, 9], num_heads=2, num_kv_heads=2, head_dim=64, seed=1).query
    assert q.dtype == np.uint16 and q.shape == (2, 1, 2, 64)


def test_rising_scores_case_moves_the_running_max():
    """The GPU parity case with moving scores does what it is there for: in the rising sequence every
    query row sees its block maximum pass the running maximum by more than 8 (log2 units) many times,
    with blocks in between whose scores sit nearly 8 above it; the falling sequence never moves it after
    its first block; the step sequence jumps by more than 60 inside block 25; and no score is large
    enough for fp32 rounding of the scores to cost fp16 a unit in the last place (|s| < 90)."""
    import math

    import gpu_helpers as G

    w = G.rising_scores_workload("bf16")
    q = G.bits_to_f64(w.query.ravel(), "bf16").reshape(w.query.shape)
    pool = G.bits_to_f64(w.key_cache.ravel(), "bf16").reshape(-1, w.num_kv_heads, w.head_dim)
    new = G.bits_to_f64(w.new_key.ravel(), "bf16").reshape(w.new_key.shape)
    g = w.num_heads // w.num_kv_heads
    for i, L in enumerate(w.context_lens.tolist()):
        p = np.arange(L - 1)
        keys = np.concatenate([pool[w.block_tables[i, p // 16].astype(np.int64) * 16 + p % 16], new[i][None]])
        for h in range(w.num_heads):
            s = keys[:, h // g] @ q[i, 0, h] * w.scale / math.log(2)
            assert np.abs(s).max() < 90
            block_max = [s[j:j + 16].max() for j in range(0, L, 16)]
            m, moves, near = -np.inf, 0, 0
            for b in block_max:
                if b > m + 8:
                    m, moves = b, moves + 1
                elif b > m + 6:
                    near += 1
            if i == 0:
                assert moves >= 8 and near >= 20, (h, moves, near)
            if i == 1:
                assert moves == 1, (h, moves)
            if i == 2:
                assert s[407:416].min() - s[400:407].max() > 60
