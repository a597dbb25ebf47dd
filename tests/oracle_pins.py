"""Pins that tie the fp64 oracle to something other than itself.

Each ``pin_*`` function takes an oracle handle and raises AssertionError when
the oracle disagrees with:
  * a library routine the case reduces to (torch / numpy dtype casts,
    ``torch.nn.functional.scaled_dot_product_attention`` in fp64 on the
    contiguous, never-paged K/V the generator drew, numpy fancy-index
    assignment for the append);
  * a closed form (one context token returns that token's V; identical V rows
    return that V; a zero query returns the mean of V; one dominant key returns
    its V);
  * an invariant the pages state or imply (physical placement does not change
    the result, "每生成一个字都要把全部权重读一遍：从 vLLM 看 LLM 推理提速",
    figure caption after the blockwise-attention equation; block sharing by
    reference count, same page, the copy-on-write paragraph; GQA groups,
    "LLM 推理优化的系统视角", section 3.2).
The same functions run against deliberately broken builds of the oracle
(``-DPLANT=n``) to show that each plausible mistake trips at least one pin.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from paged_kv_cache_265_gb300 import workload as W


# ----------------------------------------------------------------------------- helpers

def _bits_to_f64_lib(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Library widening (torch for bf16, numpy for fp16) -- independent of the oracle's."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    if dtype == "fp16":
        return b.view(np.float16).astype(np.float64)
    t = torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def _sdpa_reference(w: W.Workload) -> np.ndarray:
    """Dense attention per sequence on the generator's contiguous K/V via torch SDPA (fp64)."""
    n, q_len, hq, d = w.query.shape
    g = w.num_heads // w.num_kv_heads
    out = np.empty((n, q_len, hq, d), dtype=np.float64)
    for i in range(n):
        L = int(w.context_lens[i])
        q = torch.from_numpy(_bits_to_f64_lib(w.query[i], w.dtype)).permute(1, 0, 2)[None]      # [1,Hq,q,d]
        k = torch.from_numpy(_bits_to_f64_lib(w.logical_key[i], w.dtype)).permute(1, 0, 2)       # [Hkv,L,d]
        v = torch.from_numpy(_bits_to_f64_lib(w.logical_value[i], w.dtype)).permute(1, 0, 2)
        k = k.repeat_interleave(g, dim=0)[None]
        v = v.repeat_interleave(g, dim=0)[None]
        # bottom-right aligned causal mask: row j sees positions 0 .. L - q_len + j
        allowed = torch.arange(L)[None, :] <= (L - q_len + torch.arange(q_len))[:, None]
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=allowed, scale=w.scale)
        out[i] = o[0].permute(1, 0, 2).numpy()
    return out


def _run(orc, w: W.Workload, key_cache=None, value_cache=None, query=None, block_tables=None,
         context_lens=None):
    out, bad = orc.decode_attention(
        w.query if query is None else query,
        w.key_cache if key_cache is None else key_cache,
        w.value_cache if value_cache is None else value_cache,
        w.block_tables if block_tables is None else block_tables,
        w.context_lens if context_lens is None else context_lens,
        w.scale, w.dtype)
    assert bad == 0, f"oracle rejected {bad} sequences"
    return out


def _ulp_close(a: np.ndarray, b: np.ndarray, rel: float) -> None:
    err = np.abs(a - b)
    lim = rel * np.maximum(np.abs(a), np.abs(b)) + 1e-300
    assert np.all(err <= lim), f"max rel err {np.max(err / lim) * rel:.3e} > {rel}"


# ----------------------------------------------------------------------------- storage widening

def pin_bf16_widening(orc):
    bits = np.arange(1 << 16, dtype=np.uint16)
    mine = orc.bits_to_double(bits, "bf16")
    ref = _bits_to_f64_lib(bits, "bf16")
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])


def pin_fp16_widening(orc):
    bits = np.arange(1 << 16, dtype=np.uint16)
    mine = orc.bits_to_double(bits, "fp16")
    ref = _bits_to_f64_lib(bits, "fp16")
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])


# ----------------------------------------------------------------------------- library routine

def pin_sdpa_tiny_named(orc):
    """The tiny 4-sequence MHA workload (d = 64) against SDPA on its contiguous K/V."""
    w = W.tiny_mha(keep_logical=True, append_len=0)
    got = _run(orc, w)
    ref = _sdpa_reference(w)
    assert np.max(np.abs(got - ref)) <= 1e-12, np.max(np.abs(got - ref))


def pin_sdpa_random_small(orc):
    """Random small shapes: GQA groups 1/2/4, chunk lengths 1/3/5, d = 8/64, both dtypes,
    block tails, sequences shorter than one block and shared prefixes."""
    cases = [
        dict(lens=[1, 2, 16, 17], hq=2, hkv=2, d=8, q=1, dtype="bf16", shared=0),
        dict(lens=[5, 23, 40], hq=8, hkv=2, d=64, q=3, dtype="bf16", shared=0),
        dict(lens=[33, 40, 34, 48], hq=4, hkv=1, d=8, q=5, dtype="fp16", shared=2),
        dict(lens=[3, 31, 32, 39], hq=4, hkv=4, d=64, q=3, dtype="fp16", shared=0),
        dict(lens=[64, 100, 130], hq=4, hkv=2, d=8, q=64, dtype="bf16", shared=0),   # a prefill chunk
    ]
    for c_i, c in enumerate(cases):
        w = W.make_workload(f"pin{c_i}", c["lens"], num_heads=c["hq"], num_kv_heads=c["hkv"],
                            head_dim=c["d"], dtype=c["dtype"], q_len=c["q"], append_len=0,
                            num_blocks=48, seed=100 + c_i, shared_prefix_blocks=c["shared"],
                            keep_logical=True)
        got = _run(orc, w)
        ref = _sdpa_reference(w)
        assert np.max(np.abs(got - ref)) <= 1e-12, (c_i, np.max(np.abs(got - ref)))


# ----------------------------------------------------------------------------- closed forms

def pin_single_token_is_its_value(orc):
    """L = 1: the softmax has one term equal to 1, so O = V_0 exactly, for every head."""
    w = W.make_workload("one", [1, 1, 1], num_heads=4, num_kv_heads=2, head_dim=64, append_len=0,
                        num_blocks=8, seed=5, keep_logical=True)
    got = _run(orc, w)
    for i in range(3):
        v0 = _bits_to_f64_lib(w.logical_value[i][0], w.dtype)           # [Hkv, d]
        exp = np.repeat(v0, 2, axis=0)                                  # kv head of h is h // 2
        assert np.array_equal(got[i, 0], exp)


def pin_identical_values(orc):
    """All V rows equal to one vector v: every output row equals v (to a few ulp)."""
    w = W.make_workload("samev", [7, 29, 50], num_heads=4, num_kv_heads=2, head_dim=64, append_len=0,
                        num_blocks=16, seed=6)
    vrow = w.value_cache[w.block_tables[0, 0], 0].copy()               # one [Hkv, d] row
    vc = np.empty_like(w.value_cache)
    vc[...] = vrow
    got = _run(orc, w, value_cache=vc)
    exp = np.repeat(_bits_to_f64_lib(vrow, w.dtype), 2, axis=0)
    for i in range(3):
        _ulp_close(got[i, 0], exp, 8 * 2.0 ** -52)


def pin_zero_query_is_mean(orc):
    """Q = 0: all scores are 0, weights are 1/L, so O is the plain mean of the V rows."""
    w = W.make_workload("q0", [9, 40], num_heads=2, num_kv_heads=1, head_dim=8, append_len=0,
                        num_blocks=8, seed=7, keep_logical=True)
    q0 = np.zeros_like(w.query)
    got = _run(orc, w, query=q0)
    for i in range(2):
        v = _bits_to_f64_lib(w.logical_value[i], w.dtype)               # [L, 1, d]
        mean = np.array([math.fsum(v[:, 0, k]) / v.shape[0] for k in range(v.shape[2])])
        for h in range(2):
            _ulp_close(got[i, 0, h], mean, 64 * 2.0 ** -52)


def pin_dominant_key(orc):
    """One key scoring 32 above every other: O = V of that key to within L * e^-32."""
    L, d = 37, 8
    w = W.make_workload("dom", [L], num_heads=1, num_kv_heads=1, head_dim=d, append_len=0,
                        num_blocks=4, seed=8, keep_logical=True, scale=1.0 / 8.0)
    one = np.uint16(0x3F80)                    # bf16 1.0
    big = np.uint16(0x4380)                    # bf16 256.0
    q = np.zeros_like(w.query)
    q[0, 0, 0, 0] = one                        # q = e_0
    kc = np.zeros_like(w.key_cache)            # every key scores 0 ...
    target = 21
    blk, off = w.block_tables[0, target // 16], target % 16
    kc[blk, off, 0, 0] = big                   # ... except position 21: 256 * 1 / 8 = 32
    got = _run(orc, w, key_cache=kc, query=q)
    vt = _bits_to_f64_lib(w.logical_value[0][target, 0], w.dtype)
    assert np.max(np.abs(got[0, 0, 0] - vt)) <= L * math.exp(-32) * 8, np.max(np.abs(got[0, 0, 0] - vt))


def pin_two_keys_closed_form(orc):
    """Two positions whose scores are exactly 1 and 0 after scaling:
    O = (e * V_0 + V_1) / (e + 1)."""
    w = W.make_workload("two", [2], num_heads=1, num_kv_heads=1, head_dim=8, append_len=0,
                        num_blocks=2, seed=15, keep_logical=True, scale=1.0 / 8.0)
    q = np.zeros_like(w.query)
    q[0, 0, 0, 0] = np.uint16(0x3F80)          # bf16 1.0 -> q = e_0
    kc = np.zeros_like(w.key_cache)
    blk = w.block_tables[0, 0]
    kc[blk, 0, 0, 0] = np.uint16(0x4100)       # bf16 8.0 -> score of position 0 = 8 / 8 = 1
    got = _run(orc, w, key_cache=kc, query=q)
    v0 = _bits_to_f64_lib(w.logical_value[0][0, 0], w.dtype)
    v1 = _bits_to_f64_lib(w.logical_value[0][1, 0], w.dtype)
    exp = (math.e * v0 + v1) / (math.e + 1.0)
    assert np.max(np.abs(got[0, 0, 0] - exp)) <= 1e-15 * 4, np.max(np.abs(got[0, 0, 0] - exp))


# ----------------------------------------------------------------------------- invariants

def pin_block_permutation(orc):
    """Moving every physical block elsewhere (and fixing the tables) changes nothing, bit for bit."""
    w = W.make_workload("perm", [3, 16, 17, 45, 64], num_heads=4, num_kv_heads=2, head_dim=64,
                        append_len=0, num_blocks=24, seed=9)
    base = _run(orc, w)
    perm = np.random.Generator(np.random.PCG64(99)).permutation(w.num_blocks)
    kc = np.empty_like(w.key_cache)
    vc = np.empty_like(w.value_cache)
    kc[perm] = w.key_cache
    vc[perm] = w.value_cache
    bt = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    moved = _run(orc, w, key_cache=kc, value_cache=vc, block_tables=bt)
    assert np.array_equal(base, moved)


def pin_sharing_equals_duplication(orc):
    """Sequences mapping one shared prefix give the same output as private copies of it."""
    w = W.make_workload("share", [40, 52, 33], num_heads=4, num_kv_heads=2, head_dim=8, append_len=0,
                        num_blocks=16, seed=10, shared_prefix_blocks=2)
    shared = _run(orc, w)
    kc, vc, bt = w.key_cache.copy(), w.value_cache.copy(), w.block_tables.copy()
    used = set(int(b) for b in w.block_tables.ravel() if b >= 0)
    spare = [b for b in range(w.num_blocks) if b not in used]
    for i in range(1, w.num_seqs):                # sequence 0 keeps the originals
        for j in range(2):
            nb = spare.pop()
            kc[nb] = w.key_cache[w.block_tables[i, j]]
            vc[nb] = w.value_cache[w.block_tables[i, j]]
            bt[i, j] = nb
    dup = _run(orc, w, key_cache=kc, value_cache=vc, block_tables=bt)
    assert np.array_equal(shared, dup)


def pin_gqa_equals_replicated_mha(orc):
    """GQA with groups of g query heads equals MHA whose kv heads are the GQA heads repeated g times."""
    w = W.make_workload("gqa", [20, 35], num_heads=8, num_kv_heads=2, head_dim=8, q_len=2, append_len=0,
                        num_blocks=8, seed=11)
    gqa = _run(orc, w)
    kc = np.ascontiguousarray(np.repeat(w.key_cache, 4, axis=2))
    vc = np.ascontiguousarray(np.repeat(w.value_cache, 4, axis=2))
    mha = W.Workload(**{**w.__dict__, "num_kv_heads": 8, "key_cache": kc, "value_cache": vc})
    got = _run(orc, mha)
    assert np.array_equal(gqa, got)


def pin_chunk_rows_are_shorter_decodes(orc):
    """Row j of a q-token chunk equals a one-token decode whose context ends at that row."""
    q_len = 4
    w = W.make_workload("chunk", [4, 19, 33], num_heads=4, num_kv_heads=1, head_dim=8, q_len=q_len,
                        append_len=0, num_blocks=8, seed=12)
    full = _run(orc, w)
    for j in range(q_len):
        lens = (w.context_lens - q_len + j + 1).astype(np.int32)
        qj = np.ascontiguousarray(w.query[:, j:j + 1])
        one = W.Workload(**{**w.__dict__, "q_len": 1})
        got = _run(orc, one, query=qj, context_lens=lens)
        assert np.array_equal(full[:, j], got[:, 0]), j


# ----------------------------------------------------------------------------- append

def pin_append_matches_numpy_assignment(orc):
    """The append equals numpy fancy-index assignment on the flattened pool; negative slots
    write nothing and every other byte of the pool keeps its value."""
    w = W.make_workload("app", [5, 17, 30, 64], num_heads=4, num_kv_heads=2, head_dim=8, q_len=1,
                        append_len=3, num_blocks=20, seed=13)
    sm = w.slot_mapping.copy()
    sm[1] = -1                                    # a padding token
    kc, vc = w.key_cache.copy(), w.value_cache.copy()
    bad = orc.reshape_and_cache(w.new_key, w.new_value, kc, vc, sm)
    assert bad == 0
    ek = w.key_cache.reshape(-1, 2, 8).copy()
    ev = w.value_cache.reshape(-1, 2, 8).copy()
    keep = sm >= 0
    ek[sm[keep]] = w.new_key[keep]
    ev[sm[keep]] = w.new_value[keep]
    assert np.array_equal(kc.reshape(-1, 2, 8), ek)
    assert np.array_equal(vc.reshape(-1, 2, 8), ev)


def pin_append_completes_the_pool(orc):
    """Drawing a step with its newest rows held back and appending them gives, byte for
    byte, the pool drawn with nothing held back (same seed, same placement)."""
    kw = dict(num_heads=4, num_kv_heads=2, head_dim=8, q_len=2, num_blocks=16, seed=14)
    lens = [2, 16, 17, 47]
    held = W.make_workload("held", lens, append_len=2, **kw)
    whole = W.make_workload("whole", lens, append_len=0, **kw)
    kc, vc = held.key_cache.copy(), held.value_cache.copy()
    assert orc.reshape_and_cache(held.new_key, held.new_value, kc, vc, held.slot_mapping) == 0
    assert np.array_equal(kc, whole.key_cache)
    assert np.array_equal(vc, whole.value_cache)


def pin_copy_blocks_matches_numpy_assignment(orc):
    """Copy-on-write block copies equal numpy whole-block assignment over the pool; pairs with an
    id outside the pool are skipped and counted."""
    w = W.make_workload("cow", [40, 70, 33], num_heads=4, num_kv_heads=2, head_dim=8, append_len=0,
                        num_blocks=24, seed=16)
    mapping = np.array([[w.block_tables[0, 0], 20], [w.block_tables[1, 3], 21], [w.block_tables[2, 2], 22],
                        [5, 99]], dtype=np.int64)
    kc, vc = w.key_cache.copy(), w.value_cache.copy()
    assert orc.copy_blocks(kc, vc, mapping) == 1
    ek, ev = w.key_cache.copy(), w.value_cache.copy()
    good = mapping[:3]
    ek[good[:, 1]] = w.key_cache[good[:, 0]]
    ev[good[:, 1]] = w.value_cache[good[:, 0]]
    assert np.array_equal(kc, ek) and np.array_equal(vc, ev)


def pin_copy_on_write_fork(orc):
    """Two sequences share a 40-token prefix whose last block is partly filled.  Each copies that
    block before appending its own token 40 (copy-on-write); each then attends exactly over
    the prefix plus its own token (SDPA on contiguous arrays), and the shared block is untouched."""
    g = np.random.Generator(np.random.PCG64(17))
    hkv, d, hq, nb = 2, 8, 4, 12
    bits = lambda *shape: _bf16_bits(g.standard_normal(shape).astype(np.float32))
    kc = np.full((nb, 16, hkv, d), W.NAN_BITS["bf16"], np.uint16)
    vc = kc.copy()
    pk, pv = bits(40, hkv, d), bits(40, hkv, d)
    shared = [7, 2, 9]
    for p_ in range(40):
        kc[shared[p_ // 16], p_ % 16], vc[shared[p_ // 16], p_ % 16] = pk[p_], pv[p_]
    before = kc[9].copy()
    nk, nv = bits(2, hkv, d), bits(2, hkv, d)
    copies = [4, 11]
    assert orc.copy_blocks(kc, vc, np.array([[9, copies[0]], [9, copies[1]]])) == 0
    bt = np.array([[7, 2, copies[0]], [7, 2, copies[1]]], np.int32)
    slots = np.array([copies[0] * 16 + 8, copies[1] * 16 + 8], np.int64)
    assert orc.reshape_and_cache(nk, nv, kc, vc, slots) == 0
    assert np.array_equal(kc[9], before)
    q = bits(2, 1, hq, d)
    lens = np.array([41, 41], np.int32)
    out, bad = orc.decode_attention(q, kc, vc, bt, lens, 1 / math.sqrt(d), "bf16")
    assert bad == 0
    lk = [np.concatenate([pk, nk[i:i + 1]]) for i in range(2)]
    lv = [np.concatenate([pv, nv[i:i + 1]]) for i in range(2)]
    ref_w = W.Workload(name="fork", dtype="bf16", num_heads=hq, num_kv_heads=hkv, head_dim=d, q_len=1,
                       block_size=16, num_blocks=nb, scale=1 / math.sqrt(d), context_lens=lens, block_tables=bt,
                       query=q, key_cache=kc, value_cache=vc, new_key=nk, new_value=nv, slot_mapping=slots,
                       logical_key=lk, logical_value=lv)
    assert np.max(np.abs(out - _sdpa_reference(ref_w))) <= 1e-12


def pin_spec_verify_closed_forms(orc):
    """Equal target and draft distributions accept every draft, then draw the bonus token from
    the target's last row; a draft token the target gives probability 0 is rejected and the
    replacement comes from the positive part of target - draft."""
    v = 4
    pl = np.array([[0.1, 0.2, 0.3, 0.4]] * 3, np.float32)[None]           # [1, k+1=3, V]
    pd = pl[:, :2].copy()
    acc, out = orc.spec_verify(pl, pd, np.array([[3, 1]], np.int32), np.array([[0.9, 0.9]], np.float32),
                               np.array([0.25], np.float32))
    assert acc[0] == 2 and list(out[0]) == [3, 1, 1]                      # prefix 0.1, 0.3 > 0.25
    pl2 = np.array([[[0.5, 0.0, 0.25, 0.25]] * 2], np.float32)
    pd2 = np.array([[[0.0, 1.0, 0.0, 0.0]]], np.float32)
    acc, out = orc.spec_verify(pl2, pd2, np.array([[1]], np.int32), np.array([[0.0]], np.float32),
                               np.array([0.6], np.float32))
    assert acc[0] == 0 and list(out[0]) == [2, -1]                        # residual (0.5, 0, .25, .25)
    assert v == pl.shape[-1]


def pin_spec_verify_output_follows_target(orc):
    """The page's guarantee: the emitted tokens are distributed exactly as target-model samples.
    200,000 trials of a 6-token vocabulary, k = 2, independent positions: the first emitted token
    follows target row 0, the second (when emitted) follows target row 1, and the first draft is
    accepted with probability sum_t min(target, draft)."""
    n, k, v = 200_000, 2, 6
    g = np.random.Generator(np.random.PCG64(18))
    pl = np.array([[0.05, 0.3, 0.1, 0.25, 0.2, 0.1], [0.4, 0.1, 0.1, 0.1, 0.2, 0.1],
                   [0.2, 0.2, 0.2, 0.2, 0.1, 0.1]], np.float32)
    pd = np.array([[0.3, 0.1, 0.2, 0.1, 0.1, 0.2], [0.1, 0.4, 0.1, 0.2, 0.1, 0.1]], np.float32)
    tp = np.broadcast_to(pl, (n, k + 1, v)).copy()
    dp = np.broadcast_to(pd, (n, k, v)).copy()
    pd64 = pd.astype(np.float64)
    tokens = np.stack([g.choice(v, size=n, p=pd64[i] / pd64[i].sum()) for i in range(k)], 1)
    acc, out = orc.spec_verify(tp, dp, tokens.astype(np.int32), g.random((n, k), dtype=np.float32),
                               g.random(n, dtype=np.float32))

    def close(freq, p, m):
        return np.all(np.abs(freq - p) <= 5 * np.sqrt(p * (1 - p) / m) + 1e-9)

    f0 = np.bincount(out[:, 0], minlength=v) / n
    assert close(f0, pl[0], n), f0
    second = out[:, 1][out[:, 1] >= 0]
    f1 = np.bincount(second, minlength=v) / second.size
    assert close(f1, pl[1], second.size), f1
    p_acc = float(np.minimum(pl[0], pd[0]).sum())
    assert abs(np.mean(acc >= 1) - p_acc) <= 5 * np.sqrt(p_acc * (1 - p_acc) / n)


def pin_e4m3_codes(orc):
    """FP8 E4M3 decode of all 256 codes equals torch's float8_e4m3fn; encode equals torch's
    round-to-nearest-even cast below the overflow midpoint (464), including exact ties between
    neighbouring codes, and saturates to +-448 above it."""
    codes = np.arange(256, dtype=np.uint8)
    mine = orc.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan) and np.array_equal(mine[~nan], ref[~nan])
    g = np.random.Generator(np.random.PCG64(19))
    pos = np.sort(ref[(~nan) & (ref > 0)])
    ties = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)            # exact in fp32
    x = np.concatenate([g.standard_normal(200_000).astype(np.float32) * np.float32(40),
                        g.standard_normal(20_000).astype(np.float32) * np.float32(2 ** -8), ties, -ties])
    x = x[np.abs(x) < 464]
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(orc.e4m3_encode(x), want)
    assert list(orc.e4m3_encode(np.array([500, -1000, 464.5, 448], np.float32))) == [0x7E, 0xFE, 0x7E, 0x7E]


def pin_fp8_attention_is_attention_on_dequantised_cache(orc):
    """With power-of-two scales every dequantised value is a bf16 number, so FP8 attention must
    equal, bit for bit, the (SDPA-pinned) 16-bit attention over a bf16 copy of the dequantised
    cache.  The quantising append equals the library cast of the fp32 quotient."""
    w = W.make_workload("fp8", [5, 23, 40, 17], num_heads=8, num_kv_heads=2, head_dim=64, q_len=2,
                        num_blocks=12, seed=20)
    ks, vs = 0.25, 2.0
    kc8 = np.zeros(w.key_cache.shape, np.uint8)
    vc8 = np.zeros(w.value_cache.shape, np.uint8)
    # history: quantise the pool's valid rows; then the append quantises the new rows
    k32 = _bits_to_f64_lib(w.key_cache, "bf16").astype(np.float32)
    v32 = _bits_to_f64_lib(w.value_cache, "bf16").astype(np.float32)
    kc8[...] = orc.e4m3_encode(np.nan_to_num(k32) / np.float32(ks))
    vc8[...] = orc.e4m3_encode(np.nan_to_num(v32) / np.float32(vs))
    assert orc.reshape_and_cache_fp8(w.new_key, w.new_value, kc8, vc8, w.slot_mapping, "bf16", ks, vs) == 0
    nk32 = _bits_to_f64_lib(w.new_key, "bf16").astype(np.float32)
    want = torch.from_numpy(nk32 / np.float32(ks)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = kc8.reshape(-1, 2, 64)[w.slot_mapping]
    assert np.array_equal(got, want)
    out8, bad = orc.decode_attention_fp8(w.query, kc8, vc8, w.block_tables, w.context_lens, w.scale, "bf16", ks, vs)
    assert bad == 0
    deq_k = _bf16_bits((orc.e4m3_decode(kc8) * ks).astype(np.float32))
    deq_v = _bf16_bits((orc.e4m3_decode(vc8) * vs).astype(np.float32))
    assert np.array_equal(_bits_to_f64_lib(deq_k, "bf16"), orc.e4m3_decode(kc8) * ks)   # exact in bf16
    ref = _run(orc, w, key_cache=deq_k, value_cache=deq_v)
    assert np.array_equal(out8, ref)


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


ALL_PINS = [
    pin_bf16_widening, pin_fp16_widening, pin_sdpa_tiny_named, pin_sdpa_random_small,
    pin_single_token_is_its_value, pin_identical_values, pin_zero_query_is_mean, pin_dominant_key,
    pin_two_keys_closed_form,
    pin_block_permutation, pin_sharing_equals_duplication, pin_gqa_equals_replicated_mha,
    pin_chunk_rows_are_shorter_decodes, pin_append_matches_numpy_assignment,
    pin_append_completes_the_pool, pin_copy_blocks_matches_numpy_assignment, pin_copy_on_write_fork,
    pin_spec_verify_closed_forms, pin_spec_verify_output_follows_target, pin_e4m3_codes,
    pin_fp8_attention_is_attention_on_dequantised_cache,
]
