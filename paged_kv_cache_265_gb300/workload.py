"""Seeded synthetic inputs for paged-KV decode attention.

This module only draws random numbers and lays them out as the inputs of one
decode step; it holds none of the attention arithmetic.  Both the CUDA path
(through the tests and the benchmark) and the CPU oracle are fed from it.

What one decode step looks like (the model-runner view of "现代 LLM 推理引擎剖析",
section 1.6, and the decode-step state change of "LLM 推理优化的系统视角",
section 3.1): every sequence already holds the K/V of its earlier positions in
fixed 16-token blocks scattered through one pool, addressed by its block table;
the step appends the K/V rows of its newest ``append_len`` positions through the
slot mapping, and then its ``q_len`` query rows attend over all ``L_i``
positions (``L_i`` counts the new ones).

Recipe (the same for every workload):
  * lengths are uniform integers over inclusive bounds;
  * physical blocks come from a seeded shuffled free list, popped in sequence
    order (shared-prefix blocks are popped first and mapped by every sequence);
  * Q/K/V values are fp32 N(0, 1) draws rounded to bf16 or fp16 (round to
    nearest even); a shared prefix has one set of values that every sharing
    sequence sees;
  * every pool slot that holds no token, including the last block's tail and
    the slots the append is about to fill, holds a NaN bit pattern, so a read
    of an unused slot cannot go unnoticed.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np

BLOCK_SIZE = 16
NAN_BITS = {"bf16": 0x7FC0, "fp16": 0x7E00}
ELEM_BYTES = {"bf16": 2, "fp16": 2}

_CHUNK = 1 << 22  # values drawn per RNG stream chunk (keeps draws independent of threading)


@dataclasses.dataclass
class Workload:
    name: str
    dtype: str
    num_heads: int
    num_kv_heads: int
    head_dim: int
    q_len: int
    block_size: int
    num_blocks: int
    scale: float
    context_lens: np.ndarray          # int32 [N]
    block_tables: np.ndarray          # int32 [N, max_blocks_per_seq], -1 where unused
    query: np.ndarray                 # uint16 [N, q_len, Hq, d]
    key_cache: np.ndarray             # uint16 [NB, B, Hkv, d]  state before the append
    value_cache: np.ndarray           # uint16 [NB, B, Hkv, d]
    new_key: np.ndarray               # uint16 [T, Hkv, d]  rows the append writes
    new_value: np.ndarray             # uint16 [T, Hkv, d]
    slot_mapping: np.ndarray          # int64 [T]
    logical_key: Optional[list] = None    # per sequence uint16 [L_i, Hkv, d] (small cases)
    logical_value: Optional[list] = None
    shared_prefix_blocks: int = 0

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    @property
    def num_new_tokens(self) -> int:
        return int(self.slot_mapping.shape[0])


def _to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """fp32 -> 16-bit storage bits, round to nearest even (library casts)."""
    if dtype == "fp16":
        return x.astype(np.float16).view(np.uint16)
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _normal_bits(seed_seq: np.random.SeedSequence, n: int, dtype: str) -> np.ndarray:
    """n seeded N(0,1) values as 16-bit bits, drawn chunk by chunk from child streams."""
    out = np.empty(n, dtype=np.uint16)
    nchunks = max(1, math.ceil(n / _CHUNK))
    children = seed_seq.spawn(nchunks)
    for c, child in enumerate(children):
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        if hi <= lo:
            break
        g = np.random.Generator(np.random.PCG64(child))
        out[lo:hi] = _to_bits(g.standard_normal(hi - lo, dtype=np.float32), dtype)
    return out


def make_workload(name: str, context_lens: Sequence[int], *, num_heads: int, num_kv_heads: int,
                  head_dim: int, dtype: str = "bf16", q_len: int = 1, append_len: Optional[int] = None,
                  num_blocks: Optional[int] = None, seed: int = 0, shared_prefix_blocks: int = 0,
                  max_blocks_per_seq: Optional[int] = None, keep_logical: bool = False,
                  scale: Optional[float] = None, block_size: int = BLOCK_SIZE) -> Workload:
    """Build one decode step's inputs.

    ``append_len`` (default ``q_len``) newest positions of every sequence are
    left out of the pool and returned as rows for the append step.
    ``shared_prefix_blocks`` > 0 maps the first that many logical blocks of
    every sequence onto the same physical blocks (read-only sharing).
    """
    assert dtype in ("bf16", "fp16")
    lens = np.asarray(context_lens, dtype=np.int64)
    n = int(lens.shape[0])
    append_len = q_len if append_len is None else append_len
    assert np.all(lens >= max(1, q_len, append_len)), "every sequence needs L >= q_len, append_len"
    hkv, d, bs = num_kv_heads, head_dim, block_size
    nblk = (lens + bs - 1) // bs
    if shared_prefix_blocks:
        assert np.all(lens >= shared_prefix_blocks * bs + append_len), "append must land after the prefix"
    private = nblk - shared_prefix_blocks
    need = int(shared_prefix_blocks + private.sum())
    if num_blocks is None:
        num_blocks = need
    assert need <= num_blocks, f"pool of {num_blocks} blocks cannot hold {need}"
    mbps = int(max_blocks_per_seq if max_blocks_per_seq is not None else max(1, int(nblk.max(initial=1))))
    assert mbps >= int(nblk.max(initial=0))

    ss = np.random.SeedSequence(seed)
    s_place, s_q, s_k, s_v = ss.spawn(4)

    # Physical placement: a shuffled free list, popped in sequence order.
    free = np.random.Generator(np.random.PCG64(s_place)).permutation(num_blocks).astype(np.int32)
    shared_ids = free[:shared_prefix_blocks]
    pos = shared_prefix_blocks
    block_tables = np.full((n, mbps), -1, dtype=np.int32)
    for i in range(n):
        block_tables[i, :shared_prefix_blocks] = shared_ids
        k = int(private[i])
        block_tables[i, shared_prefix_blocks:shared_prefix_blocks + k] = free[pos:pos + k]
        pos += k

    row = hkv * d
    # Token contents.  Shared-prefix tokens are drawn once; every other token once per sequence.
    shared_tok = shared_prefix_blocks * bs
    priv_tok = lens - shared_tok
    total_priv = int(priv_tok.sum())
    k_shared = _normal_bits(s_k.spawn(1)[0], shared_tok * row, dtype).reshape(shared_tok, hkv, d)
    v_shared = _normal_bits(s_v.spawn(1)[0], shared_tok * row, dtype).reshape(shared_tok, hkv, d)
    k_priv = _normal_bits(s_k, total_priv * row, dtype).reshape(total_priv, hkv, d)
    v_priv = _normal_bits(s_v, total_priv * row, dtype).reshape(total_priv, hkv, d)
    query = _normal_bits(s_q, n * q_len * num_heads * d, dtype).reshape(n, q_len, num_heads, d)

    # Destination row (block * B + offset) of every logical token, in sequence order.
    seq_of_priv = np.repeat(np.arange(n), priv_tok)
    starts = np.concatenate([[0], np.cumsum(priv_tok)[:-1]]) if n else np.zeros(0, np.int64)
    p_priv = np.arange(total_priv, dtype=np.int64) - np.repeat(starts, priv_tok) + shared_tok
    dest_priv = block_tables[seq_of_priv, p_priv // bs].astype(np.int64) * bs + p_priv % bs
    is_new = p_priv >= np.repeat(lens, priv_tok) - append_len

    sentinel = NAN_BITS[dtype]
    key_cache = np.full((num_blocks * bs, hkv, d), sentinel, dtype=np.uint16)
    value_cache = np.full((num_blocks * bs, hkv, d), sentinel, dtype=np.uint16)
    if shared_tok:
        p_sh = np.arange(shared_tok, dtype=np.int64)
        dest_sh = shared_ids[p_sh // bs].astype(np.int64) * bs + p_sh % bs
        key_cache[dest_sh] = k_shared
        value_cache[dest_sh] = v_shared
    old = ~is_new
    key_cache[dest_priv[old]] = k_priv[old]
    value_cache[dest_priv[old]] = v_priv[old]

    new_key = np.ascontiguousarray(k_priv[is_new])
    new_value = np.ascontiguousarray(v_priv[is_new])
    slot_mapping = dest_priv[is_new].astype(np.int64)

    logical_key = logical_value = None
    if keep_logical:
        logical_key, logical_value = [], []
        for i in range(n):
            a, b = int(starts[i]), int(starts[i] + priv_tok[i])
            logical_key.append(np.concatenate([k_shared, k_priv[a:b]]))
            logical_value.append(np.concatenate([v_shared, v_priv[a:b]]))

    return Workload(
        name=name, dtype=dtype, num_heads=num_heads, num_kv_heads=hkv, head_dim=d, q_len=q_len,
        block_size=bs, num_blocks=num_blocks,
        scale=float(scale if scale is not None else 1.0 / math.sqrt(d)),
        context_lens=lens.astype(np.int32), block_tables=block_tables, query=query,
        key_cache=key_cache.reshape(num_blocks, bs, hkv, d),
        value_cache=value_cache.reshape(num_blocks, bs, hkv, d),
        new_key=new_key, new_value=new_value, slot_mapping=slot_mapping,
        logical_key=logical_key, logical_value=logical_value,
        shared_prefix_blocks=shared_prefix_blocks)


def concat_workloads(name: str, parts: Sequence[Workload]) -> Workload:
    """One batch made of several workloads side by side: their pools laid end to end (block ids
    and slots shifted accordingly), their sequences, queries and appended rows in order.  All
    parts must share dtype, head counts, head dim, q_len and scale.  Used to build batches in
    which several groups of sequences each share a different prefix."""
    first = parts[0]
    for w in parts[1:]:
        assert (w.dtype, w.num_heads, w.num_kv_heads, w.head_dim, w.q_len, w.block_size, w.scale) == \
            (first.dtype, first.num_heads, first.num_kv_heads, first.head_dim, first.q_len, first.block_size,
             first.scale), "parts must share their shapes"
    mbps = max(w.max_blocks_per_seq for w in parts)
    tables, slots, off = [], [], 0
    for w in parts:
        bt = np.full((w.num_seqs, mbps), -1, dtype=np.int32)
        bt[:, :w.max_blocks_per_seq] = np.where(w.block_tables >= 0, w.block_tables + off, -1)
        tables.append(bt)
        slots.append(w.slot_mapping + off * w.block_size)
        off += w.num_blocks
    cat = lambda xs: np.ascontiguousarray(np.concatenate(xs))  # noqa: E731
    return Workload(
        name=name, dtype=first.dtype, num_heads=first.num_heads, num_kv_heads=first.num_kv_heads,
        head_dim=first.head_dim, q_len=first.q_len, block_size=first.block_size, num_blocks=off, scale=first.scale,
        context_lens=cat([w.context_lens for w in parts]), block_tables=cat(tables),
        query=cat([w.query for w in parts]), key_cache=cat([w.key_cache for w in parts]),
        value_cache=cat([w.value_cache for w in parts]), new_key=cat([w.new_key for w in parts]),
        new_value=cat([w.new_value for w in parts]), slot_mapping=cat(slots).astype(np.int64))


# ---------------------------------------------------------------------------
# The five named decode workloads.  Seeds are 2650 + the workload number.
# ---------------------------------------------------------------------------

def _uniform_lens(seed: int, n: int, lo: int, hi: int) -> np.ndarray:
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 7])))
    return g.integers(lo, hi + 1, size=n)


def tiny_mha(**kw) -> Workload:
    """4 sequences, L = {1, 17, 33, 100}, 4 heads MHA, d = 64, bf16, 64-block pool."""
    return make_workload("tiny_mha_d64", [1, 17, 33, 100], num_heads=4, num_kv_heads=4, head_dim=64,
                         dtype="bf16", q_len=1, num_blocks=64, seed=2651, max_blocks_per_seq=8, **kw)


def opt13b_mha(**kw) -> Workload:
    """32 sequences, L ~ U[512, 2048], 40 heads MHA, d = 128, fp16, 8192-block pool."""
    lens = _uniform_lens(2652, 32, 512, 2048)
    return make_workload("opt13b_mha_fp16", lens, num_heads=40, num_kv_heads=40, head_dim=128,
                         dtype="fp16", q_len=1, num_blocks=8192, seed=2652, max_blocks_per_seq=128, **kw)


def gqa_batch128(**kw) -> Workload:
    """128 sequences, L ~ U[1, 4096], GQA 32q/8kv, d = 128, bf16, 40000-block pool."""
    lens = _uniform_lens(2653, 128, 1, 4096)
    return make_workload("gqa_batch128", lens, num_heads=32, num_kv_heads=8, head_dim=128,
                         dtype="bf16", q_len=1, num_blocks=40000, seed=2653, max_blocks_per_seq=256, **kw)


def shared_prefix_verify(**kw) -> Workload:
    """64 sequences sharing a 1024-token prefix (64 blocks) + U[16, 512] private tokens;
    5 query rows per sequence (4 drafts + 1), causal inside the chunk; GQA 32/8, d = 128."""
    suffix = _uniform_lens(2654, 64, 16, 512)
    return make_workload("shared_prefix_spec5", 1024 + suffix, num_heads=32, num_kv_heads=8,
                         head_dim=128, dtype="bf16", q_len=5, num_blocks=4096, seed=2654,
                         shared_prefix_blocks=64, max_blocks_per_seq=96, **kw)


def long_context_skewed(**kw) -> Workload:
    """16 sequences L ~ U[16384, 32768] + 240 sequences L ~ U[64, 1024], shuffled;
    GQA 64q/8kv, d = 128, bf16, 65536-block pool."""
    long_ = _uniform_lens(2655, 16, 16384, 32768)
    short = _uniform_lens(2655 + 100, 240, 64, 1024)
    lens = np.concatenate([long_, short])
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([2655, 11])))
    lens = lens[g.permutation(lens.shape[0])]
    return make_workload("long_context_skewed", lens, num_heads=64, num_kv_heads=8, head_dim=128,
                         dtype="bf16", q_len=1, num_blocks=65536, seed=2655, max_blocks_per_seq=2048, **kw)


def gqa_batch32(**kw) -> Workload:
    """Profiling-size member of the GQA family: 32 sequences, L ~ U[1, 4096], GQA 32q/8kv, d = 128,
    bf16, 10000-block pool (about 0.25 GB of K/V per step: still larger than L2)."""
    lens = _uniform_lens(2663, 32, 1, 4096)
    return make_workload("gqa_batch32", lens, num_heads=32, num_kv_heads=8, head_dim=128,
                         dtype="bf16", q_len=1, num_blocks=10000, seed=2663, max_blocks_per_seq=256, **kw)


def chunked_prefill(**kw) -> Workload:
    """Chunked prefill over the paged cache: 16 sequences, each with U[1024, 4096] tokens of
    history and a 256-token prompt chunk (256 query rows, causal inside the chunk, appended
    first); GQA 32q/8kv, d = 128, bf16, 5000-block pool."""
    hist = _uniform_lens(2666, 16, 1024, 4096)
    return make_workload("chunked_prefill_256", hist + 256, num_heads=32, num_kv_heads=8, head_dim=128,
                         dtype="bf16", q_len=256, num_blocks=5000, seed=2666, max_blocks_per_seq=272, **kw)


WORKLOADS = {
    1: tiny_mha,
    2: opt13b_mha,
    3: gqa_batch128,
    4: shared_prefix_verify,
    5: long_context_skewed,
    6: gqa_batch32,
    7: chunked_prefill,
}


@dataclasses.dataclass
class SpecInputs:
    """Inputs of one speculative-verification step: the target model's distributions at the
    k draft positions plus one, the draft model's distributions and sampled draft tokens, and
    the uniforms the accept/reject rule and the final draw consume."""
    target_probs: np.ndarray   # f32 [N, k+1, V]
    draft_probs: np.ndarray    # f32 [N, k, V]
    draft_tokens: np.ndarray   # i32 [N, k]
    u_accept: np.ndarray       # f32 [N, k]
    u_sample: np.ndarray       # f32 [N]


def spec_verify_inputs(num_seqs: int = 64, k: int = 4, vocab: int = 32000, seed: int = 2664,
                       draft_temp: float = 1.0, noise: float = 1.0) -> SpecInputs:
    """Synthetic model outputs: draft logits ~ N(0, 2^2) per token; target logits = draft logits
    + N(0, noise^2), so the two models agree partly; both turned into distributions by a
    softmax; draft tokens are drawn from the draft distributions; uniforms in [0, 1)."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed)))
    dl = g.normal(0.0, 2.0, size=(num_seqs, k + 1, vocab))
    tl = dl + g.normal(0.0, noise, size=dl.shape)

    def softmax(x):
        e = np.exp(x - x.max(axis=-1, keepdims=True))
        return e / e.sum(axis=-1, keepdims=True)

    target = softmax(tl).astype(np.float32)
    draft = softmax(dl[:, :k] / draft_temp).astype(np.float32)
    cdf = np.cumsum(draft.astype(np.float64), axis=-1)
    r = g.random((num_seqs, k, 1)) * cdf[..., -1:]
    tokens = np.minimum((cdf < r).sum(axis=-1), vocab - 1).astype(np.int32)
    return SpecInputs(target_probs=target, draft_probs=draft, draft_tokens=tokens,
                      u_accept=g.random((num_seqs, k), dtype=np.float32),
                      u_sample=g.random(num_seqs, dtype=np.float32))


def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    """Logical KV bytes one token occupies: 2 (K and V) x layers x kv heads x head dim x bytes.

    The formula of "LLM 推理优化的系统视角", section 3.2."""
    return 2 * num_layers * num_kv_heads * head_dim * elem_bytes


def block_bytes(block_size: int, num_kv_heads: int, head_size: int, elem_bytes: int) -> int:
    """Bytes of one KV block of one layer: 2 x block_size x kv heads x head size x bytes.

    The formula of "现代 LLM 推理引擎剖析", section 1.3."""
    return 2 * block_size * num_kv_heads * head_size * elem_bytes


def attention_bytes(w: Workload, kv_elem_bytes: Optional[int] = None) -> int:
    """Algorithmic HBM bytes of one decode-attention pass: each sequence's K and V rows
    (all L_i positions, every kv head) once, plus Q read and O written once.
    kv_elem_bytes overrides the cache element size (1 for an FP8 cache)."""
    e = ELEM_BYTES[w.dtype]
    kve = e if kv_elem_bytes is None else kv_elem_bytes
    kv = int(w.context_lens.astype(np.int64).sum()) * kv_bytes_per_token(1, w.num_kv_heads, w.head_dim, kve)
    qo = 2 * w.num_seqs * w.q_len * w.num_heads * w.head_dim * e
    return kv + qo


def unique_attention_bytes(w: Workload, kv_elem_bytes: Optional[int] = None) -> int:
    """HBM bytes of one attention pass if every physical block were read once: blocks that
    several sequences map (a shared prefix) count once, with the most rows any sequence uses
    from them, plus Q read and O written.  Equals attention_bytes when nothing is shared."""
    e = ELEM_BYTES[w.dtype]
    kve = e if kv_elem_bytes is None else kv_elem_bytes
    rows = {}
    for i in range(w.num_seqs):
        L = int(w.context_lens[i])
        for b in range((L + w.block_size - 1) // w.block_size):
            pb = int(w.block_tables[i, b])
            rows[pb] = max(rows.get(pb, 0), min(w.block_size, L - w.block_size * b))
    kv = sum(rows.values()) * kv_bytes_per_token(1, w.num_kv_heads, w.head_dim, kve)
    qo = 2 * w.num_seqs * w.q_len * w.num_heads * w.head_dim * e
    return kv + qo


def attention_flops(w: Workload) -> int:
    """Algorithmic flops of one attention pass: for every query row and head, 2 d flops for the
    score and 2 d for the P.V term of each position the row attends (row j of a q-row chunk
    attends L - q + j + 1 positions)."""
    lens = w.context_lens.astype(np.int64)
    q = w.q_len
    visible = int((q * (lens - q) + q * (q + 1) // 2).sum())
    return 4 * w.head_dim * w.num_heads * visible


def append_bytes(w: Workload, kv_elem_bytes: Optional[int] = None) -> int:
    """Algorithmic bytes of the KV append: each new K and V row read once (16-bit) and written
    once (kv_elem_bytes, default the input's)."""
    e = ELEM_BYTES[w.dtype]
    kve = e if kv_elem_bytes is None else kv_elem_bytes
    return w.num_new_tokens * (kv_bytes_per_token(1, w.num_kv_heads, w.head_dim, e) +
                               kv_bytes_per_token(1, w.num_kv_heads, w.head_dim, kve))
