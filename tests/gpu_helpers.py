"""Shared plumbing of the GPU parity tests: upload a workload, run one decode step
through the C ABI (append, then attention), run the oracle on the same inputs,
and compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_kv_cache_265_gb300 import pa
from paged_kv_cache_265_gb300 import workload as W

TORCH_DT = {"bf16": torch.bfloat16, "fp16": torch.float16}

# Attention tolerance: an element passes when |gpu - oracle| <= ABS_TOL or
# |gpu - oracle| <= REL_TOL * |oracle|.
ABS_TOL = 2e-3
REL_TOL = 1e-2


def to_dev(bits: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(TORCH_DT[dtype])


def to_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bits_to_f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "fp16":
        return bits.view(np.float16).astype(np.float64)
    return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()


class GpuStep:
    """Device copies of one workload's inputs; runs the append and the attention."""

    def __init__(self, w: W.Workload, partition_size: int = 0):
        self.w = w
        self.partition_size = partition_size
        dt = w.dtype
        self.key_cache = to_dev(w.key_cache, dt)
        self.value_cache = to_dev(w.value_cache, dt)
        self.new_key = to_dev(w.new_key, dt)
        self.new_value = to_dev(w.new_value, dt)
        self.slot_mapping = torch.from_numpy(w.slot_mapping).cuda()
        self.block_tables = torch.from_numpy(w.block_tables).cuda()
        self.context_lens = torch.from_numpy(w.context_lens).cuda()
        self.query = to_dev(w.query, dt)
        self.out = torch.empty_like(self.query)
        self.workspace = pa.alloc_workspace(w.num_seqs, w.q_len, w.num_heads, w.head_dim, w.max_context_len,
                                            partition_size)

    def append(self):
        pa.reshape_and_cache(self.new_key, self.new_value, self.key_cache, self.value_cache, self.slot_mapping)

    def attend(self) -> torch.Tensor:
        pa.decode_attention(self.out, self.query, self.key_cache, self.value_cache, self.block_tables,
                            self.context_lens, self.w.scale, self.w.max_context_len, self.workspace,
                            partition_size=self.partition_size)
        return self.out

    def run(self) -> np.ndarray:
        self.append()
        self.attend()
        torch.cuda.synchronize()
        return to_bits(self.out)


def oracle_step(w: W.Workload, threads: int = 0):
    """Oracle append on host copies of the pools, then oracle attention on the result."""
    orc = oracle.load()
    kc, vc = w.key_cache.copy(), w.value_cache.copy()
    bad = orc.reshape_and_cache(w.new_key, w.new_value, kc, vc, w.slot_mapping)
    assert bad == 0
    out, bad = orc.decode_attention(w.query, kc, vc, w.block_tables, w.context_lens, w.scale, w.dtype,
                                    num_threads=threads)
    assert bad == 0
    return kc, vc, out


def compare(gpu_bits: np.ndarray, ref: np.ndarray, dtype: str, what: str = ""):
    """Asserts the attention tolerance element by element; returns (max_abs, max_rel)."""
    g = bits_to_f64(gpu_bits, dtype).reshape(ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    err = np.abs(g - ref)
    rel = err / np.maximum(np.abs(ref), 1e-30)
    ok = (err <= ABS_TOL) | (rel <= REL_TOL)
    if not np.all(ok):
        i = np.unravel_index(np.argmax(np.where(ok, 0, err)), err.shape)
        raise AssertionError(f"{what}: {np.count_nonzero(~ok)} elements out of tolerance; worst at {i}: "
                             f"gpu {g[i]!r} oracle {ref[i]!r}")
    return float(err.max(initial=0.0)), float(np.where(err > ABS_TOL, rel, 0.0).max(initial=0.0))


def ulps_from_rounded_oracle(gpu_bits: np.ndarray, ref: np.ndarray, dtype: str, floor: float = 2.0 ** -6) -> int:
    """Largest distance, in units in the last place of the 16-bit type, between the GPU output
    and the oracle rounded once to that type (round to nearest even, library cast), over the
    elements with |oracle| >= floor (below it, cancellation makes the last place meaningless;
    the absolute tolerance covers those)."""
    if dtype == "fp16":
        rb = ref.astype(np.float16).view(np.uint16)
    else:
        rb = torch.from_numpy(ref).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    g = gpu_bits.reshape(ref.shape).astype(np.int64)
    r = rb.astype(np.int64)
    # map sign-magnitude bit patterns onto a monotone integer line
    g = np.where(g & 0x8000, 0x8000 - g, g)
    r = np.where(r & 0x8000, 0x8000 - r, r)
    big = np.abs(ref) >= floor
    return int(np.abs(g - r)[big].max(initial=0))


def from_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round to the 16-bit type (nearest even) and return the bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64)).to(TORCH_DT[dtype])
    return t.view(torch.int16).numpy().view(np.uint16)


def rising_scores_workload(dtype: str, seed: int = 77, gain: float = 8.0) -> W.Workload:
    """A GQA 32/8, d = 128 batch whose scores move steadily instead of staying in a narrow band,
    so that an online softmax keeps meeting scores above its running max.  Every key is a small
    random part plus a(p) times the unit direction of the sum of its kv head's query rows, and the
    queries are scaled by `gain`.  a(p), per sequence: rising from -10 to 10 over 3000 positions
    (scores from about -42..-63 to +42..+63 in log2 units, +0.3..0.5 per block: every query row's
    max passes the previous one by more than 8 on 10-18 blocks, with weights up to nearly 2^8
    against the old max in between), falling from 10 to -10 over 1700 (the first block holds the
    max; later weights underflow), a step from -10 to 10 at position 407 of 650 (a jump of 68-148
    inside a block, after 25 blocks), and rising over 40.  The gain keeps |scores| below 90: at
    gain 41 (|scores| up to 220) the fp32 rounding of the scores alone moves fp16 outputs by up
    to 1.4e-3 relative, more than one unit in the last place."""
    lens = [3000, 1700, 650, 40]
    hq, hkv, d = 32, 8, 128
    g = hq // hkv
    w = W.make_workload(f"rising_{dtype}", lens, num_heads=hq, num_kv_heads=hkv, head_dim=d, dtype=dtype,
                        q_len=1, seed=seed, keep_logical=True)
    q = bits_to_f64(w.query.ravel(), dtype).reshape(w.query.shape) * gain
    qbits = from_f64(q, dtype).reshape(w.query.shape)
    q = bits_to_f64(qbits.ravel(), dtype).reshape(w.query.shape)
    key_cache = w.key_cache.reshape(-1, hkv, d).copy()
    new_key = w.new_key.copy()
    for i, L in enumerate(lens):
        p = np.arange(L, dtype=np.float64)
        if i == 0 or i == 3:
            a = -10.0 + 20.0 * p / (L - 1)
        elif i == 1:
            a = 10.0 - 20.0 * p / (L - 1)
        else:
            a = np.where(p < 407, -10.0, 10.0)
        u = q[i, 0].reshape(hkv, g, d).sum(axis=1)
        u /= np.linalg.norm(u, axis=1, keepdims=True)
        k = 0.05 * bits_to_f64(w.logical_key[i].ravel(), dtype).reshape(L, hkv, d) + a[:, None, None] * u[None]
        kb = from_f64(k, dtype).reshape(L, hkv, d)
        slots = w.block_tables[i, np.arange(L) // w.block_size].astype(np.int64) * w.block_size + np.arange(L) % w.block_size
        key_cache[slots[:L - 1]] = kb[:L - 1]
        new_key[i] = kb[L - 1]
    assert np.array_equal(w.slot_mapping, [w.block_tables[i, (L - 1) // w.block_size] * w.block_size
                                           + (L - 1) % w.block_size for i, L in enumerate(lens)])
    import dataclasses
    return dataclasses.replace(w, query=qbits, key_cache=key_cache.reshape(w.key_cache.shape), new_key=new_key,
                               logical_key=None, logical_value=None)
