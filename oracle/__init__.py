"""fp64 CPU oracle for paged-KV decode attention and the KV append.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(the CUDA library and its Python binding) never imports it and shares no code
with it; both sides are fed by the seeded generator in
``paged_kv_cache_265_gb300.workload``, which holds none of the arithmetic.

The arithmetic lives in ``pa_oracle.c`` (plain C loops, fp64); this module only
compiles it with gcc and marshals numpy arrays.  See that file's header for the
passages of the pages each step follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_CACHE: dict[int, "Oracle"] = {}

DTYPES = {"bf16": 0, "fp16": 1}


def lib_path(plant: int = 0) -> str:
    name = "libpa_oracle.so" if plant == 0 else f"libpa_oracle_plant{plant}.so"
    return os.path.join(_BUILD, name)


def build(plant: int = 0, force: bool = False) -> str:
    """Compile the oracle (or a planted-mistake variant) with gcc; return the .so path."""
    out = lib_path(plant)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    tmp = f"{out}.{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", "-Wall", "-o", tmp, _SRC, "-lm"]
    if plant:
        cmd.insert(1, f"-DPLANT={plant}")
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_f64p = ctypes.POINTER(ctypes.c_double)


def _ptr(a: np.ndarray, t):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(t)


class Oracle:
    """ctypes handle on one build of ``pa_oracle.c``."""

    def __init__(self, path: str):
        self.path = path
        lib = ctypes.CDLL(path)
        lib.oracle_decode_attention.restype = ctypes.c_int
        lib.oracle_decode_attention.argtypes = [
            _f64p, _u16p, _u16p, _u16p, _i32p, ctypes.c_int, _i32p, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_double,
            ctypes.c_int, ctypes.c_int,
        ]
        _f32p = ctypes.POINTER(ctypes.c_float)
        lib.oracle_reshape_and_cache.restype = ctypes.c_int
        lib.oracle_reshape_and_cache.argtypes = [
            _u16p, _u16p, _u16p, _u16p, _i64p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int64,
        ]
        lib.oracle_copy_blocks.restype = ctypes.c_int
        lib.oracle_copy_blocks.argtypes = [_u16p, _u16p, _i64p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int64]
        _f32p = ctypes.POINTER(ctypes.c_float)
        lib.oracle_spec_verify.restype = ctypes.c_int
        lib.oracle_spec_verify.argtypes = [_i32p, _i32p, _f32p, _f32p, _i32p, _f32p, _f32p, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int]
        _u8p = ctypes.POINTER(ctypes.c_uint8)
        lib.oracle_e4m3_encode_vec.restype = None
        lib.oracle_e4m3_encode_vec.argtypes = [_f32p, ctypes.c_int64, _u8p]
        lib.oracle_e4m3_decode_vec.restype = None
        lib.oracle_e4m3_decode_vec.argtypes = [_u8p, ctypes.c_int64, _f64p]
        lib.oracle_reshape_and_cache_fp8.restype = ctypes.c_int
        lib.oracle_reshape_and_cache_fp8.argtypes = [_u16p, _u16p, _u8p, _u8p, _i64p, ctypes.c_int64, ctypes.c_int,
                                                     ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                                     ctypes.c_float, ctypes.c_float]
        lib.oracle_decode_attention_fp8.restype = ctypes.c_int
        lib.oracle_decode_attention_fp8.argtypes = [
            _f64p, _u16p, _u8p, _u8p, _i32p, ctypes.c_int, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_int,
            ctypes.c_float, ctypes.c_float, ctypes.c_int]
        lib.oracle_bits_to_double_vec.restype = None
        lib.oracle_bits_to_double_vec.argtypes = [_u16p, ctypes.c_int64, ctypes.c_int, _f64p]
        lib.oracle_max_threads.restype = ctypes.c_int
        self._lib = lib

    def max_threads(self) -> int:
        return int(self._lib.oracle_max_threads())

    def bits_to_double(self, bits: np.ndarray, dtype: str) -> np.ndarray:
        b = np.ascontiguousarray(bits, dtype=np.uint16)
        out = np.empty(b.shape, dtype=np.float64)
        self._lib.oracle_bits_to_double_vec(_ptr(b, _u16p), b.size, DTYPES[dtype], _ptr(out, _f64p))
        return out

    def decode_attention(self, query, key_cache, value_cache, block_tables, context_lens,
                         scale: float, dtype: str, num_threads: int = 0):
        """Returns (out fp64 [N, q_len, Hq, d], number of invalid sequences).

        query [N, q_len, Hq, d] uint16 bits; caches [NB, B, Hkv, d] uint16 bits;
        block_tables [N, max_blocks] int32; context_lens [N] int32.
        """
        q = np.ascontiguousarray(query, dtype=np.uint16)
        kc = np.ascontiguousarray(key_cache, dtype=np.uint16)
        vc = np.ascontiguousarray(value_cache, dtype=np.uint16)
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        n, q_len, hq, d = q.shape
        nb, bs, hkv, d2 = kc.shape
        assert d2 == d and vc.shape == kc.shape and bt.shape[0] == n and cl.shape == (n,)
        out = np.empty((n, q_len, hq, d), dtype=np.float64)
        bad = self._lib.oracle_decode_attention(
            _ptr(out, _f64p), _ptr(q, _u16p), _ptr(kc, _u16p), _ptr(vc, _u16p), _ptr(bt, _i32p),
            bt.shape[1], _ptr(cl, _i32p), n, q_len, hq, hkv, d, bs, nb, float(scale),
            DTYPES[dtype], int(num_threads))
        return out, int(bad)

    def reshape_and_cache(self, key, value, key_cache, value_cache, slot_mapping) -> int:
        """Writes new K/V rows into the caches IN PLACE; returns the count of out-of-pool slots."""
        k = np.ascontiguousarray(key, dtype=np.uint16)
        v = np.ascontiguousarray(value, dtype=np.uint16)
        sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        assert key_cache.flags["C_CONTIGUOUS"] and value_cache.flags["C_CONTIGUOUS"]
        assert key_cache.dtype == np.uint16 and value_cache.dtype == np.uint16
        nb, bs, hkv, d = key_cache.shape
        t = sm.shape[0]
        assert k.shape == (t, hkv, d) and v.shape == (t, hkv, d)
        return int(self._lib.oracle_reshape_and_cache(
            _ptr(k, _u16p), _ptr(v, _u16p), _ptr(key_cache, _u16p), _ptr(value_cache, _u16p),
            _ptr(sm, _i64p), t, hkv, d, bs, nb))


    def copy_blocks(self, key_cache, value_cache, block_mapping) -> int:
        """Copy-on-write block copies IN PLACE; returns the count of pairs with an id outside the pool."""
        bm = np.ascontiguousarray(block_mapping, dtype=np.int64).reshape(-1, 2)
        assert key_cache.flags["C_CONTIGUOUS"] and value_cache.flags["C_CONTIGUOUS"]
        nb, bs, hkv, d = key_cache.shape
        return int(self._lib.oracle_copy_blocks(_ptr(key_cache, _u16p), _ptr(value_cache, _u16p),
                                                _ptr(bm, _i64p), bm.shape[0], hkv, d, bs, nb))


    def spec_verify(self, target_probs, draft_probs, draft_tokens, u_accept, u_sample):
        """Speculative-decoding verification.  target [N, k+1, V] f32, draft [N, k, V] f32,
        draft_tokens [N, k] i32, u_accept [N, k] f32, u_sample [N] f32.
        Returns (num_accepted [N] i32, out_tokens [N, k+1] i32)."""
        f32p = ctypes.POINTER(ctypes.c_float)
        tp = np.ascontiguousarray(target_probs, dtype=np.float32)
        dp = np.ascontiguousarray(draft_probs, dtype=np.float32)
        dt = np.ascontiguousarray(draft_tokens, dtype=np.int32)
        ua = np.ascontiguousarray(u_accept, dtype=np.float32)
        us = np.ascontiguousarray(u_sample, dtype=np.float32)
        n, k1, v = tp.shape
        k = k1 - 1
        assert dp.shape == (n, k, v) and dt.shape == (n, k) and ua.shape == (n, k) and us.shape == (n,)
        acc = np.empty(n, np.int32)
        out = np.empty((n, k1), np.int32)
        self._lib.oracle_spec_verify(_ptr(acc, _i32p), _ptr(out, _i32p), _ptr(tp, f32p), _ptr(dp, f32p),
                                     _ptr(dt, _i32p), _ptr(ua, f32p), _ptr(us, f32p), n, k, v)
        return acc, out


    def e4m3_encode(self, x) -> np.ndarray:
        a = np.ascontiguousarray(x, dtype=np.float32)
        out = np.empty(a.shape, np.uint8)
        self._lib.oracle_e4m3_encode_vec(_ptr(a, ctypes.POINTER(ctypes.c_float)), a.size,
                                         _ptr(out, ctypes.POINTER(ctypes.c_uint8)))
        return out

    def e4m3_decode(self, b) -> np.ndarray:
        a = np.ascontiguousarray(b, dtype=np.uint8)
        out = np.empty(a.shape, np.float64)
        self._lib.oracle_e4m3_decode_vec(_ptr(a, ctypes.POINTER(ctypes.c_uint8)), a.size, _ptr(out, _f64p))
        return out

    def reshape_and_cache_fp8(self, key, value, key_cache, value_cache, slot_mapping, dtype: str,
                              k_scale: float, v_scale: float) -> int:
        """Quantising append into uint8 (e4m3) caches, IN PLACE."""
        u8p = ctypes.POINTER(ctypes.c_uint8)
        k = np.ascontiguousarray(key, dtype=np.uint16)
        v = np.ascontiguousarray(value, dtype=np.uint16)
        sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        assert key_cache.dtype == np.uint8 and key_cache.flags["C_CONTIGUOUS"] and value_cache.flags["C_CONTIGUOUS"]
        nb, bs, hkv, d = key_cache.shape
        return int(self._lib.oracle_reshape_and_cache_fp8(
            _ptr(k, _u16p), _ptr(v, _u16p), _ptr(key_cache, u8p), _ptr(value_cache, u8p), _ptr(sm, _i64p),
            sm.shape[0], hkv, d, bs, nb, DTYPES[dtype], float(k_scale), float(v_scale)))

    def decode_attention_fp8(self, query, key_cache, value_cache, block_tables, context_lens, scale: float,
                             dtype: str, k_scale: float, v_scale: float, num_threads: int = 0):
        """Attention over uint8 (e4m3) caches; query 16-bit bits of `dtype`.  Returns (out fp64, bad)."""
        u8p = ctypes.POINTER(ctypes.c_uint8)
        q = np.ascontiguousarray(query, dtype=np.uint16)
        kc = np.ascontiguousarray(key_cache, dtype=np.uint8)
        vc = np.ascontiguousarray(value_cache, dtype=np.uint8)
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        n, q_len, hq, d = q.shape
        nb, bs, hkv, _ = kc.shape
        out = np.empty((n, q_len, hq, d), dtype=np.float64)
        bad = self._lib.oracle_decode_attention_fp8(
            _ptr(out, _f64p), _ptr(q, _u16p), _ptr(kc, u8p), _ptr(vc, u8p), _ptr(bt, _i32p), bt.shape[1],
            _ptr(cl, _i32p), n, q_len, hq, hkv, d, bs, nb, float(scale), DTYPES[dtype], float(k_scale),
            float(v_scale), int(num_threads))
        return out, int(bad)


def load(plant: int = 0) -> Oracle:
    """Build (if needed) and load the oracle; ``plant`` > 0 loads a planted-mistake variant."""
    with _LOCK:
        if plant not in _CACHE:
            _CACHE[plant] = Oracle(build(plant))
        return _CACHE[plant]
