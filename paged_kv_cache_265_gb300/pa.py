"""Python binding of libpa.so (ctypes).  Argument marshalling only: every step of
the decode path runs in the library's CUDA kernels.

Tensors are torch CUDA tensors (PyTorch supplies device memory and streams);
their data pointers and the current CUDA stream are handed to the C ABI
declared in ``include/pa.h``.  A missing library raises instead of falling
back to anything else.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpa.so")

PA_BF16, PA_FP16 = 0, 1
PA_DEVERR_BLOCK_ID, PA_DEVERR_CONTEXT, PA_DEVERR_SLOT, PA_DEVERR_TIMEOUT, PA_DEVERR_INTERNAL = 1, 2, 4, 8, 16
PA_DEVERR_TOKEN = 32
PA_DEVERR_QUERY_RANGE = 64
BLOCK_SIZE = 16
DEFAULT_PARTITION = 512
NOALLOC_WORKSPACE_BYTES = 32 << 20
MAX_PREFIX_GROUPS = 256

_DT = {torch.bfloat16: PA_BF16, torch.float16: PA_FP16}

_c_int, _c_i64, _c_sz, _c_f, _vp = ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float, ctypes.c_void_p

_SIGS = {
    "pa_reshape_and_cache": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_i64, _c_int, _c_int, _c_int, _c_i64, _c_int, _vp]),
    "pa_spec_verify": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _vp]),
    "pa_reshape_and_cache_fp8": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_i64, _c_int, _c_int, _c_int, _c_i64, _c_int,
                                          _c_f, _c_f, _vp]),
    "pa_decode_attention_fp8kv": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _vp, _c_int, _c_int, _c_int, _c_int,
                                           _c_int, _c_int, _c_i64, _c_int, _c_f, _c_int, _c_f, _c_f, _c_int, _vp,
                                           _c_sz, _vp]),
    "pa_copy_blocks": (_c_int, [_vp, _vp, _vp, _c_i64, _c_int, _c_int, _c_int, _c_i64, _c_int, _vp]),
    "pa_decode_workspace_size": (_c_sz, [_c_int, _c_int, _c_int, _c_int, _c_int]),
    "pa_decode_workspace_size_ex": (_c_sz, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int]),
    "pa_decode_attention": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _vp, _c_int, _c_int, _c_int, _c_int, _c_int,
                                     _c_i64, _c_int, _c_f, _c_int, _vp, _c_sz, _vp]),
    "pa_decode_attention_multiquery": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _vp, _c_int, _c_int, _c_int,
                                                _c_int, _c_int, _c_int, _c_i64, _c_int, _c_f, _c_int, _vp, _c_sz,
                                                _vp]),
    "pa_decode_attention_ex": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _vp, _c_int, _c_int, _c_int, _c_int,
                                        _c_int, _c_int, _c_i64, _c_int, _c_f, _c_int, _c_int, _vp, _c_sz, _vp]),
    "pa_decode_attention_noalloc": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _vp, _c_int, _c_int, _c_int, _c_int,
                                             _c_int, _c_int, _c_i64, _c_int, _c_f, _c_int, _c_int, _vp]),
    "pa_decode_workspace_size_shared_prefix": (_c_sz, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int]),
    "pa_decode_attention_shared_prefix": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _vp, _c_int, _c_int, _c_int,
                                                   _c_int, _c_int, _c_int, _c_i64, _c_int, _c_f, _c_int, _c_int,
                                                   _vp, _vp, _c_int, _vp, _c_sz, _vp]),
    "pa_status_string": (ctypes.c_char_p, [_c_int]),
    "pa_get_device_error": (_c_int, [ctypes.POINTER(ctypes.c_int32), _c_int, _vp]),
    "pa_set_decode_math": (_c_int, [_c_int]),
    "pa_profile_enable": (_c_int, [_c_int]),
    "pa_profile_read": (_c_int, [ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int)]),
    "pa_profile_read_parts": (_c_int, [ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_float),
                                       ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int)]),
    "pa_set_wait_limit_ns": (_c_int, [ctypes.c_ulonglong]),
    "pa_last_launch_count": (_c_int, []),
    "pa_last_partition_size": (_c_int, []),
    "pa_version": (_c_int, []),
}

_lib: Optional[ctypes.CDLL] = None


class PaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status_string(status)} (status {status})")
        self.status = status


def lib() -> ctypes.CDLL:
    """Load libpa.so (built in-tree by ``paged_kv_cache_265_gb300.build``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libpa.so is not built ({LIB_PATH}); run paged_kv_cache_265_gb300.build.build()")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def status_string(status: int) -> str:
    return lib().pa_status_string(int(status)).decode()


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise PaError(fn, status)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


@contextlib.contextmanager
def _device_of(*tensors, stream=None):
    """Run a library call with the CUDA device of its tensors current: the library launches on
    the current device, so every tensor (and an explicit stream) must be on that one device."""
    devs = set()
    for t in tensors:
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError("arguments must be CUDA tensors")
        devs.add(t.device)
    if len(devs) != 1:
        raise ValueError(f"all tensors must be on one CUDA device (got {sorted(str(d) for d in devs)})")
    dev = devs.pop()
    if stream is not None and getattr(stream, "device", dev) != dev:
        raise ValueError(f"the stream is on {stream.device}, the tensors on {dev}")
    with torch.cuda.device(dev):
        yield


def _dev(t: torch.Tensor, name: str) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in _DT:
        raise ValueError(f"unsupported dtype {t.dtype}; use bfloat16 or float16")
    return _DT[t.dtype]


def reshape_and_cache(key: torch.Tensor, value: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
                      slot_mapping: torch.Tensor, stream=None) -> None:
    """Append new K/V rows ([T, Hkv, d]) into the paged caches ([NB, 16, Hkv, d]) at slot_mapping (int64 [T])."""
    nb, bs, hkv, d = key_cache.shape
    if key.shape != (slot_mapping.shape[0], hkv, d) or value.shape != key.shape:
        raise ValueError("key/value must be [num_tokens, num_kv_heads, head_dim]")
    if slot_mapping.dtype != torch.int64:
        raise ValueError("slot_mapping must be int64")
    if key.dtype != key_cache.dtype or value.dtype != key_cache.dtype or value_cache.dtype != key_cache.dtype:
        raise ValueError("key, value and the caches must share one dtype")
    with _device_of(key, value, key_cache, value_cache, slot_mapping, stream=stream):
        st = lib().pa_reshape_and_cache(
            _dev(key, "key"), _dev(value, "value"), _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache"),
            _dev(slot_mapping, "slot_mapping"), slot_mapping.shape[0], hkv, d, bs, nb, dtype_code(key_cache),
            _stream(stream))
    _check("pa_reshape_and_cache", st)


def copy_blocks(key_cache: torch.Tensor, value_cache: torch.Tensor, block_mapping: torch.Tensor,
                stream=None) -> None:
    """Copy-on-write: for each (src, dst) row of block_mapping (int64 [M, 2]) copy the whole K and V
    block src to dst.  dst blocks must be distinct and not sources of the same call."""
    nb, bs, hkv, d = key_cache.shape
    if value_cache.shape != key_cache.shape or value_cache.dtype != key_cache.dtype:
        raise ValueError("key_cache and value_cache must match")
    if block_mapping.dtype != torch.int64 or block_mapping.dim() != 2 or block_mapping.shape[1] != 2:
        raise ValueError("block_mapping must be int64 [num_pairs, 2]")
    with _device_of(key_cache, value_cache, block_mapping, stream=stream):
        st = lib().pa_copy_blocks(_dev(key_cache, "key_cache"), _dev(value_cache, "value_cache"),
                                  _dev(block_mapping, "block_mapping"), block_mapping.shape[0], hkv, d, bs, nb,
                                  dtype_code(key_cache), _stream(stream))
    _check("pa_copy_blocks", st)


def spec_verify(target_probs: torch.Tensor, draft_probs: torch.Tensor, draft_tokens: torch.Tensor,
                u_accept: torch.Tensor, u_sample: torch.Tensor, num_accepted: torch.Tensor = None,
                out_tokens: torch.Tensor = None, stream=None):
    """Speculative-decoding verification.  target [N, k+1, V] f32, draft [N, k, V] f32,
    draft_tokens [N, k] i32, u_accept [N, k] f32, u_sample [N] f32.
    Returns (num_accepted [N] i32, out_tokens [N, k+1] i32)."""
    n, k1, v = target_probs.shape
    k = k1 - 1
    if target_probs.dtype != torch.float32 or draft_probs.dtype != torch.float32:
        raise ValueError("probabilities must be float32")
    if draft_probs.shape != (n, k, v) or draft_tokens.shape != (n, k) or draft_tokens.dtype != torch.int32:
        raise ValueError("draft shapes/dtypes")
    if u_accept.shape != (n, k) or u_sample.shape != (n,):
        raise ValueError("uniform shapes")
    if num_accepted is None:
        num_accepted = torch.empty(n, dtype=torch.int32, device=target_probs.device)
    if out_tokens is None:
        out_tokens = torch.empty((n, k1), dtype=torch.int32, device=target_probs.device)
    with _device_of(num_accepted, out_tokens, target_probs, draft_probs, draft_tokens, u_accept, u_sample, stream=stream):
        st = lib().pa_spec_verify(_dev(num_accepted, "num_accepted"), _dev(out_tokens, "out_tokens"),
                                  _dev(target_probs, "target_probs"), _dev(draft_probs, "draft_probs"),
                                  _dev(draft_tokens, "draft_tokens"), _dev(u_accept, "u_accept"),
                                  _dev(u_sample, "u_sample"), n, k, v, _stream(stream))
    _check("pa_spec_verify", st)
    return num_accepted, out_tokens


def reshape_and_cache_fp8(key: torch.Tensor, value: torch.Tensor, key_cache: torch.Tensor,
                         value_cache: torch.Tensor, slot_mapping: torch.Tensor, k_scale: float, v_scale: float,
                         stream=None) -> None:
    """Quantising append: 16-bit K/V rows [T, Hkv, d] into uint8 (FP8 E4M3) caches [NB, 16, Hkv, d]."""
    nb, bs, hkv, d = key_cache.shape
    if key_cache.dtype != torch.uint8 or value_cache.dtype != torch.uint8 or value_cache.shape != key_cache.shape:
        raise ValueError("FP8 caches must be uint8 tensors of one shape")
    if key.shape != (slot_mapping.shape[0], hkv, d) or value.shape != key.shape or slot_mapping.dtype != torch.int64:
        raise ValueError("key/value must be [num_tokens, num_kv_heads, head_dim]; slot_mapping int64")
    with _device_of(key, value, key_cache, value_cache, slot_mapping, stream=stream):
        st = lib().pa_reshape_and_cache_fp8(
            _dev(key, "key"), _dev(value, "value"), _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache"),
            _dev(slot_mapping, "slot_mapping"), slot_mapping.shape[0], hkv, d, bs, nb, dtype_code(key), float(k_scale),
            float(v_scale), _stream(stream))
    _check("pa_reshape_and_cache_fp8", st)


def decode_attention_fp8kv(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                           value_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                           scale: float, max_context_len: int, workspace: torch.Tensor, k_scale: float,
                           v_scale: float, partition_size: int = 0, stream=None) -> torch.Tensor:
    """Decode attention over uint8 (FP8 E4M3) caches; query/out 16-bit, [N, Hq, d] or [N, q_len, Hq, d]."""
    if query.dim() == 3:
        n, hq, d = query.shape
        q_len = 1
    else:
        n, q_len, hq, d = query.shape
    nb, bs, hkv, d2 = key_cache.shape
    if key_cache.dtype != torch.uint8 or value_cache.dtype != torch.uint8 or d2 != d:
        raise ValueError("FP8 caches must be uint8 with the query's head_dim")
    if out.shape != query.shape or out.dtype != query.dtype:
        raise ValueError("out must match query")
    with _device_of(out, query, key_cache, value_cache, block_tables, context_lens, workspace, stream=stream):
        st = lib().pa_decode_attention_fp8kv(
            _dev(out, "out"), _dev(query, "query"), _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache"),
            _dev(block_tables, "block_tables"), block_tables.shape[1], _dev(context_lens, "context_lens"), n, q_len, hq,
            hkv, d, bs, nb, int(max_context_len), float(scale), dtype_code(query), float(k_scale), float(v_scale),
            int(partition_size), _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
            _stream(stream))
    _check("pa_decode_attention_fp8kv", st)
    return out


def workspace_size(num_seqs: int, q_len: int, num_heads: int, head_dim: int, max_context_len: int,
                   partition_size: int = 0) -> int:
    return int(lib().pa_decode_workspace_size_ex(num_seqs, q_len, num_heads, head_dim, max_context_len,
                                                 partition_size))


def alloc_workspace(num_seqs: int, q_len: int, num_heads: int, head_dim: int, max_context_len: int,
                    partition_size: int = 0, device=None) -> torch.Tensor:
    n = workspace_size(num_seqs, q_len, num_heads, head_dim, max_context_len, partition_size)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device or "cuda")


def _decode_shapes(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
                   block_tables: torch.Tensor, context_lens: torch.Tensor):
    """Checks the tensors of a 16-bit decode call; returns (N, q_len, Hq, Hkv, d, block_size, num_blocks)."""
    if query.dim() == 3:
        n, hq, d = query.shape
        q_len = 1
    elif query.dim() == 4:
        n, q_len, hq, d = query.shape
    else:
        raise ValueError("query must be [N, Hq, d] or [N, q_len, Hq, d]")
    if out.shape != query.shape or out.dtype != query.dtype:
        raise ValueError("out must match query in shape and dtype")
    nb, bs, hkv, d2 = key_cache.shape
    if d2 != d or value_cache.shape != key_cache.shape:
        raise ValueError("cache shape mismatch")
    if query.dtype != key_cache.dtype or value_cache.dtype != key_cache.dtype:
        raise ValueError("query and caches must share one dtype")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_tables and context_lens must be int32")
    if block_tables.dim() != 2 or block_tables.shape[0] != n or context_lens.shape != (n,):
        raise ValueError("block_tables must be [N, max_blocks] and context_lens [N]")
    return n, q_len, hq, hkv, d, bs, nb


def decode_attention(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
                     block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float, max_context_len: int,
                     workspace: torch.Tensor, partition_size: int = 0, stream=None) -> torch.Tensor:
    """Paged decode attention (pa_decode_attention_ex).  query/out are [N, Hq, d] (one query row)
    or [N, q_len, Hq, d] (q_len rows, causal inside the chunk)."""
    n, q_len, hq, hkv, d, bs, nb = _decode_shapes(out, query, key_cache, value_cache, block_tables, context_lens)
    with _device_of(out, query, key_cache, value_cache, block_tables, context_lens, workspace, stream=stream):
        st = lib().pa_decode_attention_ex(
            _dev(out, "out"), _dev(query, "query"), _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache"),
            _dev(block_tables, "block_tables"), block_tables.shape[1], _dev(context_lens, "context_lens"), n, q_len,
            hq, hkv, d, bs, nb, int(max_context_len), float(scale), dtype_code(query), int(partition_size),
            _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(), _stream(stream))
    _check("pa_decode_attention_ex", st)
    return out


def decode_attention_single(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                            value_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                            scale: float, max_context_len: int, workspace: torch.Tensor, stream=None) -> torch.Tensor:
    """pa_decode_attention: one query token per sequence, query/out [N, Hq, d]; the library
    chooses the split."""
    if query.dim() != 3:
        raise ValueError("query must be [N, Hq, d]")
    n, _, hq, hkv, d, bs, nb = _decode_shapes(out, query, key_cache, value_cache, block_tables, context_lens)
    with _device_of(out, query, key_cache, value_cache, block_tables, context_lens, workspace, stream=stream):
        st = lib().pa_decode_attention(
            _dev(out, "out"), _dev(query, "query"), _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache"),
            _dev(block_tables, "block_tables"), block_tables.shape[1], _dev(context_lens, "context_lens"), n, hq, hkv,
            d, bs, nb, int(max_context_len), float(scale), dtype_code(query), _dev(workspace, "workspace"),
            workspace.numel() * workspace.element_size(), _stream(stream))
    _check("pa_decode_attention", st)
    return out


def decode_attention_multiquery(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                                value_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                                scale: float, max_context_len: int, workspace: torch.Tensor,
                                stream=None) -> torch.Tensor:
    """pa_decode_attention_multiquery: q_len query rows per sequence, query/out [N, q_len, Hq, d],
    causal inside the chunk; the library chooses the split (and the tcgen05 kernel from 128 rows
    per kv head)."""
    if query.dim() != 4:
        raise ValueError("query must be [N, q_len, Hq, d]")
    n, q_len, hq, hkv, d, bs, nb = _decode_shapes(out, query, key_cache, value_cache, block_tables, context_lens)
    with _device_of(out, query, key_cache, value_cache, block_tables, context_lens, workspace, stream=stream):
        st = lib().pa_decode_attention_multiquery(
            _dev(out, "out"), _dev(query, "query"), _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache"),
            _dev(block_tables, "block_tables"), block_tables.shape[1], _dev(context_lens, "context_lens"), n, q_len,
            hq, hkv, d, bs, nb, int(max_context_len), float(scale), dtype_code(query), _dev(workspace, "workspace"),
            workspace.numel() * workspace.element_size(), _stream(stream))
    _check("pa_decode_attention_multiquery", st)
    return out


def workspace_size_shared_prefix(num_seqs: int, q_len: int, num_heads: int, head_dim: int, max_context_len: int,
                                 partition_size: int = 0) -> int:
    return int(lib().pa_decode_workspace_size_shared_prefix(num_seqs, q_len, num_heads, head_dim, max_context_len,
                                                            partition_size))


def alloc_workspace_shared_prefix(num_seqs: int, q_len: int, num_heads: int, head_dim: int, max_context_len: int,
                                  partition_size: int = 0, device=None) -> torch.Tensor:
    n = workspace_size_shared_prefix(num_seqs, q_len, num_heads, head_dim, max_context_len, partition_size)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device or "cuda")


def decode_attention_shared_prefix(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                                   value_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                                   scale: float, max_context_len: int, workspace: torch.Tensor, group_seq_start,
                                   group_prefix_len, partition_size: int = 0, stream=None) -> torch.Tensor:
    """pa_decode_attention_shared_prefix: decode attention where the sequences of group k
    (group_seq_start[k] .. group_seq_start[k+1] - 1) share their first group_prefix_len[k]
    positions' blocks.  The group arrays are host integer sequences."""
    n, q_len, hq, hkv, d, bs, nb = _decode_shapes(out, query, key_cache, value_cache, block_tables, context_lens)
    starts = [int(x) for x in group_seq_start]
    lens = [int(x) for x in group_prefix_len]
    ng = len(lens)
    if len(starts) != ng + 1 and not (ng == 0 and len(starts) in (0, 1)):
        raise ValueError("group_seq_start must have one more entry than group_prefix_len")
    c_starts = (ctypes.c_int32 * max(1, len(starts)))(*starts)
    c_lens = (ctypes.c_int32 * max(1, ng))(*lens)
    with _device_of(out, query, key_cache, value_cache, block_tables, context_lens, workspace, stream=stream):
        st = lib().pa_decode_attention_shared_prefix(
            _dev(out, "out"), _dev(query, "query"), _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache"),
            _dev(block_tables, "block_tables"), block_tables.shape[1], _dev(context_lens, "context_lens"), n, q_len,
            hq, hkv, d, bs, nb, int(max_context_len), float(scale), dtype_code(query), ng,
            ctypes.cast(c_starts, _vp) if starts else None, ctypes.cast(c_lens, _vp) if ng else None,
            int(partition_size), _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
            _stream(stream))
    _check("pa_decode_attention_shared_prefix", st)
    return out


def decode_attention_noalloc(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                             value_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                             scale: float, max_context_len: int, partition_size: int = 0, stream=None) -> torch.Tensor:
    """decode_attention without a workspace argument, for callers that cannot allocate device
    memory: the split-K scratch comes from the library's fixed 32 MiB device array.  Calls share
    that array, so calls that overlap on the GPU must not be issued; a problem needing more
    scratch than the array holds raises PaError (status PA_ERR_WORKSPACE)."""
    n, q_len, hq, hkv, d, bs, nb = _decode_shapes(out, query, key_cache, value_cache, block_tables, context_lens)
    with _device_of(out, query, key_cache, value_cache, block_tables, context_lens, stream=stream):
        st = lib().pa_decode_attention_noalloc(
            _dev(out, "out"), _dev(query, "query"), _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache"),
            _dev(block_tables, "block_tables"), block_tables.shape[1], _dev(context_lens, "context_lens"), n, q_len,
            hq, hkv, d, bs, nb, int(max_context_len), float(scale), dtype_code(query), int(partition_size),
            _stream(stream))
    _check("pa_decode_attention_noalloc", st)
    return out


def get_device_error(clear: bool = True, stream=None) -> int:
    v = ctypes.c_int32(0)
    _check("pa_get_device_error", lib().pa_get_device_error(ctypes.byref(v), int(clear), _stream(stream)))
    return int(v.value)


def set_decode_math(math: str) -> None:
    """'auto' (default): CUDA-core FMA for one query row per kv head, mma.sync tensor-core tiles
    for grouped heads and short chunks, the tcgen05 prefill kernel from 128 query rows per kv head;
    'fma': CUDA-core FMA up to 8 query rows per kv head; 'tensor': mma.sync tiles everywhere;
    'tcgen05': the tcgen05 prefill kernel for every 16-bit call.  Process-wide."""
    _check("pa_set_decode_math",
           lib().pa_set_decode_math({"auto": 0, "fma": 1, "tensor": 2, "tcgen05": 3}[math]))


def last_partition_size() -> int:
    """Split-K partition (tokens) of this thread's last decode call; 0 if it ran the tcgen05
    kernel without splitting."""
    return int(lib().pa_last_partition_size())


def profile_enable(on=True) -> None:
    """True / 1: time the plan, main and merge kernels of every decode call apart; 2: time the
    main and merge kernels together (their overlap kept); False / 0: stop."""
    _check("pa_profile_enable", lib().pa_profile_enable(int(on)))


def profile_read() -> tuple[float, int]:
    """(summed ms of the main kernel, calls) since the last read."""
    ms, n = ctypes.c_float(0.0), ctypes.c_int(0)
    _check("pa_profile_read", lib().pa_profile_read(ctypes.byref(ms), ctypes.byref(n)))
    return float(ms.value), int(n.value)


def profile_read_parts() -> tuple[float, float, float, int]:
    """(summed ms of the plan, main and merge kernels, calls) since the last read."""
    a, b, c, n = ctypes.c_float(0.0), ctypes.c_float(0.0), ctypes.c_float(0.0), ctypes.c_int(0)
    _check("pa_profile_read_parts",
           lib().pa_profile_read_parts(ctypes.byref(a), ctypes.byref(b), ctypes.byref(c), ctypes.byref(n)))
    return float(a.value), float(b.value), float(c.value), int(n.value)


def set_wait_limit_ns(ns: int) -> None:
    """Limit of the kernels' pipeline waits for later launches (a test hook); 0 = the default 2 s."""
    _check("pa_set_wait_limit_ns", lib().pa_set_wait_limit_ns(int(ns)))


def last_launch_count() -> int:
    return int(lib().pa_last_launch_count())
