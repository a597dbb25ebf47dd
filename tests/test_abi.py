"""The C ABI without a GPU: the library builds, loads, exports every symbol its
header declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

from paged_kv_cache_265_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa.h")


@pytest.fixture(scope="module")
def lib():
    path = B.build()
    from paged_kv_cache_265_gb300 import pa

    return pa.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n


def test_binding_constants_match_header():
    """Every PA_* integer the header defines that the binding also names has the same value there."""
    from paged_kv_cache_265_gb300 import pa

    defines = dict(re.findall(r"^#define\s+(PA_[A-Z0-9_]+)\s+(0x[0-9a-fA-F]+|\d+)\b", open(HEADER).read(), flags=re.M))
    assert "PA_DEVERR_QUERY_RANGE" in defines
    shared = [n for n in defines if hasattr(pa, n)]
    assert len(shared) >= 7
    for n in shared:
        assert getattr(pa, n) == int(defines[n], 0), n


def test_status_strings(lib):
    for code, text in [(0, "ok"), (1, "invalid argument"), (2, "unsupported"), (3, "workspace"), (4, "CUDA")]:
        assert text in lib.pa_status_string(code).decode()
    assert lib.pa_status_string(99).decode() == "unknown status"
    assert lib.pa_version() >= 100


FAKE = 1 << 20  # an aligned, never-dereferenced "device" address


def _decode(lib, **kw):
    a = dict(out=FAKE, query=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, mbps=8, cl=FAKE, n=2, q_len=1, hq=4, hkv=4, d=64,
             bs=16, nb=64, max_ctx=100, scale=0.125, dtype=0, part=0, ws=FAKE, ws_bytes=1 << 30, stream=None)
    a.update(kw)
    return lib.pa_decode_attention_ex(a["out"], a["query"], a["kc"], a["vc"], a["bt"], a["mbps"], a["cl"], a["n"],
                                      a["q_len"], a["hq"], a["hkv"], a["d"], a["bs"], a["nb"], a["max_ctx"],
                                      a["scale"], a["dtype"], a["part"], a["ws"], a["ws_bytes"], a["stream"])


def test_decode_host_validation(lib):
    assert _decode(lib, n=0) == 0                       # nothing to do
    assert _decode(lib, hkv=3) == 1                     # heads not a multiple of kv heads
    assert _decode(lib, q_len=0) == 1
    assert _decode(lib, dtype=7) == 1
    assert _decode(lib, scale=float("nan")) == 1
    assert _decode(lib, part=24) == 1                   # partition not a multiple of 16
    assert _decode(lib, max_ctx=8 * 16 + 1) == 1        # longer than the block table can map
    assert _decode(lib, out=None) == 1
    assert _decode(lib, query=FAKE + 8) == 1            # misaligned
    assert _decode(lib, d=96) == 2                      # head_dim not compiled
    assert _decode(lib, bs=32) == 2                     # block size other than 16
    assert _decode(lib, hq=64, hkv=1, q_len=2000, max_ctx=128) == 2   # 128,000 rows per kv head
    assert _decode(lib, hq=1 << 20, hkv=1 << 20) == 2                 # absurd head count
    assert _decode(lib, ws=None) == 3
    assert _decode(lib, ws_bytes=16) == 3


def test_workspace_size(lib):
    lib.pa_decode_workspace_size_ex.restype = ctypes.c_size_t
    lib.pa_decode_workspace_size.restype = ctypes.c_size_t
    small = lib.pa_decode_workspace_size(4, 1, 4, 64, 100)
    assert small > 0
    # one partition per sequence: no partial buffers
    assert lib.pa_decode_workspace_size_ex(4, 1, 4, 64, 100, 1 << 20) == small
    split = lib.pa_decode_workspace_size_ex(4, 1, 4, 64, 100, 16)
    # 7 partitions x 4 seqs x 4 heads x (64 fp32 + 2 fp32) at least
    assert split >= small + 7 * 4 * 4 * (64 + 2) * 4
    assert lib.pa_decode_workspace_size_ex(4, 1, 4, 64, 100, 24) == 0


def test_reshape_host_validation(lib):
    f = lib.pa_reshape_and_cache
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 4, 64, 16, 64, 0, None) == 0      # no tokens
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 4, 96, 16, 64, 0, None) == 2      # head_dim
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 4, 64, 8, 64, 0, None) == 2       # block size
    assert f(None, FAKE, FAKE, FAKE, FAKE, 4, 4, 64, 16, 64, 0, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE + 4, 4, 4, 64, 16, 64, 0, None) == 1  # slot_mapping alignment
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, -1, 4, 64, 16, 64, 0, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 1 << 20, 128, 16, 64, 0, None) == 2   # absurd head count
    assert lib.pa_copy_blocks(FAKE, FAKE, FAKE, 1, 1 << 20, 128, 16, 64, 0, None) == 2


def _prefix_call(lib, starts, lens, **kw):
    a = dict(n=4, q_len=1, hq=4, hkv=4, d=64, max_ctx=100, ws=FAKE, ws_bytes=1 << 30)
    a.update(kw)
    ng = len(lens)
    c_starts = (ctypes.c_int32 * max(1, len(starts)))(*starts)
    c_lens = (ctypes.c_int32 * max(1, ng))(*lens)
    return lib.pa_decode_attention_shared_prefix(
        FAKE, FAKE, FAKE, FAKE, FAKE, 8, FAKE, a["n"], a["q_len"], a["hq"], a["hkv"], a["d"], 16, 64, a["max_ctx"],
        ctypes.c_float(0.125), 0, ng, ctypes.cast(c_starts, ctypes.c_void_p) if starts else None,
        ctypes.cast(c_lens, ctypes.c_void_p) if ng else None, 0, a["ws"], ctypes.c_size_t(a["ws_bytes"]), None)


def test_shared_prefix_host_validation(lib):
    """The group table is checked on the host before anything is enqueued."""
    lib.pa_decode_attention_shared_prefix.restype = ctypes.c_int
    assert _prefix_call(lib, [0, 5], [16]) == 1            # a group past the batch
    assert _prefix_call(lib, [2, 1], [16]) == 1            # starts decreasing
    assert _prefix_call(lib, [0, 2], [8]) == 1             # not whole blocks
    assert _prefix_call(lib, [0, 2], [-16]) == 1
    assert _prefix_call(lib, [0, 2], [112]) == 1           # more than max_context_len - q_len
    assert _prefix_call(lib, [], [1] * 0, n=0) == 0        # nothing to do
    assert _prefix_call(lib, [0, 1] + [1] * 256, [16] * 257) == 1   # more than PA_MAX_PREFIX_GROUPS groups
    assert _prefix_call(lib, [0, 2], [16], ws=None) == 3
    assert _prefix_call(lib, [0, 2], [16], ws_bytes=64) == 3


def test_shared_prefix_workspace_size(lib):
    f = lib.pa_decode_workspace_size_shared_prefix
    f.restype = ctypes.c_size_t
    plain = lib.pa_decode_workspace_size_ex
    plain.restype = ctypes.c_size_t
    # one extra piece per sequence (the prefix's), partials always reserved
    assert f(4, 5, 32, 128, 1536, 512) > plain(4, 5, 32, 128, 1536, 512)
    assert f(4, 5, 32, 128, 1536, 0) == f(4, 5, 32, 128, 1536, 512)   # sized for the finest split
    assert f(4, 5, 32, 128, 1536, 24) == 0
