"""GPU parity of the copy-on-write block copy (pa_copy_blocks) against the oracle:
bit-exact over the whole pool, bad ids flagged, and a fork of a shared, partly
filled prefix block followed by the append and attention."""
import math

import numpy as np
import pytest
import torch

from paged_kv_cache_265_gb300 import pa
from paged_kv_cache_265_gb300 import workload as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import gpu_helpers as G
    import oracle


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from paged_kv_cache_265_gb300 import build

    build.build()
    pa.get_device_error(clear=True)
    yield
    assert pa.get_device_error(clear=True) == 0


@pytest.mark.parametrize("dtype,hkv,d", [("bf16", 8, 128), ("fp16", 4, 64)])
def test_copy_blocks_bit_exact(dtype, hkv, d):
    w = W.make_workload("cow", [700, 333, 1000, 45], num_heads=hkv, num_kv_heads=hkv, head_dim=d, dtype=dtype,
                        append_len=0, num_blocks=400, seed=31)
    used = np.unique(w.block_tables[w.block_tables >= 0])
    free = np.setdiff1d(np.arange(w.num_blocks), used)
    g = np.random.Generator(np.random.PCG64(32))
    src = g.choice(used, size=60, replace=False)
    dst = g.choice(free, size=60, replace=False)
    mapping = np.stack([src, dst], axis=1).astype(np.int64)
    kc, vc = G.to_dev(w.key_cache, dtype), G.to_dev(w.value_cache, dtype)
    pa.copy_blocks(kc, vc, torch.from_numpy(mapping).cuda())
    torch.cuda.synchronize()
    hk, hv = w.key_cache.copy(), w.value_cache.copy()
    assert oracle.load().copy_blocks(hk, hv, mapping) == 0
    assert np.array_equal(G.to_bits(kc), hk) and np.array_equal(G.to_bits(vc), hv)
    assert pa.last_launch_count() == 1


def test_copy_blocks_bad_ids_flagged():
    w = W.make_workload("cowbad", [40, 20], num_heads=2, num_kv_heads=2, head_dim=64, append_len=0, num_blocks=8,
                        seed=33)
    kc, vc = G.to_dev(w.key_cache, "bf16"), G.to_dev(w.value_cache, "bf16")
    before = G.to_bits(kc)
    pa.copy_blocks(kc, vc, torch.tensor([[0, 8], [-1, 3]], dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    assert pa.get_device_error(clear=True) & pa.PA_DEVERR_BLOCK_ID
    assert np.array_equal(G.to_bits(kc), before)


def test_fork_of_a_shared_partial_block():
    """64 sequences share a 1000-token prefix (its last block holds 8 tokens).  Each copies that
    block, appends its own token 1000 into the copy and attends; the shared block is never
    written, and everything matches the oracle running the same steps."""
    g = np.random.Generator(np.random.PCG64(34))
    n, hq, hkv, d, nb, prefix = 64, 32, 8, 128, 256, 1000
    bits = lambda *shape: g.standard_normal(shape).astype(np.float32)
    to_b = lambda x: torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    kc = np.full((nb, 16, hkv, d), W.NAN_BITS["bf16"], np.uint16)
    vc = kc.copy()
    pk, pv = to_b(bits(prefix, hkv, d)), to_b(bits(prefix, hkv, d))
    shared = g.permutation(nb)[: (prefix + 15) // 16]
    for p_ in range(prefix):
        kc[shared[p_ // 16], p_ % 16], vc[shared[p_ // 16], p_ % 16] = pk[p_], pv[p_]
    last = shared[-1]
    copies = np.setdiff1d(np.arange(nb), shared)[:n]
    mapping = np.stack([np.full(n, last), copies], axis=1).astype(np.int64)
    bt = np.tile(shared, (n, 1)).astype(np.int32)
    bt[:, -1] = copies
    slots = (copies.astype(np.int64) * 16 + prefix % 16)
    nk, nv = to_b(bits(n, hkv, d)), to_b(bits(n, hkv, d))
    q = to_b(bits(n, 1, hq, d))
    lens = np.full(n, prefix + 1, np.int32)
    scale = 1 / math.sqrt(d)
    # GPU: copy, append, attend
    dk, dv = G.to_dev(kc, "bf16"), G.to_dev(vc, "bf16")
    pa.copy_blocks(dk, dv, torch.from_numpy(mapping).cuda())
    pa.reshape_and_cache(G.to_dev(nk, "bf16"), G.to_dev(nv, "bf16"), dk, dv, torch.from_numpy(slots).cuda())
    dq = G.to_dev(q, "bf16")
    out = torch.empty_like(dq)
    ws = pa.alloc_workspace(n, 1, hq, d, prefix + 1)
    pa.decode_attention(out, dq, dk, dv, torch.from_numpy(bt).cuda(), torch.from_numpy(lens).cuda(), scale,
                        prefix + 1, ws)
    torch.cuda.synchronize()
    # oracle: the same steps
    orc = oracle.load()
    assert orc.copy_blocks(kc, vc, mapping) == 0
    assert orc.reshape_and_cache(nk, nv, kc, vc, slots) == 0
    ref, bad = orc.decode_attention(q, kc, vc, bt, lens, scale, "bf16")
    assert bad == 0
    assert np.array_equal(G.to_bits(dk), kc) and np.array_equal(G.to_bits(dv), vc)
    assert np.all(kc[last, prefix % 16:] == W.NAN_BITS["bf16"])    # the shared block was not written
    G.compare(G.to_bits(out), ref, "bf16", "fork")
