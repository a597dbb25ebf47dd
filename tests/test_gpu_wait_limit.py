"""The kernels' bounded waits, made to run out on purpose (failure detection without a GPU
fault).

Every mbarrier wait inside the decode and tcgen05 kernels gives up after a limit, sets
PA_DEVERR_TIMEOUT in the device error word and stops its CTA; the CTA still waits (under the
default 2 s limit) for its own copies and tensor-core products before it exits, so the
context stays usable.  Here the pipeline waits get a 1 ns limit (pa_set_wait_limit_ns), so
the first wait of a CTA that is not already complete gives up; the call must report the
timeout, and the next call with the default limit must again match the oracle.
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
    pa.set_wait_limit_ns(0)
    pa.set_decode_math("auto")
    assert pa.get_device_error(clear=True) == 0


def _timeout_then_recover(w, math):
    step = G.GpuStep(w)
    step.append()
    torch.cuda.synchronize()
    _, _, ref = G.oracle_step(w)
    pa.set_decode_math(math)
    try:
        pa.set_wait_limit_ns(1)
        step.attend()
        torch.cuda.synchronize()
        pa.set_wait_limit_ns(0)
        flags = pa.get_device_error(clear=True)
        assert flags & pa.PA_DEVERR_TIMEOUT, f"no wait ran out (flags {flags:#x})"
        assert flags & ~pa.PA_DEVERR_TIMEOUT == 0, f"unexpected flags {flags:#x}"
        step.out.fill_(float("nan"))
        got = G.to_bits(step.attend())
        torch.cuda.synchronize()
    finally:
        pa.set_wait_limit_ns(0)
        pa.set_decode_math("auto")
    assert pa.get_device_error(clear=True) == 0
    G.compare(got, ref, w.dtype, f"{w.name} after a timed-out call")
    assert G.ulps_from_rounded_oracle(got, ref, w.dtype) <= 1


def test_decode_kernel_wait_runs_out_and_recovers():
    _timeout_then_recover(W.gqa_batch32(), "auto")


def test_tcgen05_kernel_wait_runs_out_and_recovers():
    w = W.make_workload("chunk_timeout", [300, 900, 1500], num_heads=8, num_kv_heads=2, head_dim=128, q_len=64,
                        num_blocks=200, seed=41)
    _timeout_then_recover(w, "auto")
    assert pa.last_partition_size() == 0          # the call ran on the tcgen05 kernel


def test_shared_prefix_kernels_wait_runs_out_and_recover():
    """A shared-prefix call: the one-CTA order kernel, the persistent suffix kernel (256 units on
    at most one CTA per SM, so CTAs walk several units) and the prefix kernel stop on a wait that
    runs out, and the next call with the default limit matches the oracle."""
    lens = 256 + 16 + 23 * np.arange(32)
    w = W.make_workload("sp_timeout", lens, num_heads=32, num_kv_heads=8, head_dim=128, q_len=5, seed=77,
                        shared_prefix_blocks=16)
    step = G.GpuStep(w)
    step.append()
    torch.cuda.synchronize()
    _, _, ref = G.oracle_step(w)
    ws = pa.alloc_workspace_shared_prefix(w.num_seqs, w.q_len, w.num_heads, w.head_dim, w.max_context_len, 0)
    out = torch.full_like(step.query, float("nan"))

    def call():
        pa.decode_attention_shared_prefix(out, step.query, step.key_cache, step.value_cache, step.block_tables,
                                          step.context_lens, w.scale, w.max_context_len, ws, [0, w.num_seqs],
                                          [16 * w.shared_prefix_blocks])
        torch.cuda.synchronize()

    try:
        pa.set_wait_limit_ns(1)
        call()
        pa.set_wait_limit_ns(0)
        flags = pa.get_device_error(clear=True)
        assert flags & pa.PA_DEVERR_TIMEOUT, f"no wait ran out (flags {flags:#x})"
        assert flags & ~pa.PA_DEVERR_TIMEOUT == 0, f"unexpected flags {flags:#x}"
        assert pa.last_launch_count() == 3       # order, suffix and prefix kernels
        out.fill_(float("nan"))
        call()
        got = G.to_bits(out)
    finally:
        pa.set_wait_limit_ns(0)
    assert pa.get_device_error(clear=True) == 0
    G.compare(got, ref, w.dtype, "shared prefix after a timed-out call")
    assert G.ulps_from_rounded_oracle(got, ref, w.dtype) <= 1
