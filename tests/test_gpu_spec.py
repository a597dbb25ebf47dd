"""GPU parity of speculative-decoding verification (pa_spec_verify) against the oracle.
Outputs are integers (accepted counts and tokens), so the comparison is exact."""
import numpy as np
import pytest
import torch

from paged_kv_cache_265_gb300 import pa
from paged_kv_cache_265_gb300 import workload as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
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


def run_both(x: W.SpecInputs):
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    acc, out = pa.spec_verify(d(x.target_probs), d(x.draft_probs), d(x.draft_tokens), d(x.u_accept),
                              d(x.u_sample))
    torch.cuda.synchronize()
    ra, ro = oracle.load().spec_verify(x.target_probs, x.draft_probs, x.draft_tokens, x.u_accept, x.u_sample)
    return acc.cpu().numpy(), out.cpu().numpy(), ra, ro


@pytest.mark.parametrize("n,k,v,noise,seed", [(64, 4, 32000, 1.0, 1), (257, 1, 1000, 0.5, 2), (16, 8, 32000, 3.0, 3),
                                              (64, 4, 32000, 0.0, 4), (33, 4, 4096, 6.0, 5), (8, 0, 513, 1.0, 6),
                                              (16, 4, 32001, 1.0, 10), (12, 3, 4097, 2.0, 11),
                                              (10, 2, 20478, 1.5, 12)])
def test_spec_verify_matches_oracle(n, k, v, noise, seed):
    x = W.spec_verify_inputs(num_seqs=n, k=k, vocab=v, seed=seed, noise=noise)
    acc, out, ra, ro = run_both(x)
    assert np.array_equal(acc, ra)
    assert np.array_equal(out, ro)
    if noise == 0.0:
        assert np.all(acc == k)                   # identical models accept every draft


def test_spec_verify_zero_residual_falls_back_to_target():
    x = W.spec_verify_inputs(num_seqs=32, k=2, vocab=2000, seed=7)
    x.target_probs[:, :2] = 0.5 * x.draft_probs   # unnormalised: every draft rejected w.p. 1/2, residual 0
    acc, out, ra, ro = run_both(x)
    assert np.array_equal(acc, ra) and np.array_equal(out, ro)
    assert np.all(out[np.arange(32), acc] >= 0)


def test_spec_verify_bad_draft_token_is_flagged():
    x = W.spec_verify_inputs(num_seqs=4, k=3, vocab=100, seed=8)
    x.draft_tokens[2, 1] = 100
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    acc, out = pa.spec_verify(d(x.target_probs), d(x.draft_probs), d(x.draft_tokens), d(x.u_accept), d(x.u_sample))
    torch.cuda.synchronize()
    assert pa.get_device_error(clear=True) & pa.PA_DEVERR_TOKEN
    assert acc[2].item() <= 1


def test_spec_verify_largest_vocabulary_last_chunk():
    """The largest vocabulary (64 chunks of 4096 entries) with uniforms that put every draw in
    the last chunk."""
    x = W.spec_verify_inputs(num_seqs=8, k=2, vocab=262144, seed=9)
    x.u_sample[:] = np.float32(0.999999)
    acc, out, ra, ro = run_both(x)
    assert np.array_equal(acc, ra) and np.array_equal(out, ro)
    assert np.all(out[np.arange(8), acc] >= 262144 - 4096)
