"""The Python binding's argument checks, without a GPU: every entry point refuses host tensors
before it reaches the library, so nothing is ever launched on pointers of the wrong kind."""
import pytest
import torch

from paged_kv_cache_265_gb300 import pa


def _cpu(*shape, dtype=torch.bfloat16):
    return torch.zeros(shape, dtype=dtype)


def test_append_refuses_host_tensors():
    with pytest.raises(ValueError, match="CUDA"):
        pa.reshape_and_cache(_cpu(2, 2, 64), _cpu(2, 2, 64), _cpu(4, 16, 2, 64), _cpu(4, 16, 2, 64),
                             torch.zeros(2, dtype=torch.int64))


def test_attention_refuses_host_tensors():
    q = _cpu(2, 4, 64)
    with pytest.raises(ValueError, match="CUDA"):
        pa.decode_attention(torch.empty_like(q), q, _cpu(4, 16, 2, 64), _cpu(4, 16, 2, 64),
                            torch.zeros((2, 4), dtype=torch.int32), torch.ones(2, dtype=torch.int32), 0.125, 16,
                            torch.zeros(64, dtype=torch.uint8))


def test_copy_blocks_and_spec_verify_refuse_host_tensors():
    with pytest.raises(ValueError, match="CUDA"):
        pa.copy_blocks(_cpu(4, 16, 2, 64), _cpu(4, 16, 2, 64), torch.zeros((1, 2), dtype=torch.int64))
    f = torch.float32
    with pytest.raises(ValueError, match="CUDA"):
        pa.spec_verify(_cpu(2, 3, 10, dtype=f), _cpu(2, 2, 10, dtype=f), torch.zeros((2, 2), dtype=torch.int32),
                       _cpu(2, 2, dtype=f), _cpu(2, dtype=f), num_accepted=torch.zeros(2, dtype=torch.int32),
                       out_tokens=torch.zeros((2, 3), dtype=torch.int32))
