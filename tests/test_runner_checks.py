"""Argument checks of the torch convenience layer (runner), on CPU: the C ABI
takes raw pointers, so runner refuses tensors whose layout or type the
kernels would misread (strided views, other dtypes, shape mismatches, CPU
tensors) before any pointer reaches the library."""
import pytest
import torch

from flashattention_attention_backward_gb300 import runner


def _t(*shape, dtype=torch.bfloat16):
    return torch.zeros(*shape, dtype=dtype)


def test_forward_rejects_bad_tensors():
    q, k = _t(1, 2, 8, 64), _t(1, 1, 8, 64)
    with pytest.raises(ValueError, match="CUDA"):
        runner.forward(q, k, k.clone(), 0.125, True)            # CPU tensors
    with pytest.raises(ValueError, match="bfloat16"):
        runner.forward(q.float(), k, k, 0.125, True)
    with pytest.raises(ValueError, match="contiguous"):
        runner.forward(_t(1, 2, 64, 8).transpose(2, 3), k, k, 0.125, True)
    with pytest.raises(ValueError, match="shape"):
        runner.forward(q, _t(1, 1, 9, 64), _t(1, 1, 9, 64), 0.125, True)
    with pytest.raises(ValueError, match="4-D"):
        runner.forward(_t(2, 8, 64), k, k, 0.125, True)


def test_backward_rejects_bad_tensors():
    q, k = _t(1, 2, 8, 64), _t(1, 1, 8, 64)
    lse = torch.zeros(1, 2, 8)
    with pytest.raises(ValueError, match="matches neither"):
        runner.backward(q, k, k, q, _t(1, 2, 8, 32), lse, 0.125, True)  # dO shape
    with pytest.raises(ValueError, match="bfloat16"):
        runner.backward(q, k, k, q, q.float(), lse, 0.125, True)         # dO dtype
    with pytest.raises(ValueError, match="CUDA"):
        runner.backward(q, k, k, q, q, lse, 0.125, True)                 # CPU tensors
