"""Argument marshalling of the Python binding, on the host: tensors of the wrong
dtype, shape, layout or device are rejected before any pointer reaches the C
ABI, which receives bare pointers and cannot check them."""

import pytest
import torch

from moe_decode_router_gb300 import flint_moe as F


def bf16(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


def test_tensor_checks():
    with pytest.raises(TypeError, match="x: expected a torch.Tensor"):
        F._expect([0.0], "x", torch.bfloat16, (1, F.HIDDEN))
    with pytest.raises(ValueError, match="x: dtype"):
        F._expect(torch.zeros(2, F.HIDDEN), "x", torch.bfloat16, (2, F.HIDDEN))
    with pytest.raises(ValueError, match=r"x: shape \(2, 1024\), expected \(2, 2048\)"):
        F._expect(bf16(2, 1024), "x", torch.bfloat16, (2, F.HIDDEN))
    with pytest.raises(ValueError, match="x: must be contiguous"):
        F._expect(bf16(F.HIDDEN, 2).t(), "x", torch.bfloat16, (2, F.HIDDEN))
    with pytest.raises(ValueError, match="x: must be on the current CUDA device"):
        F._expect(bf16(2, F.HIDDEN), "x", torch.bfloat16, (2, F.HIDDEN))
    with pytest.raises(ValueError, match="ws: expected a 1-D byte buffer"):
        F._expect(torch.zeros(4, 4, dtype=torch.uint8), "ws", torch.uint8, None)


def test_activation_rows():
    assert F._rows(bf16(3, F.HIDDEN)) == 3
    with pytest.raises(ValueError, match="x: expected"):
        F._rows(bf16(F.HIDDEN))
    with pytest.raises(ValueError, match="x: shape"):
        F._check_io(bf16(2, 1024), bf16(2, 1024), None, None)


def test_pack_weights_checks_plain_shapes_before_the_call():
    ne = F.N_EXPERTS + F.N_SHARED
    good_scales = torch.zeros(ne, 2 * F.INTER, F.HIDDEN // 16, dtype=torch.uint8)
    with pytest.raises(ValueError, match="gate_up: shape"):
        F.pack_weights(torch.zeros(ne, 2 * F.INTER, F.HIDDEN, dtype=torch.uint8), good_scales, None, None,
                       torch.zeros(16, dtype=torch.uint8))
    with pytest.raises(ValueError, match="gate_up: dtype"):
        F.pack_weights(torch.zeros(ne, 2 * F.INTER, F.HIDDEN, dtype=torch.uint8), None, None, None,
                       torch.zeros(16, dtype=torch.uint8), weight_dtype=F.W_BF16)
