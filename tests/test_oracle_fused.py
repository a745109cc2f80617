"""Pins of the oracle's depthwise + activation + 1x1 projection block
(``Oracle.dw_pw_block``), on the CPU: torch's fp64 convolutions composed
independently, the identity projection, and the activations' clamps."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from depthwise_convolution_forward_gb300 import inputs


def _problem(N, C, H, W, s, p, dtype="bf16"):
    return inputs.Workload("blk", 0, 0, 2, N, C, 1, 1, (1, H, W), (1, 3, 3), (1, s, s), (0, p, p), (1, 1, 1),
                           dtype, True)


def _torch_block(wl, x, w_dw, b_dw, act, w_pw, b_pw, tdt):
    """The same block from torch's own conv2d in float64 (NCHW)."""
    C = wl.G
    xt = x.double().reshape(wl.N, wl.inp[1], wl.inp[2], C).permute(0, 3, 1, 2)
    wt = w_dw.double().reshape(C, 1, 3, 3)
    h = F.conv2d(xt, wt, b_dw.double().reshape(C), stride=wl.stride[1], padding=wl.pad[1], groups=C)
    if act == 1:
        h = h.clamp(min=0)
    elif act == 2:
        h = h.clamp(0, 6)
    h = h.to(tdt).double()
    y = F.conv2d(h, w_pw.double().reshape(w_pw.shape[0], C, 1, 1),
                 None if b_pw is None else b_pw.double())
    return y.permute(0, 2, 3, 1).numpy()


@pytest.mark.parametrize("act", [0, 1, 2])
@pytest.mark.parametrize("s,p", [(1, 1), (2, 1), (1, 0)])
def test_matches_torch_composition(act, s, p):
    wl = _problem(2, 16, 9, 11, s, p)
    x, w, b = inputs.make_inputs(wl)
    x = x * 8  # push some depthwise outputs past 6 so ReLU6 clamps at the top too
    g = torch.Generator().manual_seed(5)
    w_pw = (torch.randn(24, 16, generator=g) / 4).to(torch.bfloat16)
    b_pw = (torch.rand(24, generator=g) - 0.5).to(torch.bfloat16)
    got = oracle.get().dw_pw_block(wl, x, w, b, act, w_pw, b_pw, torch.bfloat16)
    ref = _torch_block(wl, x, w, b, act, w_pw, b_pw, torch.bfloat16)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_identity_projection_is_the_rounded_depthwise_output():
    """K = C, w_pw = I, no bias, no activation: y is the depthwise layer's
    output rounded to the storage type."""
    wl = _problem(1, 32, 7, 8, 1, 1, "f16")
    x, w, b = inputs.make_inputs(wl)
    eye = torch.eye(32).to(torch.float16)
    y = oracle.get().dw_pw_block(wl, x, w, b, 0, eye, None, torch.float16)
    h = oracle.get().forward(wl, x, w, b).reshape(y.shape)
    assert np.array_equal(y, torch.from_numpy(h).to(torch.float16).double().numpy())


def test_relu6_clamps_both_ends():
    """Large depthwise outputs: with ReLU6 and an identity projection every
    value lies in [0, 6] and both ends are reached."""
    wl = _problem(1, 16, 8, 8, 1, 1)
    x, w, b = inputs.make_inputs(wl)
    x = x * 50
    eye = torch.eye(16).to(torch.bfloat16)
    y = oracle.get().dw_pw_block(wl, x, w, b, 2, eye, None, torch.bfloat16)
    assert y.min() == 0.0 and y.max() == 6.0
