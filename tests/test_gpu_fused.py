"""Fused depthwise + activation + 1x1 projection (grouped_conv_fwd_dw_pw)
through the C ABI, against the oracle's block (Oracle.dw_pw_block) element
by element: MobileNetV2 shapes at reduced batch and at full size, strides 1
and 2, every activation, both 16-bit types, with and without biases, ragged
row and column tiles, wide rows, the 4-channel compute form and forced tile
shapes, and canary bands around y."""
import numpy as np
import pytest
import torch

import depthwise_convolution_forward_gb300 as gc
from depthwise_convolution_forward_gb300 import _binding as B
from depthwise_convolution_forward_gb300 import inputs
from gpu_util import GUARD, assert_close, out_shape_of, require_gpu

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _pw(wl, K, seed):
    """Projection weights [K, C] ~ N(0, 1/C) and bias ~ U(-0.1, 0.1), drawn in
    fp32 and rounded once to the storage type."""
    g = torch.Generator().manual_seed(seed)
    dt = inputs.DTYPES[wl.dtype]
    w = (torch.randn(K, wl.G, generator=g) / wl.G ** 0.5).to(dt)
    b = ((torch.rand(K, generator=g) * 2 - 1) * 0.1).to(dt)
    return w, b


def run_fused(wl, x, w_dw, b_dw, w_pw, b_pw, act, tile=(0, 0, 0, 0)):
    dt = inputs.DTYPES[wl.dtype]
    K = w_pw.shape[0]
    shp = out_shape_of(wl)[:3] + (K,)
    n = int(np.prod(shp))
    buf = torch.empty(n + 2 * GUARD, dtype=dt, device=DEV)
    buf.view(torch.int16).fill_(-1)
    y = buf[GUARD:GUARD + n].view(shp)
    opt = B.gconv_options()
    opt.debug = 1
    for i, v in enumerate(tile):
        opt.tile[i] = v
    dev = [t.to(DEV) if t is not None else None for t in (x, w_dw, b_dw, w_pw, b_pw)]
    gc.grouped_conv_fwd_dw_pw_ex(*dev, y, gc.problem_of(wl), K, act, gc.DTYPE_CODES[wl.dtype],
                                 torch.cuda.current_stream(DEV), opt)
    torch.cuda.synchronize(DEV)
    assert opt.selected == B.KERNEL_DW_PW
    assert bool((buf[:GUARD].view(torch.int16) == -1).all()), "wrote before y"
    assert bool((buf[GUARD + n:].view(torch.int16) == -1).all()), "wrote after y"
    return y.cpu()


def _check(orc, wl, K, act, bias=True, seed=0, tile=(0, 0, 0, 0)):
    x, w, b = inputs.make_inputs(wl)
    w_pw, b_pw = _pw(wl, K, 8800 + seed)
    if not bias:
        b, b_pw = None, None
    y = run_fused(wl, x, w, b, w_pw, b_pw, act, tile)
    ref = orc.dw_pw_block(wl, x, w, b, act, w_pw, b_pw, inputs.DTYPES[wl.dtype])
    assert_close(y.double().numpy(), ref, wl.dtype, f"{wl.name} K={K} act={act} bias={bias} tile={tile}")


@pytest.mark.parametrize("name", ["mbv2_dw_s1_f16", "mbv2_dw_s2_f16"])
@pytest.mark.parametrize("act", [0, 1, 2])
def test_mobilenet_reduced_batch(orc, name, act):
    _check(orc, inputs.by_name(name).with_(N=2), 24, act)


@pytest.mark.parametrize("name", ["mbv2_dw_s1_f16", "mbv2_dw_s2_f16"])
def test_mobilenet_full_size(orc, name):
    _check(orc, inputs.by_name(name), 24, 2, seed=1)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("K", [8, 32, 64, 256])
def test_channel_counts(orc, dtype, K):
    wl = inputs.Workload("fz_k", 0, K, 2, 2, 64, 1, 1, (1, 17, 19), (1, 3, 3), (1, 1, 1), (0, 1, 1), (1, 1, 1),
                         dtype, True)
    _check(orc, wl, K, 2, seed=K)


CASES = [
    # (C, H, W, stride, pad): ragged row tiles, no padding, 128 output columns,
    # stride 2 with an odd input, one output row per tile, 256 channels, a
    # width split into ragged column tiles
    (16, 13, 13, 1, 1),
    (32, 10, 9, 1, 0),
    (16, 7, 128, 1, 1),
    (48, 15, 21, 2, 1),
    (32, 5, 253, 2, 1),
    (256, 6, 14, 1, 1),
    (64, 9, 300, 1, 1),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "C%d_%dx%d_s%d_p%d" % c)
def test_shapes(orc, case):
    C, H, W, s, p = case
    wl = inputs.Workload("fz_shape", 0, C + H, 2, 3, C, 1, 1, (1, H, W), (1, 3, 3), (1, s, s), (0, p, p),
                         (1, 1, 1), "bf16", True)
    _check(orc, wl, 24, 1, seed=C + W)


def test_without_biases(orc):
    _check(orc, inputs.by_name("mbv2_dw_s1_f16").with_(N=1), 24, 2, bias=False, seed=3)


def test_unsupported_shape_launches_nothing():
    """C not a multiple of 16: refused on the host, y untouched."""
    wl = inputs.Workload("fz_bad", 0, 0, 2, 1, 20, 1, 1, (1, 8, 8), (1, 3, 3), (1, 1, 1), (0, 1, 1), (1, 1, 1),
                         "f16", True)
    assert not gc.grouped_conv_fwd_dw_pw_supported(gc.problem_of(wl), 24, 2, gc.DTYPE_CODES["f16"])
    x, w, b = inputs.make_inputs(wl)
    w_pw, b_pw = _pw(wl, 24, 1)
    with pytest.raises(gc.GconvError):
        run_fused(wl, x, w, b, w_pw, b_pw, 2)


FORCED = [
    # (workload, K, (channels per thread, TH, TW, MMA issuer)): the
    # 4-channel form with twice the compute warps, walks of one row and of
    # many, segments, the dedicated issuing warp (1) and the compute warps
    # issuing (2) on both strides
    ("mbv2_dw_s1_f16", 24, (4, 0, 0, 0)),
    ("mbv2_dw_s2_f16", 24, (4, 0, 0, 0)),
    ("mbv2_dw_s1_f16", 24, (8, 7, 14, 0)),
    ("mbv2_dw_s2_f16", 24, (4, 14, 7, 0)),
    ("mbv2_dw_s1_f16", 32, (4, 1, 14, 0)),
    ("mbv2_dw_s2_f16", 16, (8, 4, 14, 0)),
    ("mbv2_dw_s1_f16", 24, (0, 0, 0, 2)),
    ("mbv2_dw_s2_f16", 24, (0, 0, 0, 1)),
    ("mbv2_dw_s1_f16", 40, (4, 0, 0, 2)),
    ("mbv2_dw_s2_f16", 40, (4, 0, 0, 1)),
]


@pytest.mark.parametrize("case", FORCED, ids=lambda c: "%s_K%d_cp%d_th%d_tw%d_mma%d" % ((c[0], c[1]) + c[2]))
def test_forced_forms(orc, case):
    name, K, tile = case
    _check(orc, inputs.by_name(name).with_(N=1), K, 2, seed=K + tile[0], tile=tile)


@pytest.mark.parametrize("case", CASES[:3] + CASES[-2:], ids=lambda c: "C%d_%dx%d_s%d_p%d" % c)
def test_shapes_four_channel_form(orc, case):
    C, H, W, s, p = case
    wl = inputs.Workload("fz_shape4", 0, C + H, 2, 3, C, 1, 1, (1, H, W), (1, 3, 3), (1, s, s), (0, p, p),
                         (1, 1, 1), "bf16", True)
    _check(orc, wl, 24, 1, seed=C + W + 1, tile=(4, 0, 0, 0))


def test_override_that_does_not_fit_raises():
    """A tile shape outside the kernel (TW > 16) is refused, y untouched."""
    wl = inputs.by_name("mbv2_dw_s1_f16").with_(N=1)
    x, w, b = inputs.make_inputs(wl)
    w_pw, b_pw = _pw(wl, 24, 2)
    with pytest.raises(gc.GconvError):
        run_fused(wl, x, w, b, w_pw, b_pw, 2, (8, 4, 17, 0))


@pytest.mark.parametrize("case", CASES, ids=lambda c: "C%d_%dx%d_s%d_p%d" % c)
def test_shapes_other_mma_issuer(orc, case):
    """The same shapes with the MMA issuer the planner did not choose."""
    C, H, W, s, p = case
    wl = inputs.Workload("fz_shape_m", 0, C + H, 2, 3, C, 1, 1, (1, H, W), (1, 3, 3), (1, s, s), (0, p, p),
                         (1, 1, 1), "f16", True)
    for mode in (1, 2):
        _check(orc, wl, 32, 2, seed=C + W + 2 + mode, tile=(0, 0, 0, mode))
