"""Backward weight (the gradient with respect to w) through the C ABI,
against the oracle's fp64 backward weight, element by element.

* every workload family at reduced batch, and three at full size;
* random small 2D/3D problems over all dtypes, strides, paddings, dilations;
* misaligned x / dy (narrower vectors), integer inputs that must be exact,
  two calls that must agree bit for bit (fixed split and summation order);
* canary bands around dw.
"""
import numpy as np
import pytest
import torch

import depthwise_convolution_forward_gb300 as gc
from depthwise_convolution_forward_gb300 import _binding as B
from depthwise_convolution_forward_gb300 import inputs
from gpu_util import GUARD, TOL, assert_close, out_shape_of, require_gpu

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def make_dy(wl, seed):
    """dy ~ U(-1, 1) in the forward output layout, drawn in fp32 on the host
    and rounded once to the storage dtype."""
    g = torch.Generator().manual_seed(seed)
    return (torch.rand(out_shape_of(wl), generator=g, dtype=torch.float32) * 2 - 1).to(inputs.DTYPES[wl.dtype])


def run_bww(wl, x, dy, offset=0):
    """dw on the host and the selected kernel; x and dy start `offset`
    elements into their allocations."""
    dt = inputs.DTYPES[wl.dtype]
    p = gc.problem_of(wl)
    code = gc.DTYPE_CODES[wl.dtype]

    def place(t):
        if not offset:
            return t.to(DEV)
        buf = torch.empty(t.numel() + offset, dtype=dt, device=DEV)
        v = buf[offset:].view(t.shape)
        v.copy_(t)
        return v

    xd, dyd = place(x), place(dy)
    n = int(np.prod(wl.w_shape()))
    buf = torch.empty(n + 2 * GUARD, dtype=dt, device=DEV)
    words = torch.int32 if dt == torch.float32 else torch.int16
    buf.view(words).fill_(-1)
    dw = buf[GUARD:GUARD + n].view(wl.w_shape())
    need = gc.grouped_conv_bwd_weight_workspace_size(p, code)
    ws = torch.full((need // 4,), float("nan"), dtype=torch.float32, device=DEV)  # stale contents must not matter
    opt = B.gconv_options()
    opt.debug = 1
    gc.grouped_conv_bwd_weight_ex(xd, dyd, dw, p, code, ws, need, torch.cuda.current_stream(DEV), opt)
    torch.cuda.synchronize(DEV)
    assert bool((buf[:GUARD].view(words) == -1).all()), "wrote before dw"
    assert bool((buf[GUARD + n:].view(words) == -1).all()), "wrote after dw"
    return dw.cpu(), opt.selected


FAMILY = ["mbv2_dw_s1_f16", "mbv2_dw_s2_f16", "resnext_a_bf16", "resnext_b_bf16", "resnext3d_n1_f16",
          "grouped2d_f32_smoke", "sweep_g512_d2_s1_bf16", "sweep_g256_d2_s2_bf16", "sweep_g64_d1_s1_bf16",
          "sweep_g8_d2_s1_bf16"]


@pytest.mark.parametrize("name", FAMILY)
def test_reduced_batch_full_compare(orc, name):
    wl = inputs.by_name(name)
    wl = wl.with_(N=min(wl.N, 2), bias=False)
    x, _, _ = inputs.make_inputs(wl)
    dy = make_dy(wl, 300 + wl.variant)
    dw, sel = run_bww(wl, x, dy)
    assert sel == B.KERNEL_BWD_WEIGHT
    assert_close(dw.double().numpy(), orc.bwd_weight(wl, x, dy), wl.dtype, name)


@pytest.mark.parametrize("name", ["mbv2_dw_s1_f16", "resnext_b_bf16", "resnext3d_n8_f16"])
def test_full_size(orc, name):
    wl = inputs.by_name(name).with_(bias=False)
    x, _, _ = inputs.make_inputs(wl)
    dy = make_dy(wl, 400 + wl.variant)
    dw, _ = run_bww(wl, x, dy)
    assert_close(dw.double().numpy(), orc.bwd_weight(wl, x, dy), wl.dtype, name)


@pytest.mark.parametrize("seed", range(24))
def test_random_small_problems(orc, seed):
    rng = np.random.default_rng(5000 + seed)
    wl = inputs.random_problem(rng, max_c=12, max_hw=10).with_(bias=False)
    x, _, _ = inputs.make_inputs(wl)
    dy = make_dy(wl, 6000 + seed)
    dw, _ = run_bww(wl, x, dy)
    assert_close(dw.double().numpy(), orc.bwd_weight(wl, x, dy), wl.dtype, f"seed {seed}: {wl}")


@pytest.mark.parametrize("offset", [1, 2, 4])
def test_misaligned_inputs(orc, offset):
    """x and dy shifted by an element count that breaks 16-, 8- or 4-byte
    vectors: the kernel narrows its vectors and the result is unchanged."""
    for wl in (inputs.by_name("mbv2_dw_s2_f16").with_(N=1, bias=False),
               inputs.by_name("resnext_b_bf16").with_(N=1, bias=False)):
        x, _, _ = inputs.make_inputs(wl)
        dy = make_dy(wl, 77)
        dw, _ = run_bww(wl, x, dy, offset=offset)
        assert_close(dw.double().numpy(), orc.bwd_weight(wl, x, dy), wl.dtype, f"{wl.name} offset {offset}")


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
def test_integer_inputs_exact(orc, dt):
    """Small integers: every product and partial sum is an exact integer in
    fp32 and the results fit the storage type, so dw must equal the oracle."""
    for wl in (inputs.Workload("int_dw", 8, 0, 2, 2, 32, 1, 1, (1, 11, 10), (1, 3, 3), (1, 1, 1), (0, 1, 1),
                               (1, 1, 1), dt, False),
               inputs.Workload("int_grp", 8, 1, 2, 1, 4, 3, 5, (1, 7, 6), (1, 3, 3), (1, 2, 1), (0, 1, 1),
                               (1, 1, 2), dt, False)):
        g = torch.Generator().manual_seed(11)
        tdt = inputs.DTYPES[dt]
        x = torch.randint(-1, 2, wl.x_shape(), generator=g).to(tdt)
        dy = torch.randint(-1, 2, out_shape_of(wl), generator=g).to(tdt)
        ref = orc.bwd_weight(wl, x, dy)
        assert np.abs(ref).max() < 256  # exact in every storage type
        dw, _ = run_bww(wl, x, dy)
        assert np.array_equal(dw.double().numpy(), ref), wl.name


def test_deterministic():
    """Two calls on the same inputs give the same bits."""
    wl = inputs.by_name("resnext_a_bf16").with_(N=4, bias=False)
    x, _, _ = inputs.make_inputs(wl)
    dy = make_dy(wl, 9)
    a, _ = run_bww(wl, x, dy)
    b, _ = run_bww(wl, x, dy)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
