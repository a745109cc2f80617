"""Backward weight (the gradient with respect to w) through the C ABI,
against the oracle's fp64 backward weight, element by element.

* every workload family at reduced batch, and four at full size;
* the tensor-core route (16-bit, Cg == Kg dividing 64, C % 64 == 0) on the
  families it takes, forced against the FFMA route, and on random problems
  over its shape range (strides 1 and 2, dilation, padding, 3D, odd widths);
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


def tc_route(wl):
    """The shapes the tensor-core route takes (the FFMA route runs the rest)."""
    return (wl.dtype != "f32" and wl.Cg == wl.Kg and 64 % wl.Cg == 0 and (wl.G * wl.Cg) % 64 == 0
            and wl.stride[1] == wl.stride[2] and wl.stride[1] <= 2 and wl.ker[2] <= 4)


def run_bww(wl, x, dy, offset=0, force=0):
    """dw on the host and the selected kernel; x and dy start `offset`
    elements into their allocations; `force` is gconv_options.force_kernel."""
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
    opt.force_kernel = force
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
    assert sel == (B.KERNEL_IGEMM_TC if tc_route(wl) else B.KERNEL_BWD_WEIGHT), sel
    assert_close(dw.double().numpy(), orc.bwd_weight(wl, x, dy), wl.dtype, name)


@pytest.mark.parametrize("name", ["mbv2_dw_s1_f16", "resnext_b_bf16", "resnext3d_n8_f16", "sweep_g64_d1_s1_bf16"])
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


TC_FAMILY = ["resnext_a_bf16", "resnext_b_bf16", "sweep_g512_d1_s2_bf16", "sweep_g256_d2_s2_bf16",
             "sweep_g64_d2_s1_bf16", "sweep_g32_d1_s2_bf16", "sweep_g8_d1_s1_bf16"]


@pytest.mark.parametrize("name", TC_FAMILY)
def test_tc_route_against_ffma_route(orc, name):
    """Both routes, forced, on the same inputs: each within tolerance of the
    oracle."""
    wl = inputs.by_name(name).with_(N=2, bias=False)
    assert tc_route(wl)
    x, _, _ = inputs.make_inputs(wl)
    dy = make_dy(wl, 700 + wl.variant)
    ref = orc.bwd_weight(wl, x, dy)
    dw_tc, sel_tc = run_bww(wl, x, dy, force=B.KERNEL_IGEMM_TC)
    dw_ff, sel_ff = run_bww(wl, x, dy, force=B.KERNEL_BWD_WEIGHT)
    assert (sel_tc, sel_ff) == (B.KERNEL_IGEMM_TC, B.KERNEL_BWD_WEIGHT)
    assert_close(dw_tc.double().numpy(), ref, wl.dtype, f"{name} tensor cores")
    assert_close(dw_ff.double().numpy(), ref, wl.dtype, f"{name} FFMA")


def _tc_problem(rng, i):
    Cg = int(rng.choice([1, 2, 4, 8, 16, 32, 64]))
    G = 64 // Cg * int(rng.integers(1, 3))
    nd = 3 if i % 5 == 4 else 2
    s = int(rng.integers(1, 3))
    k = int(rng.integers(1, 5))
    d = int(rng.integers(1, 3))
    hw = (int(rng.integers(3, 24)), int(rng.integers(3, 40)))
    inp = (int(rng.integers(3, 7)) if nd == 3 else 1, *hw)
    ker = (int(rng.integers(1, 4)) if nd == 3 else 1, k, k)
    pad = (int(rng.integers(0, 2)) if nd == 3 else 0, int(rng.integers(0, k)), int(rng.integers(0, k)))
    strides = (int(rng.integers(1, 3)) if nd == 3 else 1, s, s)
    return inputs.Workload(f"tcbw{i}", 9, i, nd, int(rng.integers(1, 4)), G, Cg, Cg, inp, ker, strides, pad,
                           (1, d, d), "bf16" if i % 2 else "f16", False)


@pytest.mark.parametrize("seed", range(30))
def test_tc_random_problems(orc, seed):
    """Random problems across the tensor-core route's range, forced onto it."""
    rng = np.random.default_rng(8100 + seed)
    def extents(w):
        return [(w.inp[i] + 2 * w.pad[i] - w.dil[i] * (w.ker[i] - 1) - 1) // w.stride[i] + 1 for i in range(3)]

    wl = _tc_problem(rng, seed)
    while min(extents(wl)) < 1:
        wl = _tc_problem(rng, seed)
    x, _, _ = inputs.make_inputs(wl)
    dy = make_dy(wl, 8200 + seed)
    dw, sel = run_bww(wl, x, dy, force=B.KERNEL_IGEMM_TC)
    assert sel == B.KERNEL_IGEMM_TC
    assert_close(dw.double().numpy(), orc.bwd_weight(wl, x, dy), wl.dtype, f"seed {seed}: {wl}")


def test_tc_integer_inputs_exact(orc):
    """Integer inputs on the tensor-core route: exact like the FFMA route."""
    for wl in (inputs.Workload("int_tc", 8, 2, 2, 2, 16, 4, 4, (1, 9, 13), (1, 3, 3), (1, 1, 1), (0, 1, 1),
                               (1, 1, 1), "bf16", False),
               inputs.Workload("int_tc2", 8, 3, 2, 1, 2, 32, 32, (1, 12, 11), (1, 3, 3), (1, 2, 2), (0, 1, 1),
                               (1, 1, 1), "f16", False)):
        g = torch.Generator().manual_seed(12)
        tdt = inputs.DTYPES[wl.dtype]
        x = torch.randint(-1, 2, wl.x_shape(), generator=g).to(tdt)
        dy = torch.randint(-1, 2, out_shape_of(wl), generator=g).to(tdt)
        ref = orc.bwd_weight(wl, x, dy)
        assert np.abs(ref).max() < 256
        dw, sel = run_bww(wl, x, dy, force=B.KERNEL_IGEMM_TC)
        assert sel == B.KERNEL_IGEMM_TC
        assert np.array_equal(dw.double().numpy(), ref), wl.name


def test_tc_deterministic_and_misaligned_fallback(orc):
    """Two tensor-core calls give the same bits; misaligned x falls back to
    the FFMA route with the same workspace."""
    wl = inputs.by_name("resnext_b_bf16").with_(N=2, bias=False)
    x, _, _ = inputs.make_inputs(wl)
    dy = make_dy(wl, 31)
    a, sa = run_bww(wl, x, dy)
    b, _ = run_bww(wl, x, dy)
    assert sa == B.KERNEL_IGEMM_TC
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    c, sc = run_bww(wl, x, dy, offset=1)
    assert sc == B.KERNEL_BWD_WEIGHT
    assert_close(c.double().numpy(), orc.bwd_weight(wl, x, dy), wl.dtype, "misaligned")

