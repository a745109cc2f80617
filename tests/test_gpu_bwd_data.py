"""Backward data (the gradient with respect to x) through the C ABI, against
the oracle's fp64 adjoint, element by element.

* every workload family at reduced batch, on the route the library picks:
  stride 1 runs the forward kernels on transposed, flipped weights (depthwise,
  tensor-core or generic), other strides the direct gather kernel;
* three workloads at full size;
* the same stride-1 problems forced onto the direct kernel, so both routes
  are checked on one problem;
* random small 2D/3D problems over all dtypes;
* canary bands around dx.
"""
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


def make_dy(wl, seed):
    """dy ~ U(-1, 1) in the forward output layout, drawn in fp32 on the host
    and rounded once to the storage dtype."""
    g = torch.Generator().manual_seed(seed)
    return (torch.rand(out_shape_of(wl), generator=g, dtype=torch.float32) * 2 - 1).to(inputs.DTYPES[wl.dtype])


def run_bwd(wl, dy, w, force=0, test_flags=0):
    """dx on the host and the kernel that produced it (test_flags bit 1: one
    launch per stride phase instead of the stacked launch)."""
    dt = inputs.DTYPES[wl.dtype]
    p = gc.problem_of(wl)
    code = gc.DTYPE_CODES[wl.dtype]
    dyd, wd = dy.to(DEV), w.to(DEV)
    n = int(np.prod(wl.x_shape()))
    buf = torch.empty(n + 2 * GUARD, dtype=dt, device=DEV)
    words = torch.int32 if dt == torch.float32 else torch.int16
    buf.view(words).fill_(-1)
    dx = buf[GUARD:GUARD + n].view(wl.x_shape())
    need = gc.grouped_conv_bwd_data_workspace_size(p, code)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=DEV) if need else None
    opt = B.gconv_options()
    opt.force_kernel = force
    opt.test_flags = test_flags
    opt.debug = 1
    gc.grouped_conv_bwd_data_ex(dyd, wd, dx, p, code, ws, need, torch.cuda.current_stream(DEV), opt)
    torch.cuda.synchronize(DEV)
    assert bool((buf[:GUARD].view(words) == -1).all()), "wrote before dx"
    assert bool((buf[GUARD + n:].view(words) == -1).all()), "wrote after dx"
    return dx.cpu(), opt.selected, need


def _reduced(wl):
    return wl.with_(N=min(wl.N, 2))


FAMILY = ["mbv2_dw_s1_f16", "mbv2_dw_s2_f16", "resnext_a_bf16", "resnext_b_bf16", "resnext3d_n1_f16",
          "grouped2d_f32_smoke", "sweep_g8_d2_s1_bf16", "sweep_g64_d1_s1_bf16", "sweep_g256_d2_s2_bf16",
          "sweep_g512_d2_s1_bf16", "sweep_g8_d1_s2_bf16", "sweep_g32_d1_s2_bf16", "sweep_g64_d2_s2_bf16",
          "sweep_g512_d1_s2_bf16"]


def _expected_route(wl):
    """The route the library reports (0 direct gather, 1 stride-1
    transposed weights, 2 stride phases); stride-1 problems with
    pad <= dil*(k-1) always take route 1."""
    route, _ = gc.grouped_conv_bwd_data_route(gc.problem_of(wl), gc.DTYPE_CODES[wl.dtype])
    stride1 = all(s == 1 for s in wl.stride)
    fits = all(p <= d * (k - 1) for p, d, k in zip(wl.pad, wl.dil, wl.ker))
    assert (route == 1) == (stride1 and fits)
    return route


@pytest.mark.parametrize("name", FAMILY)
def test_reduced_batch_full_compare(orc, name):
    wl = _reduced(inputs.by_name(name))
    _, w, _ = inputs.make_inputs(wl)
    dy = make_dy(wl, 9000 + wl.cfg * 10 + wl.variant)
    dx, sel, need = run_bwd(wl, dy, w)
    route = _expected_route(wl)
    assert (sel != B.KERNEL_BWD_DATA_DIRECT) == (route != 0), (name, sel)
    assert (need > 0) == (route != 0)
    assert_close(dx.double().numpy(), orc.bwd_data(wl, dy, w), wl.dtype, f"{name} (kernel {sel})")


@pytest.mark.parametrize("name", ["mbv2_dw_s1_f16", "resnext_a_bf16", "resnext_b_bf16"])
def test_full_size(orc, name):
    wl = inputs.by_name(name)
    _, w, _ = inputs.make_inputs(wl)
    dy = make_dy(wl, 9100 + wl.cfg * 10 + wl.variant)
    dx, sel, _ = run_bwd(wl, dy, w)
    assert_close(dx.double().numpy(), orc.bwd_data(wl, dy, w), wl.dtype, f"{name} (kernel {sel})")


@pytest.mark.parametrize("name", ["mbv2_dw_s1_f16", "resnext_a_bf16", "resnext3d_n1_f16", "grouped2d_f32_smoke"])
def test_both_routes(orc, name):
    wl = _reduced(inputs.by_name(name))
    _, w, _ = inputs.make_inputs(wl)
    dy = make_dy(wl, 9200 + wl.cfg * 10 + wl.variant)
    ref = orc.bwd_data(wl, dy, w)
    for force in (0, B.KERNEL_BWD_DATA_DIRECT, B.KERNEL_DIRECT_GENERIC):
        dx, sel, _ = run_bwd(wl, dy, w, force)
        if force:
            assert sel == force
        assert_close(dx.double().numpy(), ref, wl.dtype, f"{name} force {force} (kernel {sel})")


@pytest.mark.parametrize("seed", range(24))
def test_random_small_problems(orc, seed):
    rng = np.random.default_rng(5000 + seed)
    wl = inputs.random_problem(rng)
    _, w, _ = inputs.make_inputs(wl)
    dy = make_dy(wl, 9300 + seed)
    dx, sel, _ = run_bwd(wl, dy, w)
    assert_close(dx.double().numpy(), orc.bwd_data(wl, dy, w), wl.dtype, f"{wl} (kernel {sel})")


PHASE_CASES = [
    # (name, workload): grouped stride-2 problems on the stride-phase route
    inputs.by_name("resnext_b_bf16").with_(N=2, bias=False),
    inputs.by_name("sweep_g256_d2_s2_bf16").with_(N=2, bias=False),
    # odd extents and no padding: phases of unequal size and empty edges
    inputs.Workload("ph_odd", 9, 1, 2, 2, 4, 16, 16, (1, 13, 11), (1, 3, 3), (1, 2, 2), (0, 0, 0), (1, 1, 1),
                    "bf16", False),
    # 5x5 filter, pad 2, f16
    inputs.Workload("ph_k5", 9, 2, 2, 1, 2, 16, 32, (1, 12, 10), (1, 5, 5), (1, 2, 2), (0, 2, 2), (1, 1, 1),
                    "f16", False),
    # dilation 2 with stride 2 (half the phases get no taps), pad 1
    inputs.Workload("ph_d2", 9, 3, 2, 2, 4, 16, 16, (1, 12, 12), (1, 3, 3), (1, 2, 2), (0, 1, 1), (1, 2, 2),
                    "bf16", False),
    # stride 2 in H only, stride 3 in W
    inputs.Workload("ph_s23", 9, 4, 2, 1, 2, 32, 16, (1, 11, 14), (1, 3, 3), (1, 2, 3), (0, 1, 1), (1, 1, 1),
                    "bf16", False),
    # 3D stride 2 in every dimension
    inputs.Workload("ph_3d", 9, 5, 3, 1, 4, 16, 16, (7, 9, 8), (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1),
                    "f16", False),
]


@pytest.mark.parametrize("wl", PHASE_CASES, ids=lambda w: w.name)
def test_stride_phase_route(orc, wl):
    """Stride-phase route: the stacked launch (every phase as output
    channels of one tensor-core problem) and one launch per phase, both
    writing dx directly, against the oracle and the direct kernel."""
    route, launches = gc.grouped_conv_bwd_data_route(gc.problem_of(wl), gc.DTYPE_CODES[wl.dtype])
    assert route == 2 and launches >= 2, (route, launches)
    _, w, _ = inputs.make_inputs(wl)
    dy = make_dy(wl, 9400 + wl.variant)
    ref = orc.bwd_data(wl, dy, w)
    dx, sel, need = run_bwd(wl, dy, w)
    assert need > 0 and sel == B.KERNEL_IGEMM_TC
    assert_close(dx.double().numpy(), ref, wl.dtype, f"{wl.name} stacked phases (kernel {sel})")
    dx1, sel1, _ = run_bwd(wl, dy, w, test_flags=2)
    assert sel1 == B.KERNEL_IGEMM_TC
    assert_close(dx1.double().numpy(), ref, wl.dtype, f"{wl.name} one launch per phase (kernel {sel1})")
    dx2, sel2, _ = run_bwd(wl, dy, w, B.KERNEL_BWD_DATA_DIRECT)
    assert sel2 == B.KERNEL_BWD_DATA_DIRECT
    assert_close(dx2.double().numpy(), ref, wl.dtype, f"{wl.name} direct")


@pytest.mark.parametrize("wl", PHASE_CASES[:3] + PHASE_CASES[-1:], ids=lambda w: w.name)
def test_stride_phase_buffered_placement(orc, wl):
    """A phase kernel that cannot write dx itself (the generic kernel,
    forced) goes through the workspace's phase buffer and the scatter copy:
    same dx."""
    _, w, _ = inputs.make_inputs(wl)
    dy = make_dy(wl, 9450 + wl.variant)
    dx, sel, _ = run_bwd(wl, dy, w, force=B.KERNEL_DIRECT_GENERIC)
    assert sel == B.KERNEL_DIRECT_GENERIC
    assert_close(dx.double().numpy(), orc.bwd_data(wl, dy, w), wl.dtype, f"{wl.name} buffered phases")
