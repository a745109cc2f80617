"""grouped_conv_bwd_data_noalloc: backward data for callers that may not
allocate device memory while they run (an engine plugin enqueued on a stream
it does not own, a runtime that reserves all memory up front).  The library's
fixed scratch array replaces the caller's workspace; the result must match
grouped_conv_bwd_data with a workspace, on two calls in a row (the second
call finds the first call's contents in the shared array).

This file is collected last, so a run that stops at the first failure has
run every other test before it; it passes alone in a fresh process too.
"""
import ctypes

import numpy as np
import pytest
import torch

import depthwise_convolution_forward_gb300 as gc
from depthwise_convolution_forward_gb300 import _binding as B
from depthwise_convolution_forward_gb300 import inputs
from gpu_util import TOL, out_shape_of, require_gpu

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _dy(wl, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.rand(out_shape_of(wl), generator=g, dtype=torch.float32) * 2 - 1).to(inputs.DTYPES[wl.dtype])


# stride-1 problems use the scratch (transposed, flipped weights) on the
# depthwise, tensor-core and generic kernels; the depthwise stride-2 one
# needs none; the grouped stride-2 one would need more than the fixed array
# on its stride-phase route and runs on the direct kernel instead
CASES = ["mbv2_dw_s1_f16", "resnext_a_bf16", "sweep_g8_d1_s1_bf16", "grouped2d_f32_smoke", "mbv2_dw_s2_f16",
         "resnext_b_bf16"]


@pytest.mark.parametrize("name", CASES)
def test_noalloc_matches_workspace_call(name):
    wl = inputs.by_name(name)
    wl = wl.with_(N=min(wl.N, 2), bias=False)
    _, w, _ = inputs.make_inputs(wl)
    p = gc.problem_of(wl)
    code = gc.DTYPE_CODES[wl.dtype]
    lib = B.load_library()
    need = gc.grouped_conv_bwd_data_workspace_size(p, code)
    if name == "resnext_b_bf16":
        assert need > B.GCONV_NOALLOC_SCRATCH_BYTES
    else:
        assert need <= B.GCONV_NOALLOC_SCRATCH_BYTES
    if name != "mbv2_dw_s2_f16":
        assert need > 0
    wd = w.to(DEV)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=DEV)
    s = torch.cuda.current_stream(DEV)
    atol, rtol = TOL[wl.dtype]
    for call in range(2):  # two calls in a row, new dy each time
        dy = _dy(wl, 700 + call).to(DEV)
        dx_ref = torch.full(wl.x_shape(), float("nan"), dtype=w.dtype, device=DEV)
        dx = torch.full(wl.x_shape(), float("nan"), dtype=w.dtype, device=DEV)
        gc.grouped_conv_bwd_data(dy, wd, dx_ref, p, code, ws, need, s)
        st = lib.grouped_conv_bwd_data_noalloc(dy.data_ptr(), wd.data_ptr(), dx.data_ptr(), ctypes.byref(p), code,
                                               s.cuda_stream)
        assert st == 0, gc.gconv_last_error()
        torch.cuda.synchronize(DEV)
        got = dx.cpu().double().numpy()
        ref = dx_ref.cpu().double().numpy()
        assert np.all(np.isfinite(got)), f"{name} call {call}: non-finite output"
        bad = np.abs(got - ref) > atol + rtol * np.abs(ref)
        assert not bad.any(), f"{name} call {call}: {bad.sum()} elements differ"


def test_noalloc_rejects_scratch_beyond_limit():
    """A stride-1 problem whose transposed weights exceed the fixed scratch
    is refused before any launch, with a reason."""
    wl = inputs.Workload("big_w", 9, 0, 2, 1, 4, 256, 256, (1, 8, 8), (1, 3, 3), (1, 1, 1), (0, 1, 1),
                         (1, 1, 1), "bf16", False)
    p = gc.problem_of(wl)
    code = gc.DTYPE_CODES[wl.dtype]
    assert gc.grouped_conv_bwd_data_workspace_size(p, code) > B.GCONV_NOALLOC_SCRATCH_BYTES
    lib = B.load_library()
    dy = torch.zeros(out_shape_of(wl), dtype=torch.bfloat16, device=DEV)
    w = torch.zeros(wl.w_shape(), dtype=torch.bfloat16, device=DEV)
    dx = torch.zeros(wl.x_shape(), dtype=torch.bfloat16, device=DEV)
    st = lib.grouped_conv_bwd_data_noalloc(dy.data_ptr(), w.data_ptr(), dx.data_ptr(), ctypes.byref(p), code,
                                           torch.cuda.current_stream(DEV).cuda_stream)
    assert st == B.GCONV_ERR_UNSUPPORTED
    assert "scratch" in gc.gconv_last_error()
