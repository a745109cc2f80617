"""Maximum-size problems: x and y hold more than 2^31 elements, so every
element offset past the boundary needs 64-bit arithmetic.

Inputs are drawn on the device from a seeded generator (4.3 GB per tensor).
The oracle then checks whole images as N=1 problems: the first image, the
image that straddles element 2^31 of x and of y, and the last image.  Each
kernel is forced in turn: the depthwise kernel and the generic kernel on a
MobileNetV2-shaped depthwise problem, the tensor-core kernel on a grouped
sweep shape.
"""
import numpy as np
import pytest
import torch

import depthwise_convolution_forward_gb300 as gc
from depthwise_convolution_forward_gb300 import _binding as B
from depthwise_convolution_forward_gb300 import inputs
from gpu_util import assert_close, out_shape_of, require_gpu

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
LIMIT = 2 ** 31
GUARD = 4096


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _images_to_check(n_images, per_image_x, per_image_y):
    return sorted({0, LIMIT // per_image_x, LIMIT // per_image_y, n_images - 1})


CASES = {
    # name: (workload, forced kernel)
    "depthwise": (inputs.by_name("mbv2_dw_s1_f16").with_(N=4800), B.KERNEL_DIRECT_DW),
    "generic": (inputs.by_name("mbv2_dw_s1_f16").with_(N=4800), B.KERNEL_DIRECT_GENERIC),
    "tensor_core": (inputs.by_name("sweep_g32_d1_s1_bf16").with_(N=5400), B.KERNEL_IGEMM_TC),
}


@pytest.mark.parametrize("case", list(CASES))
def test_more_than_2_31_elements(orc, case):
    wl, force = CASES[case]
    dt = inputs.DTYPES[wl.dtype]
    xshape = wl.x_shape()
    yshape = out_shape_of(wl)
    nx, ny = int(np.prod(xshape)), int(np.prod(yshape))
    assert nx > LIMIT and ny > LIMIT
    g = torch.Generator(device=DEV)
    g.manual_seed(7000 + wl.cfg)
    x = torch.rand(xshape, generator=g, dtype=dt, device=DEV).mul_(2).sub_(1)
    _, w, b = inputs.make_inputs(wl.with_(N=1))  # weights and bias do not depend on N
    wd, bd = w.to(DEV), b.to(DEV)
    buf = torch.empty(ny + 2 * GUARD, dtype=dt, device=DEV)
    buf.view(torch.int16).fill_(-1)
    y = buf[GUARD:GUARD + ny].view(yshape)
    opt = B.gconv_options()
    opt.force_kernel = force
    opt.debug = 1
    gc.grouped_conv_fwd_ex(x, wd, bd, y, gc.problem_of(wl), gc.DTYPE_CODES[wl.dtype],
                           torch.cuda.current_stream(DEV), opt)
    torch.cuda.synchronize(DEV)
    assert opt.selected == force
    assert bool((buf[:GUARD].view(torch.int16) == -1).all()), "wrote before y"
    assert bool((buf[GUARD + ny:].view(torch.int16) == -1).all()), "wrote after y"
    one = wl.with_(N=1)
    per_x, per_y = nx // wl.N, ny // wl.N
    for n in _images_to_check(wl.N, per_x, per_y):
        ref = orc.forward(one, x[n:n + 1].cpu(), w, b)
        got = y[n:n + 1].cpu().double().numpy()
        assert_close(got, ref, wl.dtype, f"{case}: image {n} of {wl.N} (x offset {n * per_x}, y offset {n * per_y})")
    del x, y, buf
    torch.cuda.empty_cache()
