"""Failure detection without faulting the GPU: a copy is withheld on
purpose so the kernel's first bounded wait cannot complete; the kernel must
report a timeout through its status word, return, and leave the context
usable for the next, correct call."""
import pytest
import torch

import depthwise_convolution_forward_gb300 as gc
from depthwise_convolution_forward_gb300 import _binding as B
from depthwise_convolution_forward_gb300 import inputs
from gpu_util import assert_close, out_shape_of, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _call(wl, x, w, b, y, test_flags, debug, limit_ns=2_000_000, force=0):
    opt = B.gconv_options()
    opt.debug = debug
    opt.test_flags = test_flags
    opt.wait_limit_ns = limit_ns
    opt.force_kernel = force
    return gc.grouped_conv_fwd_ex(x, w, b, y, gc.problem_of(wl), gc.DTYPE_CODES[wl.dtype],
                                  torch.cuda.current_stream(), opt)


@pytest.mark.parametrize("name", ["mbv2_dw_s1_f16"])
def test_withheld_copy_times_out_then_recovers(orc, name):
    wl = inputs.by_name(name).with_(N=2)
    x, w, b = inputs.make_inputs(wl)
    dev = torch.device("cuda:0")
    xd, wd, bd = x.to(dev), w.to(dev), b.to(dev)
    y = torch.zeros(out_shape_of(wl), dtype=x.dtype, device=dev)
    with pytest.raises(gc.GconvError) as e:
        _call(wl, xd, wd, bd, y, test_flags=1, debug=1)
    assert e.value.status == B.GCONV_ERR_TIMEOUT
    # status word was cleared by the debug read
    assert gc.gconv_device_status(torch.cuda.current_stream()) == (0, 0)
    # without debug the call returns OK and the status word records the expiry
    _call(wl, xd, wd, bd, y, test_flags=1, debug=0)
    code, where = gc.gconv_device_status(torch.cuda.current_stream())
    assert code == 1 and where != 0
    # the context is still healthy: a normal call is correct
    _call(wl, xd, wd, bd, y, test_flags=0, debug=1)
    torch.cuda.synchronize()
    assert_close(y.cpu().double().numpy(), orc.forward(wl, x, w, b), wl.dtype, "after timeout")
