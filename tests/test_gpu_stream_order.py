"""Stream order under programmatic dependent launch, through the C ABI.

By default every kernel is launched so that its CTAs may start while the
previous kernel in the stream is still running; it may touch global memory
only once that kernel has completed.  These tests launch chains of dependent
convolutions back to back, with no host synchronisation in between, and
check each result against the oracle:

* read after write: each convolution reads the previous one's output;
* write after read: a convolution overwrites the input that the previous
  one reads;

over the depthwise, tensor-core and generic kernels, with the dependent
launch on (default) and off (``serial_launch = 1``).  Intermediate buffers
start as NaN, so a read that runs ahead of its producer shows.
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


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _launch(wl, x, w, b, y, force, serial, stream):
    opt = B.gconv_options()
    opt.force_kernel = force
    opt.serial_launch = serial
    gc.grouped_conv_fwd_ex(x, w, b, y, gc.problem_of(wl), gc.DTYPE_CODES[wl.dtype], stream, opt)
    return opt.selected


def _nan_buffer(shape, dtype):
    t = torch.empty(shape, dtype=dtype, device=DEV)
    t.view(torch.uint8).fill_(0xFF)  # NaN in fp16 / bf16
    return t


def _stage(name, N, G, Cg, Kg, hw, dtype, variant):
    """A 3x3, stride-1, pad-1 convolution that keeps the image shape, so
    stages can feed one another."""
    return inputs.Workload(name, 90, variant, 2, N, G, Cg, Kg, (1, hw, hw), (1, 3, 3), (1, 1, 1), (0, 1, 1),
                           (1, 1, 1), dtype, True)


# (stage workloads, forced kernel per stage: 1 depthwise, 2 generic, 3 tensor core)
CHAINS = {
    # MobileNetV2 depthwise at its full size: 2 CTAs per SM fill the GPU, so
    # the dependent grid's CTAs start as the producer's CTAs retire
    "dw_dw": ([_stage("dw_a", 32, 144, 1, 1, 56, "f16", 0), _stage("dw_b", 32, 144, 1, 1, 56, "f16", 1)],
              [1, 1]),
    "dw_tc_generic_dw": ([_stage("m_dw", 8, 256, 1, 1, 28, "bf16", 2), _stage("m_tc", 8, 8, 32, 32, 28, "bf16", 3),
                          _stage("m_gen", 2, 8, 32, 32, 28, "bf16", 4), _stage("m_dw2", 2, 256, 1, 1, 28, "bf16", 5)],
                         [1, 3, 2, 1]),
}


@pytest.mark.parametrize("serial", [0, 1], ids=["pdl", "serial"])
@pytest.mark.parametrize("chain", list(CHAINS))
def test_read_after_write_chain(orc, chain, serial):
    stages, forces = CHAINS[chain]
    s = torch.cuda.Stream(DEV)
    params = []
    for wl in stages:
        _, w, b = inputs.make_inputs(wl)
        params.append((w.to(DEV), b.to(DEV)))
    x0, _, _ = inputs.make_inputs(stages[0])
    # later stages may use a smaller batch: they read the leading images
    acts = [x0.to(DEV)]
    with torch.cuda.stream(s):
        for wl in stages:
            acts.append(_nan_buffer(out_shape_of(wl), inputs.DTYPES[wl.dtype]))
    s.synchronize()
    selected = []
    for i, wl in enumerate(stages):
        xin = acts[i][: wl.N]
        selected.append(_launch(wl, xin, params[i][0], params[i][1], acts[i + 1], forces[i], serial, s))
    s.synchronize()
    assert selected == forces
    for i, wl in enumerate(stages):
        xin = acts[i][: wl.N].cpu()
        ref = orc.forward(wl, xin, params[i][0].cpu(), params[i][1].cpu())
        assert_close(acts[i + 1].cpu().double().numpy(), ref, wl.dtype, f"{chain} stage {i} ({wl.name})")


@pytest.mark.parametrize("serial", [0, 1], ids=["pdl", "serial"])
@pytest.mark.parametrize("force", [1, 3, 2], ids=["depthwise", "tensor_core", "generic"])
def test_write_after_read(orc, force, serial):
    """Convolution 1 reads A and writes B; convolution 2, launched right
    after it, writes A.  B must be the convolution of A's original values."""
    if force == 1:
        wl = _stage("war_dw", 32, 144, 1, 1, 56, "f16", 6)
    elif force == 3:
        wl = _stage("war_tc", 8, 8, 32, 32, 28, "bf16", 7)
    else:
        wl = _stage("war_gen", 2, 8, 32, 32, 28, "bf16", 8)
    wl2 = wl.with_(variant=9)
    x, w, b = inputs.make_inputs(wl)
    x2, w2, b2 = inputs.make_inputs(wl2)
    s = torch.cuda.Stream(DEV)
    with torch.cuda.stream(s):
        A = x.to(DEV)
        Bout = _nan_buffer(out_shape_of(wl), inputs.DTYPES[wl.dtype])
        X2 = x2.to(DEV)
        wd, bd, w2d, b2d = w.to(DEV), b.to(DEV), w2.to(DEV), b2.to(DEV)
    s.synchronize()
    _launch(wl, A, wd, bd, Bout, force, serial, s)
    _launch(wl2, X2, w2d, b2d, A.view(out_shape_of(wl2)), force, serial, s)
    s.synchronize()
    assert_close(Bout.cpu().double().numpy(), orc.forward(wl, x, w, b), wl.dtype, "convolution 1 (reads A)")
    assert_close(A.cpu().double().numpy().reshape(out_shape_of(wl2)), orc.forward(wl2, x2, w2, b2), wl.dtype,
                 "convolution 2 (writes A)")


def test_serial_launch_matches_default(orc):
    """Both launch modes give bit-identical outputs (same kernels, same order
    of arithmetic)."""
    wl = inputs.by_name("resnext_b_bf16").with_(N=2)
    x, w, b = inputs.make_inputs(wl)
    s = torch.cuda.current_stream(DEV)
    xd, wd, bd = x.to(DEV), w.to(DEV), b.to(DEV)
    outs = []
    for serial in (0, 1):
        y = _nan_buffer(out_shape_of(wl), inputs.DTYPES[wl.dtype])
        _launch(wl, xd, wd, bd, y, 0, serial, s)
        outs.append(y)
    torch.cuda.synchronize(DEV)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert np.isfinite(outs[0].cpu().double().numpy()).all()
