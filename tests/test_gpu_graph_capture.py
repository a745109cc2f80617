"""The C-ABI calls inside a CUDA graph: capture a forward depthwise, a
forward tensor-core and a backward-data call once, then replay the graph over
new input values copied into the captured buffers, and compare every output
with the oracle after each replay (the batch-1 launch-overhead path: one graph
launch for a sequence of layers)."""
import pytest
import torch

import depthwise_convolution_forward_gb300 as gc
from depthwise_convolution_forward_gb300 import inputs
from gpu_util import assert_close, out_shape_of, require_gpu

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def test_capture_and_replay(orc):
    dw = inputs.by_name("mbv2_dw_s1_f16").with_(N=2)
    tc = inputs.by_name("resnext_b_bf16").with_(N=2)
    bw = inputs.by_name("resnext_a_bf16").with_(N=1, bias=False)
    cases = []
    for wl in (dw, tc):
        x, w, b = inputs.make_inputs(wl)
        cases.append(dict(wl=wl, x=x.to(DEV), w=w.to(DEV), b=b.to(DEV),
                          y=torch.empty(out_shape_of(wl), dtype=x.dtype, device=DEV)))
    _, wb, _ = inputs.make_inputs(bw)
    dy = torch.empty(out_shape_of(bw), dtype=wb.dtype, device=DEV)
    wbd = wb.to(DEV)
    dx = torch.empty(bw.x_shape(), dtype=wb.dtype, device=DEV)
    need = gc.grouped_conv_bwd_data_workspace_size(gc.problem_of(bw), gc.DTYPE_CODES[bw.dtype])
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=DEV)

    s = torch.cuda.Stream(DEV)
    graph = torch.cuda.CUDAGraph()
    s.wait_stream(torch.cuda.current_stream(DEV))
    with torch.cuda.stream(s):
        for c in cases:  # warm-up outside capture: plans cached, attributes set
            gc.grouped_conv_fwd(c["x"], c["w"], c["b"], c["y"], gc.problem_of(c["wl"]),
                                gc.DTYPE_CODES[c["wl"].dtype], s)
        gc.grouped_conv_bwd_data(dy, wbd, dx, gc.problem_of(bw), gc.DTYPE_CODES[bw.dtype], ws, need, s)
    s.synchronize()
    with torch.cuda.graph(graph, stream=s):
        for c in cases:
            gc.grouped_conv_fwd(c["x"], c["w"], c["b"], c["y"], gc.problem_of(c["wl"]),
                                gc.DTYPE_CODES[c["wl"].dtype], s)
        gc.grouped_conv_bwd_data(dy, wbd, dx, gc.problem_of(bw), gc.DTYPE_CODES[bw.dtype], ws, need, s)

    for rep in range(3):
        gen = torch.Generator().manual_seed(4242 + rep)
        host = []
        for c in cases:
            xh = (torch.rand(c["x"].shape, generator=gen) * 2 - 1).to(c["x"].dtype)
            c["x"].copy_(xh)
            host.append(xh)
        dyh = (torch.rand(dy.shape, generator=gen) * 2 - 1).to(dy.dtype)
        dy.copy_(dyh)
        c_y = [c["y"] for c in cases]
        for y in c_y:
            y.fill_(float("nan"))
        dx.fill_(float("nan"))
        torch.cuda.synchronize(DEV)
        graph.replay()
        torch.cuda.synchronize(DEV)
        for c, xh in zip(cases, host):
            ref = orc.forward(c["wl"], xh, c["w"].cpu(), c["b"].cpu())
            assert_close(c["y"].cpu().double().numpy(), ref, c["wl"].dtype, f"replay {rep}: {c['wl'].name}")
        assert_close(dx.cpu().double().numpy(), orc.bwd_data(bw, dyh, wb), bw.dtype, f"replay {rep}: bwd data")


FIRST_CALL_SCRIPT = r"""
import sys
sys.path.insert(0, {root!r})
sys.path.insert(0, {tests!r})
import numpy as np
import torch
import depthwise_convolution_forward_gb300 as gc
from depthwise_convolution_forward_gb300 import inputs
import oracle
from gpu_util import out_shape_of, TOL
dev = torch.device("cuda:0")
torch.zeros(1, device=dev)
cases = []
for name in ("mbv2_dw_s2_f16", "resnext_b_bf16", "grouped2d_f32_smoke"):
    wl = inputs.by_name(name).with_(N=1)
    x, w, b = inputs.make_inputs(wl)
    cases.append((wl, x, w, b, x.to(dev), w.to(dev), b.to(dev) if b is not None else None,
                  torch.full(out_shape_of(wl), float("nan"), dtype=x.dtype, device=dev)))
s = torch.cuda.Stream(dev)
s.wait_stream(torch.cuda.current_stream(dev))
torch.cuda.synchronize(dev)
g = torch.cuda.CUDAGraph()
with torch.cuda.graph(g, stream=s):  # the library's first calls in this process
    for wl, _, _, _, xd, wd, bd, yd in cases:
        gc.grouped_conv_fwd(xd, wd, bd, yd, gc.problem_of(wl), gc.DTYPE_CODES[wl.dtype], s)
g.replay()
torch.cuda.synchronize(dev)
orc = oracle.get()
for wl, x, w, b, _, _, _, yd in cases:
    ref = orc.forward(wl, x, w, b)
    got = yd.cpu().double().numpy()
    atol, rtol = TOL[wl.dtype]
    ok = np.all(np.isfinite(got)) and np.all(np.abs(got - ref) <= atol + rtol * np.abs(ref))
    print(wl.name, "ok" if ok else "MISMATCH")
"""


def test_first_call_inside_capture():
    """A fresh process whose first library calls are made inside a stream
    capture (torch.cuda.graph, global capture mode): the per-device set-up
    does nothing that a capture forbids, and the replayed graph computes the
    right outputs on the depthwise, tensor-core and generic kernels."""
    import os
    import subprocess
    import sys

    here = os.path.dirname(os.path.abspath(__file__))
    code = FIRST_CALL_SCRIPT.format(root=os.path.dirname(here), tests=here)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.endswith(("ok", "MISMATCH"))]
    assert len(lines) == 3 and all(ln.endswith(" ok") for ln in lines), r.stdout
