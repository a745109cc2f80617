"""Helpers shared by the GPU tests: run the CUDA path through the C ABI with
guard bands around the output, and compare against the oracle."""
from __future__ import annotations

import numpy as np
import torch

import depthwise_convolution_forward_gb300 as gc
from depthwise_convolution_forward_gb300 import _binding as B
from depthwise_convolution_forward_gb300 import build, inputs

# spec tolerances: |gpu - ref| <= atol + rtol * |ref| (fp32 accumulation)
TOL = {"f16": (1e-3, 1e-2), "bf16": (1e-2, 2e-2), "f32": (1e-5, 1e-5)}
GUARD = 4096  # elements of canary on each side of y


def require_gpu():
    if not torch.cuda.is_available():
        raise RuntimeError("GPU tests need a CUDA device")
    build.build()
    B.load_library()


def out_shape_of(wl):
    Do, Ho, Wo = gc.grouped_conv_out_shape(gc.problem_of(wl))
    if wl.ndim == 2:
        return (wl.N, Ho, Wo, wl.G, wl.Kg)
    return (wl.N, Do, Ho, Wo, wl.G, wl.Kg)


def run_gpu(wl, x, w, b, force=0, tile=None, debug=True, stream=None, x_offset=0):
    """Run one forward pass on cuda:0; returns (y on host as torch, selected kernel).

    The output sits between two canary bands that must survive the call.
    ``x_offset`` (elements) shifts x inside its allocation to test alignment.
    """
    dev = torch.device("cuda:0")
    dt = inputs.DTYPES[wl.dtype]
    if x_offset:
        xbuf = torch.empty(x.numel() + x_offset, dtype=dt, device=dev)
        xd = xbuf[x_offset:].view(x.shape)
        xd.copy_(x)
    else:
        xd = x.to(dev)
    wd = w.to(dev)
    bd = b.to(dev) if b is not None else None
    shape = out_shape_of(wl)
    n = int(np.prod(shape))
    buf = torch.empty(n + 2 * GUARD, dtype=dt, device=dev)
    buf.view(torch.uint8 if dt != torch.float32 else torch.int32).fill_(-1 if dt == torch.float32 else 0xFF)
    canary = buf[:GUARD].clone()
    y = buf[GUARD:GUARD + n].view(shape)
    opt = B.gconv_options()
    opt.force_kernel = force
    opt.debug = 1 if debug else 0
    if tile:
        for i, t in enumerate(tile):
            opt.tile[i] = t
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    gc.grouped_conv_fwd_ex(xd, wd, bd, y, gc.problem_of(wl), gc.DTYPE_CODES[wl.dtype], s, opt)
    torch.cuda.synchronize(dev)
    assert torch.equal(buf[:GUARD].view(torch.int16 if dt != torch.float32 else torch.int32),
                       canary.view(torch.int16 if dt != torch.float32 else torch.int32)), "wrote before y"
    assert torch.equal(buf[GUARD + n:].view(torch.int16 if dt != torch.float32 else torch.int32),
                       canary.view(torch.int16 if dt != torch.float32 else torch.int32)), "wrote after y"
    return y.cpu(), opt.selected


def assert_close(got, ref, dtype, what=""):
    atol, rtol = TOL[dtype]
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - r)
    lim = atol + rtol * np.abs(r)
    bad = err > lim
    if bad.any():
        i = np.argmax(err - lim)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst at flat "
                             f"{i}: got {g.flat[i]!r} ref {r.flat[i]!r}")


def sample_indices(shape, n_random, seed):
    """Random flat indices into y plus every output of the spatial border of
    the first and last image (padding-affected positions) for a few channels."""
    rng = np.random.default_rng(seed)
    total = int(np.prod(shape))
    idx = [rng.integers(0, total, size=n_random)]
    sp = shape[1:-2]  # spatial dims (Ho, Wo) or (Do, Ho, Wo)
    ch = shape[-2] * shape[-1]
    chans = np.unique(np.concatenate([[0, ch - 1], rng.integers(0, ch, size=6)]))
    grids = np.meshgrid(*[np.arange(s) for s in sp], indexing="ij")
    border = np.zeros(sp, dtype=bool)
    for ax, gx in enumerate(grids):
        border |= (gx == 0) | (gx == sp[ax] - 1)
    pos = np.flatnonzero(border.reshape(-1))
    nsp = int(np.prod(sp))
    for n in {0, shape[0] - 1}:
        for c in chans:
            idx.append((n * nsp + pos) * ch + c)
    return np.unique(np.concatenate(idx).astype(np.int64))
