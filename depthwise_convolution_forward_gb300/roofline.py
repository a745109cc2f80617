"""Algorithmic work and traffic of one grouped-convolution forward pass.

FLOP counts only the multiply-adds of real weights, per group:
    FLOP = 2 * N * Do*Ho*Wo * K * Cg * taps
(each of the N*Do*Ho*Wo*K outputs takes Cg*taps MACs; the TileOps review's
roofline discussion asks for per-group C_in_g rather than the full C, and its
3D case prints 802,816 outputs x 54 MACs x 2 = ~86.7 MFLOP).  Zeros that a
kernel multiplies because it merges groups into block-diagonal tiles are not
credited.

Bytes count each tensor moved once:  x + y + w (+ bias), in the storage dtype.
For every benchmarked problem the filter windows cover the whole input, so
all of x is read at least once.
"""
from __future__ import annotations

ES = {"f32": 4, "f16": 2, "bf16": 2}


def outputs(wl, out_shape) -> int:
    Do, Ho, Wo = out_shape
    return wl.N * Do * Ho * Wo * wl.K


def flops(wl, out_shape) -> int:
    return 2 * outputs(wl, out_shape) * wl.Cg * wl.taps


def tensor_bytes(wl, out_shape) -> dict:
    es = ES[wl.dtype]
    D, H, W = wl.inp
    x = wl.N * D * H * W * wl.C * es
    y = outputs(wl, out_shape) * es
    w = wl.K * wl.taps * wl.Cg * es
    b = wl.K * es if wl.bias else 0
    return {"x": x, "y": y, "w": w, "bias": b}


def algorithmic_bytes(wl, out_shape) -> int:
    return sum(tensor_bytes(wl, out_shape).values())
