"""Algorithmic work and traffic of one grouped-convolution forward pass.

FLOP counts only the multiply-adds of real weights, per group:
    FLOP = 2 * N * Do*Ho*Wo * K * Cg * taps
(each of the N*Do*Ho*Wo*K outputs takes Cg*taps MACs; the TileOps review's
roofline discussion asks for per-group C_in_g rather than the full C, and its
3D case prints 802,816 outputs x 54 MACs x 2 = ~86.7 MFLOP).  Zeros that a
kernel multiplies because it merges groups into block-diagonal tiles are not
credited.

Bytes count each tensor moved once:  x + y + w (+ bias), in the storage dtype,
where x counts only the input positions some filter tap reads.  With stride 2
and dilation 2 (pad 2) only every other row and column of the input is ever
read, so a quarter of x; every other benchmarked problem reads all of it.

The backward passes move the same three tensors: backward weight reads
x (the touched positions) and dy (y's size) and writes dw (w's size);
backward data reads dy and w and writes every position of dx, zeros
included, so there x counts in full (``op="bwd_data"``).
"""
from __future__ import annotations

ES = {"f32": 4, "f16": 2, "bf16": 2}


def outputs(wl, out_shape) -> int:
    Do, Ho, Wo = out_shape
    return wl.N * Do * Ho * Wo * wl.K


def flops(wl, out_shape) -> int:
    return 2 * outputs(wl, out_shape) * wl.Cg * wl.taps


def touched(i_ext: int, o_ext: int, k: int, s: int, p: int, d: int) -> int:
    """Input positions along one dimension that some tap of some output
    reads: o*s - p + t*d inside [0, i_ext) for o < o_ext, t < k."""
    return len({o * s - p + t * d for o in range(o_ext) for t in range(k)} & set(range(i_ext)))


def tensor_bytes(wl, out_shape, op: str = "fwd") -> dict:
    es = ES[wl.dtype]
    read = 1
    for i in range(3):
        read *= wl.inp[i] if op == "bwd_data" else \
            touched(wl.inp[i], out_shape[i], wl.ker[i], wl.stride[i], wl.pad[i], wl.dil[i])
    x = wl.N * read * wl.C * es
    y = outputs(wl, out_shape) * es
    w = wl.K * wl.taps * wl.Cg * es
    b = wl.K * es if wl.bias else 0
    return {"x": x, "y": y, "w": w, "bias": b}


def algorithmic_bytes(wl, out_shape, op: str = "fwd") -> int:
    return sum(tensor_bytes(wl, out_shape, op).values())


def fused_block_bytes(wl, out_shape, K: int) -> dict:
    """Tensors the fused depthwise + 1x1 projection block moves once: x (the
    touched positions), the depthwise weights and bias, the projection's
    weights [K, C] and bias [K], and y [N, Ho, Wo, K].  h, the depthwise
    output, stays on chip; ``h_saved`` is the HBM traffic of writing it and
    reading it back that a separate projection would add."""
    es = ES[wl.dtype]
    t = tensor_bytes(wl, out_shape)
    pix = wl.N * out_shape[0] * out_shape[1] * out_shape[2]
    return {"x": t["x"], "w_dw": t["w"], "b_dw": t["bias"], "w_pw": K * wl.C * es, "b_pw": K * es,
            "y": pix * K * es, "h_saved": 2 * pix * wl.C * es}


def fused_block_flops(wl, out_shape, K: int) -> int:
    """Depthwise multiply-adds (9 per output channel) plus the projection's
    (C per output of K)."""
    pix = wl.N * out_shape[0] * out_shape[1] * out_shape[2]
    return 2 * pix * wl.C * wl.taps + 2 * pix * wl.C * K
