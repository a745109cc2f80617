"""CPU oracle for grouped convolution forward, backward data and backward
weight -- TEST INFRASTRUCTURE ONLY.

The oracle (``oracle.c``) is a plain fp64 direct-loop grouped convolution
written from the definition (see the header of ``oracle.c`` for the formula,
the passages it follows and the readings it takes).  Only ``tests/``, the
package smoke check and the benchmark's CPU-baseline leg may import this
module.  It shares no code with the CUDA library and must never be used as a
fallback for it.

``build()`` compiles ``oracle.c`` with gcc (OpenMP when available) into
``oracle/liboracle.so``; ``load(path)`` can load an alternative build, which
the mutation tests use to show that the pins catch planted mistakes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

_i32p = ctypes.POINTER(ctypes.c_int32)
_dp = ctypes.POINTER(ctypes.c_double)


def compile_source(src: str, out: str, openmp: bool = True) -> str:
    """Compile one C source file into a shared library with gcc."""
    cmd = ["gcc", "-O2", "-std=c99", "-shared", "-fPIC", src, "-o", out]
    if openmp:
        cmd.insert(1, "-fopenmp")
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return out


def build(force: bool = False) -> str:
    """Build ``liboracle.so`` next to the source if it is missing or stale."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SOURCE):
        tmp = LIB + f".tmp{os.getpid()}"
        try:
            compile_source(SOURCE, tmp, openmp=True)
        except subprocess.CalledProcessError:
            compile_source(SOURCE, tmp, openmp=False)
        os.replace(tmp, LIB)
    return LIB


class Oracle:
    """ctypes view of one oracle build."""

    def __init__(self, path: str):
        self.path = path
        lib = ctypes.CDLL(path)
        lib.oracle_out_extent.restype = ctypes.c_long
        lib.oracle_out_extent.argtypes = [ctypes.c_long] * 5
        lib.oracle_grouped_conv_fwd.restype = ctypes.c_int
        lib.oracle_grouped_conv_fwd.argtypes = [_dp, _dp, _dp, _dp] + [ctypes.c_long] * 4 + [_i32p] * 5
        lib.oracle_grouped_conv_fwd_points.restype = ctypes.c_int
        lib.oracle_grouped_conv_fwd_points.argtypes = (
            [_dp, _dp, _dp] + [ctypes.c_long] * 4 + [_i32p] * 5
            + [ctypes.POINTER(ctypes.c_int64), ctypes.c_long, _dp])
        lib.oracle_grouped_conv_bwd_weight.restype = ctypes.c_int
        lib.oracle_grouped_conv_bwd_weight.argtypes = [_dp, _dp, _dp] + [ctypes.c_long] * 4 + [_i32p] * 5
        lib.oracle_grouped_conv_bwd_data.restype = ctypes.c_int
        lib.oracle_grouped_conv_bwd_data.argtypes = [_dp, _dp, _dp] + [ctypes.c_long] * 4 + [_i32p] * 5
        self.lib = lib

    # -- helpers ---------------------------------------------------------
    @staticmethod
    def _f64(a):
        if a is None:
            return None
        if hasattr(a, "detach"):  # torch tensor: exact widening to float64
            a = a.detach().to("cpu").double().contiguous().numpy()
        return np.ascontiguousarray(a, dtype=np.float64)

    @staticmethod
    def _v3(v):
        return (ctypes.c_int32 * 3)(*[int(t) for t in v])

    def out_extent(self, i: int, k: int, s: int, p: int, d: int) -> int:
        return int(self.lib.oracle_out_extent(i, k, s, p, d))

    def out_shape(self, prob) -> tuple:
        return tuple(self.out_extent(prob.inp[i], prob.ker[i], prob.stride[i], prob.pad[i],
                                     prob.dil[i]) for i in range(3))

    def _args(self, prob):
        return (prob.N, prob.G, prob.Cg, prob.Kg, self._v3(prob.inp), self._v3(prob.ker),
                self._v3(prob.stride), self._v3(prob.pad), self._v3(prob.dil))

    def forward(self, prob, x, w, bias=None) -> np.ndarray:
        """Full output as float64 [N, (Do), Ho, Wo, G, Kg] (Do omitted for 2D)."""
        xd, wd, bd = self._f64(x), self._f64(w), self._f64(bias)
        Do, Ho, Wo = self.out_shape(prob)
        shape = (prob.N, Do, Ho, Wo, prob.G, prob.Kg)
        y = np.empty(shape, dtype=np.float64)
        rc = self.lib.oracle_grouped_conv_fwd(
            xd.ctypes.data_as(_dp), wd.ctypes.data_as(_dp),
            bd.ctypes.data_as(_dp) if bd is not None else None,
            y.ctypes.data_as(_dp), *self._args(prob))
        if rc != 0:
            raise ValueError("oracle rejected the problem")
        if prob.ndim == 2:
            y = y.reshape(prob.N, Ho, Wo, prob.G, prob.Kg)
        return y

    def points(self, prob, x, w, bias, idx) -> np.ndarray:
        """Outputs at flat indices ``idx`` into the [N,Do,Ho,Wo,G,Kg] layout."""
        xd, wd, bd = self._f64(x), self._f64(w), self._f64(bias)
        ii = np.ascontiguousarray(idx, dtype=np.int64)
        out = np.empty(ii.shape[0], dtype=np.float64)
        rc = self.lib.oracle_grouped_conv_fwd_points(
            xd.ctypes.data_as(_dp), wd.ctypes.data_as(_dp),
            bd.ctypes.data_as(_dp) if bd is not None else None, *self._args(prob),
            ii.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), ii.shape[0],
            out.ctypes.data_as(_dp))
        if rc != 0:
            raise ValueError("oracle rejected the problem or an index")
        return out


    def bwd_data(self, prob, dy, w) -> np.ndarray:
        """Backward data: dx as float64 in x's layout [N, (D), H, W, G, Cg] (D
        omitted for 2D), the adjoint of ``forward`` in x applied to ``dy``."""
        dyd, wd = self._f64(dy), self._f64(w)
        D, H, W = prob.inp
        dx = np.empty((prob.N, D, H, W, prob.G, prob.Cg), dtype=np.float64)
        rc = self.lib.oracle_grouped_conv_bwd_data(
            dyd.ctypes.data_as(_dp), wd.ctypes.data_as(_dp), dx.ctypes.data_as(_dp), *self._args(prob))
        if rc != 0:
            raise ValueError("oracle rejected the problem")
        if prob.ndim == 2:
            dx = dx.reshape(prob.N, H, W, prob.G, prob.Cg)
        return dx


    def bwd_weight(self, prob, x, dy) -> np.ndarray:
        """Backward weight: dw as float64 in w's layout [G, Kg, (Z), Y, X, Cg]
        (Z omitted for 2D), the gradient of <forward(x, w), dy> with respect to w."""
        xd, dyd = self._f64(x), self._f64(dy)
        Z, Y, X = prob.ker
        dw = np.empty((prob.G, prob.Kg, Z, Y, X, prob.Cg), dtype=np.float64)
        rc = self.lib.oracle_grouped_conv_bwd_weight(
            xd.ctypes.data_as(_dp), dyd.ctypes.data_as(_dp), dw.ctypes.data_as(_dp), *self._args(prob))
        if rc != 0:
            raise ValueError("oracle rejected the problem")
        if prob.ndim == 2:
            dw = dw.reshape(prob.G, prob.Kg, Y, X, prob.Cg)
        return dw


    def dw_pw_block(self, prob, x, w_dw, b_dw, act, w_pw, b_pw, dtype) -> np.ndarray:
        """Depthwise convolution, activation, then a 1x1 projection: the tail
        of a MobileNetV2-style block (the pages' depthwise benchmark layer and
        its pointwise neighbour).  ``prob`` is the depthwise problem (G = C,
        Cg = Kg = 1); ``w_pw`` is [K, C] (the 1x1 weight in GKYXC with G = 1),
        ``b_pw`` [K] or None; ``act`` 0 none, 1 ReLU, 2 ReLU6 (min(max(v, 0),
        6)).  The intermediate h = act(dw(x) + b_dw) is rounded once to the
        storage ``dtype`` (a torch dtype), as a separate depthwise layer would
        store it, then y = h @ w_pw^T + b_pw in float64 [N, Ho, Wo, K]."""
        import torch  # the rounding step; the oracle's arithmetic stays float64

        h = self.forward(prob, x, w_dw, b_dw)  # [N, Ho, Wo, C, 1]
        if act == 1:
            h = np.maximum(h, 0.0)
        elif act == 2:
            h = np.minimum(np.maximum(h, 0.0), 6.0)
        elif act != 0:
            raise ValueError("act must be 0, 1 or 2")
        h = torch.from_numpy(np.ascontiguousarray(h)).to(dtype).double().numpy()
        N, Ho, Wo = h.shape[0], h.shape[1], h.shape[2]
        C = prob.G
        wp = self._f64(w_pw).reshape(-1, C)
        K = wp.shape[0]

        class _Pw:  # the projection as a grouped convolution with G = 1, 1x1
            ndim = 2
            inp = (1, Ho, Wo)
            ker = stride = dil = (1, 1, 1)
            pad = (0, 0, 0)

        pw = _Pw()
        pw.N, pw.G, pw.Cg, pw.Kg = N, 1, C, K
        y = self.forward(pw, h.reshape(N, Ho, Wo, C), wp, b_pw)
        return y.reshape(N, Ho, Wo, K)


_default: Optional[Oracle] = None


def get() -> Oracle:
    """The oracle built from ``oracle.c`` (built on first use)."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def load(path: str) -> Oracle:
    return Oracle(path)
