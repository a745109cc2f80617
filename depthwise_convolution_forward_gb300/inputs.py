"""Seeded synthetic workloads for grouped convolution forward.

This module holds problem descriptions and random-number recipes only.  It
contains none of the convolution's arithmetic (no output-size rule, no
accumulation), so both the CUDA path's tests and the CPU oracle's tests can
draw identical inputs from it without sharing any of the method.

Workloads follow the benchmark cases named on the pages:

* "TileOps PR #1568 review" (Code Review section): MobileNetV2 depthwise and
  ResNeXt grouped benchmark cases, and the 3D case N=1, C 64->128,
  DxHxW 8x28x28, 3x3x3, groups 32, with a batch>=8 data point requested.
* CK "Grouped Convolution -- Python Examples" (Config-options harness):
  the small smoke problem N=1, G=2, C=K=64, Hi=Wi=8, 3x3.

The pages name these cases but do not publish their tensors, so every tensor
here is drawn from a seeded CPU ``torch.Generator`` with the stated
distributions:  x ~ U(-1, 1), w ~ N(0, 1/fan_in) with fan_in = Cg * taps
(variance, not standard deviation), bias ~ U(-0.1, 0.1).  Values are drawn in
fp32 and rounded once to the workload's storage dtype; callers that need exact
values (the oracle) convert the stored tensor to float64.

Seeds: ``x = 1000*cfg + 10*variant + 0``, ``w = ... + 1``, ``bias = ... + 2``.
"""
from __future__ import annotations

import dataclasses
from typing import Iterator, Optional

import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Workload:
    """One grouped-convolution problem plus its input recipe.

    Layouts: x is [N, (D), H, W, G, Cg] (channels-last, groups outermost
    within a pixel), w is [G, Kg, (Z), Y, X, Cg], bias is [G*Kg].
    """

    name: str
    cfg: int  # index of the workload family (seed base)
    variant: int  # index within the family (seed offset)
    ndim: int
    N: int
    G: int
    Cg: int
    Kg: int
    inp: tuple  # (D, H, W); D == 1 for 2D
    ker: tuple  # (Z, Y, X); Z == 1 for 2D
    stride: tuple
    pad: tuple
    dil: tuple
    dtype: str
    bias: bool
    w_dist: str = "normal"  # "normal" (N(0, 1/fan_in)) or "uniform" (U(-1,1))

    @property
    def C(self) -> int:
        return self.G * self.Cg

    @property
    def K(self) -> int:
        return self.G * self.Kg

    @property
    def taps(self) -> int:
        return self.ker[0] * self.ker[1] * self.ker[2]

    def x_shape(self) -> tuple:
        D, H, W = self.inp
        if self.ndim == 2:
            return (self.N, H, W, self.G, self.Cg)
        return (self.N, D, H, W, self.G, self.Cg)

    def w_shape(self) -> tuple:
        Z, Y, X = self.ker
        if self.ndim == 2:
            return (self.G, self.Kg, Y, X, self.Cg)
        return (self.G, self.Kg, Z, Y, X, self.Cg)

    def seeds(self) -> tuple:
        base = 1000 * self.cfg + 10 * self.variant
        return base, base + 1, base + 2

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def make_inputs(wl: Workload, seed_offset: int = 0):
    """Return (x, w, bias_or_None) as CPU tensors in the workload's dtype."""
    sx, sw, sb = (s + seed_offset for s in wl.seeds())
    dt = DTYPES[wl.dtype]
    g = torch.Generator().manual_seed(sx)
    x = (torch.rand(wl.x_shape(), generator=g, dtype=torch.float32) * 2.0 - 1.0).to(dt)
    g = torch.Generator().manual_seed(sw)
    if wl.w_dist == "uniform":
        w = torch.rand(wl.w_shape(), generator=g, dtype=torch.float32) * 2.0 - 1.0
    else:
        std = (1.0 / (wl.Cg * wl.taps)) ** 0.5
        w = torch.randn(wl.w_shape(), generator=g, dtype=torch.float32) * std
    w = w.to(dt)
    b = None
    if wl.bias:
        g = torch.Generator().manual_seed(sb)
        b = ((torch.rand((wl.K,), generator=g, dtype=torch.float32) * 2.0 - 1.0) * 0.1).to(dt)
    return x, w, b


def _w2d(name, cfg, variant, N, G, Cg, Kg, H, W, k, s, p, d, dtype, bias, w_dist="normal"):
    return Workload(name, cfg, variant, 2, N, G, Cg, Kg, (1, H, W), (1, k, k),
                    (1, s, s), (0, p, p), (1, d, d), dtype, bias, w_dist)


def config_workloads(cfg: int) -> list:
    """The workload families used for parity tests and measurement.

    1: small fp32 grouped smoke problem (CK examples page, Config-options
       harness).
    2: MobileNetV2-style depthwise, fp16, stride 1 and stride 2.
    3: ResNeXt-50 32x4d grouped, bf16: (a) C=128 56x56 s1, (b) C=1024 28->14 s2.
    4: ResNeXt-style grouped 3D, fp16, N=1 and N=8 (TileOps review, batch-1
       case and the requested batch>=8 point).
    5: bf16 grouped sweep over G, dilation and stride at N=64, 28x28, C=512.
    """
    if cfg == 1:
        return [_w2d("grouped2d_f32_smoke", 1, 0, 1, 2, 32, 32, 8, 8, 3, 1, 1, 1,
                     "f32", False, "uniform")]
    if cfg == 2:
        return [
            _w2d("mbv2_dw_s1_f16", 2, 0, 32, 144, 1, 1, 56, 56, 3, 1, 1, 1, "f16", True),
            _w2d("mbv2_dw_s2_f16", 2, 1, 32, 144, 1, 1, 56, 56, 3, 2, 1, 1, "f16", True),
        ]
    if cfg == 3:
        return [
            _w2d("resnext_a_bf16", 3, 0, 32, 32, 4, 4, 56, 56, 3, 1, 1, 1, "bf16", True),
            _w2d("resnext_b_bf16", 3, 1, 32, 32, 32, 32, 28, 28, 3, 2, 1, 1, "bf16", True),
        ]
    if cfg == 4:
        out = []
        for v, n in enumerate((1, 8)):
            out.append(Workload(f"resnext3d_n{n}_f16", 4, v, 3, n, 32, 2, 4, (8, 28, 28),
                                (3, 3, 3), (1, 1, 1), (1, 1, 1), (1, 1, 1), "f16", True))
        return out
    if cfg == 5:
        out = []
        v = 0
        for G in (512, 256, 64, 32, 8):
            for d in (1, 2):
                for s in (1, 2):
                    Cg = 512 // G
                    out.append(_w2d(f"sweep_g{G}_d{d}_s{s}_bf16", 5, v, 64, G, Cg, Cg, 28, 28, 3,
                                    s, d, d, "bf16", True))
                    v += 1
        return out
    raise ValueError(f"unknown workload family {cfg}")


def all_workloads() -> Iterator[Workload]:
    for cfg in range(1, 6):
        yield from config_workloads(cfg)


def by_name(name: str) -> Workload:
    for wl in all_workloads():
        if wl.name == name:
            return wl
    raise KeyError(name)


def random_problem(rng, ndim: Optional[int] = None, dtype: Optional[str] = None,
                   max_c: int = 16, max_hw: int = 9) -> Workload:
    """A small random problem for property and parity sweeps (numpy Generator)."""
    nd = ndim if ndim is not None else int(rng.choice([2, 2, 3]))
    G = int(rng.integers(1, 5))
    Cg = int(rng.integers(1, max_c + 1))
    Kg = int(rng.integers(1, max_c + 1))
    ks = [int(rng.choice([1, 2, 3])) for _ in range(3)]
    if nd == 2:
        ks[0] = 1
    inp = [int(rng.integers(1, max_hw + 1)) for _ in range(3)]
    if nd == 2:
        inp[0] = 1
    st = [int(rng.integers(1, 3)) for _ in range(3)]
    dl = [int(rng.integers(1, 3)) for _ in range(3)]
    pd = [int(rng.integers(0, 3)) for _ in range(3)]
    if nd == 2:
        st[0], dl[0], pd[0] = 1, 1, 0
    # keep the output non-empty: grow the input until every span fits
    for i in range(3):
        span = dl[i] * (ks[i] - 1) + 1
        if inp[i] + 2 * pd[i] < span:
            inp[i] = span - 2 * pd[i]
    dt = dtype if dtype is not None else str(rng.choice(["f32", "f16", "bf16"]))
    return Workload("random", 99, int(rng.integers(0, 10**6)), nd, int(rng.integers(1, 3)), G, Cg,
                    Kg, tuple(inp), tuple(ks), tuple(st), tuple(pd), tuple(dl), dt,
                    bool(rng.integers(0, 2)), "normal")
