"""Pins that tie the CPU oracle to facts outside itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with:

* an independent NumPy formulation (explicit zero-padded tensor, strided
  window gather, einsum) on tiny problems -- brute force;
* PyTorch's CPU float64 ``conv2d`` / ``conv3d`` with ``groups`` (a library
  routine the grouped case reduces to after a layout permutation);
* the split into G independent dense convolutions whose outputs are
  concatenated (rocm-libraries PR #10064, Technical Details: grouped channel
  decode c = g*Cg + c_in_group and output fold k_out = g*Kg + n);
* closed forms: a centred delta kernel is the identity, an off-centre delta is
  a shift (this fixes cross-correlation, i.e. no kernel flip), and all-ones
  inputs give Cg times the number of in-bounds taps;
* the output extents torch reports.

``ALL_PINS`` is used both on the real oracle and on deliberately broken
copies of it (tests/test_oracle_mutations.py).
"""
from __future__ import annotations

import itertools

import numpy as np
import torch

from depthwise_convolution_forward_gb300.inputs import Workload


def wl(ndim, N, G, Cg, Kg, inp, ker, st, pd, dl, bias=True, dtype="f32"):
    if ndim == 2:
        inp, ker, st, pd, dl = (1,) + tuple(inp), (1,) + tuple(ker), (1,) + tuple(st), \
            (0,) + tuple(pd), (1,) + tuple(dl)
    return Workload("pin", 0, 0, ndim, N, G, Cg, Kg, tuple(inp), tuple(ker), tuple(st),
                    tuple(pd), tuple(dl), dtype, bias)


def rand_inputs(p: Workload, seed: int, integer: bool = False):
    rng = np.random.default_rng(seed)
    if integer:
        x = rng.integers(-2, 3, size=p.x_shape()).astype(np.float64)
        w = rng.integers(-2, 3, size=p.w_shape()).astype(np.float64)
        b = rng.integers(-3, 4, size=(p.K,)).astype(np.float64) if p.bias else None
    else:
        x = rng.uniform(-1, 1, size=p.x_shape())
        w = rng.normal(0, 1, size=p.w_shape())
        b = rng.uniform(-1, 1, size=(p.K,)) if p.bias else None
    return x, w, b


# ---------------------------------------------------------------------------
# Independent formulation: zero-pad, gather windows, einsum.
# ---------------------------------------------------------------------------
def _count_positions(i, k, s, p, d):
    """Number of window placements: step o while the last tap stays inside."""
    o = 0
    while o * s + d * (k - 1) <= i + 2 * p - 1:
        o += 1
    return o


def brute_numpy(p: Workload, x, w, b):
    x5 = np.asarray(x, dtype=np.float64).reshape(p.N, p.inp[0], p.inp[1], p.inp[2], p.G, p.Cg)
    w5 = np.asarray(w, dtype=np.float64).reshape(p.G, p.Kg, p.ker[0], p.ker[1], p.ker[2], p.Cg)
    pads = [(0, 0)] + [(p.pad[i], p.pad[i]) for i in range(3)] + [(0, 0), (0, 0)]
    xp = np.pad(x5, pads)
    outs = [_count_positions(p.inp[i], p.ker[i], p.stride[i], p.pad[i], p.dil[i]) for i in range(3)]
    slabs = []
    for z, yy, xx in itertools.product(range(p.ker[0]), range(p.ker[1]), range(p.ker[2])):
        starts = (z * p.dil[0], yy * p.dil[1], xx * p.dil[2])
        sl = xp[:,
                starts[0]: starts[0] + (outs[0] - 1) * p.stride[0] + 1: p.stride[0],
                starts[1]: starts[1] + (outs[1] - 1) * p.stride[1] + 1: p.stride[1],
                starts[2]: starts[2] + (outs[2] - 1) * p.stride[2] + 1: p.stride[2]]
        slabs.append(sl)
    win = np.stack(slabs, axis=5)  # [N, Do, Ho, Wo, G, T, Cg]
    wt = w5.reshape(p.G, p.Kg, -1, p.Cg)  # [G, Kg, T, Cg]
    y = np.einsum("nabcgtq,gktq->nabcgk", win, wt)
    if b is not None:
        y = y + np.asarray(b, dtype=np.float64).reshape(p.G, p.Kg)
    if p.ndim == 2:
        y = y[:, 0]
    return y


def torch_reference(p: Workload, x, w, b):
    """torch.nn.functional.conv{2,3}d(groups=G) on CPU float64, layouts permuted."""
    xt = torch.as_tensor(np.asarray(x, dtype=np.float64))
    wt = torch.as_tensor(np.asarray(w, dtype=np.float64))
    bt = None if b is None else torch.as_tensor(np.asarray(b, dtype=np.float64))
    if p.ndim == 2:
        xc = xt.reshape(p.N, p.inp[1], p.inp[2], p.C).permute(0, 3, 1, 2)
        wc = wt.reshape(p.K, p.ker[1], p.ker[2], p.Cg).permute(0, 3, 1, 2)
        y = torch.nn.functional.conv2d(xc, wc, bt, stride=p.stride[1:], padding=p.pad[1:],
                                       dilation=p.dil[1:], groups=p.G)
        return y.permute(0, 2, 3, 1).reshape(p.N, y.shape[2], y.shape[3], p.G, p.Kg).numpy()
    xc = xt.reshape(p.N, *p.inp, p.C).permute(0, 4, 1, 2, 3)
    wc = wt.reshape(p.K, *p.ker, p.Cg).permute(0, 4, 1, 2, 3)
    y = torch.nn.functional.conv3d(xc, wc, bt, stride=p.stride, padding=p.pad,
                                   dilation=p.dil, groups=p.G)
    return y.permute(0, 2, 3, 4, 1).reshape(p.N, *y.shape[2:], p.G, p.Kg).numpy()


def _close(a, b, tol=1e-11):
    a = np.asarray(a)
    b = np.asarray(b)
    assert a.shape == b.shape, (a.shape, b.shape)
    err = np.max(np.abs(a - b)) if a.size else 0.0
    assert err <= tol * (1.0 + np.max(np.abs(b)) if b.size else 1.0), err


# ---------------------------------------------------------------------------
# Pins
# ---------------------------------------------------------------------------
def tiny_problems():
    """Small 2D and 3D problems over stride {1,2} x pad {0,1,2} x dilation {1,2}."""
    out = []
    for s, pd, d in itertools.product((1, 2), (0, 1, 2), (1, 2)):
        out.append(wl(2, 2, 3, 2, 3, (6, 5), (3, 2), (s, s), (pd, pd), (d, d)))
    out.append(wl(2, 1, 2, 3, 1, (5, 7), (1, 3), (2, 1), (0, 1), (1, 2), bias=False))
    out.append(wl(3, 2, 2, 2, 3, (4, 5, 5), (3, 2, 3), (1, 2, 1), (1, 0, 2), (1, 1, 2)))
    out.append(wl(3, 1, 4, 1, 2, (3, 6, 4), (2, 3, 1), (2, 1, 2), (1, 1, 0), (2, 1, 1)))
    return out


def pin_brute_force(orc):
    for i, p in enumerate(tiny_problems()):
        x, w, b = rand_inputs(p, 100 + i)
        _close(orc.forward(p, x, w, b), brute_numpy(p, x, w, b))


def pin_brute_force_integer_exact(orc):
    # small integers: every partial sum is exact in float64, so equality is exact
    for i, p in enumerate(tiny_problems()[::3]):
        x, w, b = rand_inputs(p, 300 + i, integer=True)
        assert np.array_equal(orc.forward(p, x, w, b), brute_numpy(p, x, w, b))


def pin_torch_groups(orc):
    probs = [
        wl(2, 2, 4, 3, 2, (9, 7), (3, 3), (1, 1), (1, 1), (1, 1)),
        wl(2, 1, 6, 1, 1, (8, 8), (3, 3), (2, 2), (1, 1), (1, 1)),  # depthwise
        wl(2, 1, 3, 2, 5, (10, 9), (3, 3), (2, 1), (2, 2), (2, 2)),
        wl(3, 1, 2, 3, 2, (5, 6, 6), (3, 3, 3), (1, 2, 1), (1, 1, 1), (1, 1, 2)),
        wl(2, 2, 1, 5, 4, (7, 6), (3, 2), (1, 1), (1, 0), (1, 1)),  # groups == 1
    ]
    for i, p in enumerate(probs):
        x, w, b = rand_inputs(p, 200 + i)
        _close(orc.forward(p, x, w, b), torch_reference(p, x, w, b))


def pin_groups_split(orc):
    """Grouped output == G dense convolutions on channel slices, concatenated."""
    for p in (wl(2, 2, 3, 2, 4, (6, 6), (3, 3), (1, 1), (1, 1), (1, 1)),
              wl(3, 1, 4, 3, 2, (4, 5, 5), (3, 1, 3), (1, 2, 1), (1, 0, 1), (1, 1, 1))):
        x, w, b = rand_inputs(p, 7)
        full = orc.forward(p, x, w, b)
        x6 = x.reshape(p.N, *p.inp, p.G, p.Cg)
        w6 = w.reshape(p.G, p.Kg, *p.ker, p.Cg)
        b2 = b.reshape(p.G, p.Kg)
        one = p.with_(G=1)
        parts = []
        for g in range(p.G):
            yg = orc.forward(one, x6[..., g:g + 1, :].copy(), w6[g:g + 1].copy(), b2[g].copy())
            parts.append(yg)
        cat = np.concatenate(parts, axis=-2)  # the G axis sits before Kg
        _close(full, cat)


def pin_delta_identity(orc):
    """Depthwise, centred delta, pad = d*(k-1)/2, stride 1: y == x exactly."""
    for ndim, k, d in ((2, 3, 1), (2, 5, 2), (3, 3, 1), (2, 1, 1)):
        kk = (k, k, k) if ndim == 3 else (k, k)
        pp = tuple(d * (k - 1) // 2 for _ in kk)
        dd = (d,) * len(kk)
        inp = (4, 6, 5) if ndim == 3 else (7, 6)
        p = wl(ndim, 2, 5, 1, 1, inp, kk, (1,) * len(kk), pp, dd, bias=False)
        x, _, _ = rand_inputs(p, 11)
        w = np.zeros(p.w_shape())
        c = (k - 1) // 2
        if ndim == 3:
            w[:, :, c, c, c, :] = 1.0
        else:
            w[:, :, c, c, :] = 1.0
        y = orc.forward(p, x, w, None)
        assert np.array_equal(y, x.reshape(y.shape)), "centred delta is not the identity"


def pin_delta_shift(orc):
    """Delta at tap (0,0), pad 1: y[h, w] = x[h-1, w-1], zero on the border.

    Cross-correlation (no flip) puts the copy at offset -1; a convolution
    (flipped kernel) would put it at +1.
    """
    p = wl(2, 1, 3, 1, 1, (6, 7), (3, 3), (1, 1), (1, 1), (1, 1), bias=False)
    x, _, _ = rand_inputs(p, 12)
    w = np.zeros(p.w_shape())
    w[:, :, 0, 0, :] = 1.0
    y = orc.forward(p, x, w, None)
    x4 = x.reshape(1, 6, 7, 3)
    want = np.zeros_like(x4)
    want[:, 1:, 1:, :] = x4[:, :-1, :-1, :]
    assert np.array_equal(y.reshape(want.shape), want)
    # 3D: delta at (0, 0, 0) with pad 1 shifts along all three axes
    p3 = wl(3, 1, 2, 1, 1, (4, 5, 6), (3, 3, 3), (1, 1, 1), (1, 1, 1), (1, 1, 1), bias=False)
    x3, _, _ = rand_inputs(p3, 13)
    w3 = np.zeros(p3.w_shape())
    w3[:, :, 0, 0, 0, :] = 1.0
    y3 = orc.forward(p3, x3, w3, None).reshape(1, 4, 5, 6, 2)
    x3r = x3.reshape(1, 4, 5, 6, 2)
    want3 = np.zeros_like(x3r)
    want3[:, 1:, 1:, 1:, :] = x3r[:, :-1, :-1, :-1, :]
    assert np.array_equal(y3, want3)


def _inbounds_taps_1d(o, i, k, s, p, d):
    return sum(1 for t in range(k) if 0 <= o * s - p + t * d < i)


def pin_all_ones(orc):
    """x = w = 1: y = Cg * (in-bounds taps), a product of per-axis counts."""
    for p in (wl(2, 2, 3, 4, 2, (7, 6), (3, 3), (2, 1), (1, 2), (1, 2), bias=False),
              wl(3, 1, 2, 3, 1, (5, 4, 6), (3, 2, 3), (1, 2, 2), (2, 1, 1), (2, 1, 1), bias=False)):
        x = np.ones(p.x_shape())
        w = np.ones(p.w_shape())
        y = orc.forward(p, x, w, None)
        y6 = y.reshape(p.N, *orc.out_shape(p), p.G, p.Kg)
        Do, Ho, Wo = orc.out_shape(p)
        for od, oh, ow in itertools.product(range(Do), range(Ho), range(Wo)):
            cnt = 1
            for ax, o in enumerate((od, oh, ow)):
                cnt *= _inbounds_taps_1d(o, p.inp[ax], p.ker[ax], p.stride[ax], p.pad[ax], p.dil[ax])
            assert np.all(y6[:, od, oh, ow] == p.Cg * cnt)


def pin_bias_only(orc):
    """Zero weights: every output equals its bias, bias[g*Kg + k]."""
    p = wl(2, 2, 3, 2, 4, (5, 5), (3, 3), (1, 1), (1, 1), (1, 1))
    x, _, b = rand_inputs(p, 21)
    w = np.zeros(p.w_shape())
    y = orc.forward(p, x, w, b)
    assert np.array_equal(y, np.broadcast_to(b.reshape(p.G, p.Kg), y.shape))


def pin_out_extent_vs_torch(orc):
    for i, k, s, pd, d in itertools.product((1, 2, 5, 8, 13), (1, 2, 3, 5), (1, 2, 3),
                                            (0, 1, 2), (1, 2, 3)):
        if i + 2 * pd < d * (k - 1) + 1:
            assert orc.out_extent(i, k, s, pd, d) <= 0
            continue
        t = torch.nn.functional.conv1d(torch.zeros(1, 1, i), torch.zeros(1, 1, k), stride=s,
                                       padding=pd, dilation=d)
        assert orc.out_extent(i, k, s, pd, d) == t.shape[-1], (i, k, s, pd, d)


def pin_points_match_forward(orc):
    p = wl(3, 2, 3, 2, 3, (4, 5, 6), (3, 3, 2), (1, 2, 1), (1, 1, 0), (1, 1, 2))
    x, w, b = rand_inputs(p, 31)
    full = orc.forward(p, x, w, b).reshape(-1)
    idx = np.random.default_rng(0).integers(0, full.size, size=50)
    assert np.array_equal(orc.points(p, x, w, b, idx), full[idx])
    _close(full[idx], brute_numpy(p, x, w, b).reshape(-1)[idx])


ALL_PINS = [
    pin_brute_force,
    pin_brute_force_integer_exact,
    pin_torch_groups,
    pin_groups_split,
    pin_delta_identity,
    pin_delta_shift,
    pin_all_ones,
    pin_bias_only,
    pin_out_extent_vs_torch,
    pin_points_match_forward,
]


# ---------------------------------------------------------------------------
# Backward data: pins that do not use the oracle's own backward code
# ---------------------------------------------------------------------------
def torch_bwd_data(p: Workload, dy, w):
    """torch.nn.grad.conv{2,3}d_input(groups=G) on CPU float64, layouts permuted."""
    dyt = torch.as_tensor(np.asarray(dy, dtype=np.float64))
    wt = torch.as_tensor(np.asarray(w, dtype=np.float64))
    if p.ndim == 2:
        Ho, Wo = dyt.shape[1], dyt.shape[2]
        dyc = dyt.reshape(p.N, Ho, Wo, p.K).permute(0, 3, 1, 2)
        wc = wt.reshape(p.K, p.ker[1], p.ker[2], p.Cg).permute(0, 3, 1, 2)
        dx = torch.nn.grad.conv2d_input((p.N, p.C, p.inp[1], p.inp[2]), wc, dyc, stride=p.stride[1:],
                                        padding=p.pad[1:], dilation=p.dil[1:], groups=p.G)
        return dx.permute(0, 2, 3, 1).reshape(p.N, p.inp[1], p.inp[2], p.G, p.Cg).numpy()
    dyc = dyt.reshape(p.N, *dyt.shape[1:4], p.K).permute(0, 4, 1, 2, 3)
    wc = wt.reshape(p.K, *p.ker, p.Cg).permute(0, 4, 1, 2, 3)
    dx = torch.nn.grad.conv3d_input((p.N, p.C, *p.inp), wc, dyc, stride=p.stride, padding=p.pad,
                                    dilation=p.dil, groups=p.G)
    return dx.permute(0, 2, 3, 4, 1).reshape(p.N, *p.inp, p.G, p.Cg).numpy()


def bwd_problems():
    return [
        wl(2, 2, 4, 3, 2, (9, 7), (3, 3), (1, 1), (1, 1), (1, 1)),
        wl(2, 1, 6, 1, 1, (8, 9), (3, 3), (2, 2), (1, 1), (1, 1)),  # depthwise, stride 2
        wl(2, 1, 3, 2, 5, (10, 9), (3, 3), (2, 1), (2, 2), (2, 2)),
        wl(3, 1, 2, 3, 2, (5, 6, 6), (3, 3, 3), (1, 2, 1), (1, 1, 1), (1, 1, 2)),
        wl(2, 2, 1, 5, 4, (7, 6), (3, 2), (1, 1), (1, 0), (1, 1)),  # groups == 1
        wl(2, 1, 2, 2, 3, (6, 6), (1, 1), (1, 1), (1, 1), (1, 1)),  # pad beyond the filter
    ]


def _rand_dy(p: Workload, orc, seed):
    out = orc.out_shape(p)
    shape = (p.N, out[1], out[2], p.G, p.Kg) if p.ndim == 2 else (p.N, *out, p.G, p.Kg)
    return np.random.default_rng(seed).uniform(-1, 1, size=shape)


def pin_bwd_adjoint(orc):
    """Backward data is the adjoint of the (pinned) forward map in x:
    <forward(x), dy> == <x, bwd_data(dy)> for any x, dy (no bias)."""
    for i, p in enumerate(bwd_problems()):
        x, w, _ = rand_inputs(p, 300 + i)
        dy = _rand_dy(p, orc, 400 + i)
        lhs = float(np.sum(orc.forward(p, x, w, None) * dy))
        rhs = float(np.sum(x.reshape(orc.bwd_data(p, dy, w).shape) * orc.bwd_data(p, dy, w)))
        assert abs(lhs - rhs) <= 1e-10 * (1.0 + abs(lhs)), (i, lhs, rhs)


def pin_bwd_torch(orc):
    for i, p in enumerate(bwd_problems()):
        _, w, _ = rand_inputs(p, 500 + i)
        dy = _rand_dy(p, orc, 600 + i)
        _close(orc.bwd_data(p, dy, w), torch_bwd_data(p, dy, w))


BWD_PINS = [pin_bwd_adjoint, pin_bwd_torch]


# ---------------------------------------------------------------------------
# Backward weight: pins that do not use the oracle's own backward code
# ---------------------------------------------------------------------------
def torch_bwd_weight(p: Workload, x, dy):
    """torch.nn.grad.conv{2,3}d_weight(groups=G) on CPU float64, layouts permuted."""
    xt = torch.as_tensor(np.asarray(x, dtype=np.float64))
    dyt = torch.as_tensor(np.asarray(dy, dtype=np.float64))
    if p.ndim == 2:
        xc = xt.reshape(p.N, p.inp[1], p.inp[2], p.C).permute(0, 3, 1, 2)
        dyc = dyt.reshape(p.N, dyt.shape[1], dyt.shape[2], p.K).permute(0, 3, 1, 2)
        dw = torch.nn.grad.conv2d_weight(xc, (p.K, p.Cg, p.ker[1], p.ker[2]), dyc, stride=p.stride[1:],
                                         padding=p.pad[1:], dilation=p.dil[1:], groups=p.G)
        return dw.permute(0, 2, 3, 1).reshape(p.G, p.Kg, p.ker[1], p.ker[2], p.Cg).numpy()
    xc = xt.reshape(p.N, *p.inp, p.C).permute(0, 4, 1, 2, 3)
    dyc = dyt.reshape(p.N, *dyt.shape[1:4], p.K).permute(0, 4, 1, 2, 3)
    dw = torch.nn.grad.conv3d_weight(xc, (p.K, p.Cg, *p.ker), dyc, stride=p.stride, padding=p.pad,
                                     dilation=p.dil, groups=p.G)
    return dw.permute(0, 2, 3, 4, 1).reshape(p.G, p.Kg, *p.ker, p.Cg).numpy()


def pin_bwd_weight_adjoint(orc):
    """The forward pass is linear in w: <forward(x, w), dy> == <w, bwd_weight(x, dy)>."""
    for i, p in enumerate(bwd_problems()):
        x, w, _ = rand_inputs(p, 700 + i)
        dy = _rand_dy(p, orc, 800 + i)
        lhs = float(np.sum(orc.forward(p, x, w, None) * dy))
        dw = orc.bwd_weight(p, x, dy)
        rhs = float(np.sum(np.asarray(w).reshape(dw.shape) * dw))
        assert abs(lhs - rhs) <= 1e-10 * (1.0 + abs(lhs)), (i, lhs, rhs)


def pin_bwd_weight_torch(orc):
    for i, p in enumerate(bwd_problems()):
        x, _, _ = rand_inputs(p, 900 + i)
        dy = _rand_dy(p, orc, 1000 + i)
        _close(orc.bwd_weight(p, x, dy), torch_bwd_weight(p, x, dy))


BWD_WEIGHT_PINS = [pin_bwd_weight_adjoint, pin_bwd_weight_torch]
