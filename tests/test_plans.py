"""Host-side tile planners against the invariants their kernels rely on (no GPU).

The planners of the depthwise and tensor-core kernels are compiled into two
host-only harnesses (``tests/harness/plan_*.cu``, built with nvcc) and run on
every workload family, random problems and maximum-size problems:

* shared memory within the per-block and per-SM budgets, for the planned
  CTAs per SM; thread counts within the kernels' launch bounds;
* TMA boxes within 256 elements per dimension, with 16-byte inner extents,
  and stage / operand bases 1024-byte aligned;
* tiles that cover the whole output; halo extents that match the filter;
* tensor-core plans: TMEM columns a power of two that holds the double-
  buffered (partial) accumulators, the host MMA table within its bound and
  its offsets inside the operand regions, the grid = group chunks x CTAs
  per chunk; the staged epilogue's output boxes (TMA store) inside shared
  memory, 1024-byte aligned, covering the CTA's channels;
* the fused depthwise + projection planner: supported exactly on its shape
  rules, tiles within the MMA's 128 rows, every input box read inside its
  stage, the operand regions disjoint and inside shared memory.
"""
import json
import os
import shutil
import subprocess

import numpy as np
import pytest

from depthwise_convolution_forward_gb300 import inputs

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SMEM_BLOCK = 232448  # opt-in shared memory per block on sm_103a
SMEM_SM = 233472     # shared memory per SM
RESERVED = 1024      # per-block reservation


@pytest.fixture(scope="module")
def harness(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    out = tmp_path_factory.mktemp("plans")
    exes = {}
    for name in ("plan_tc", "plan_dw", "plan_select", "plan_bwt", "plan_fused"):
        exe = str(out / name)
        subprocess.run([nvcc, "-std=c++17", "-O1", "-gencode", "arch=compute_103a,code=sm_103a",
                        "--expt-relaxed-constexpr", "-I" + os.path.join(ROOT, "include"),
                        os.path.join(HERE, "harness", name + ".cu"), "-o", exe],
                       check=True, capture_output=True, text=True)
        exes[name] = exe
    return exes


def _extent(i, k, s, p, d):
    room = i + 2 * p - (d * (k - 1) + 1)
    return room // s + 1 if room >= 0 else 0


def _geom(wl):
    out = [_extent(wl.inp[i], wl.ker[i], wl.stride[i], wl.pad[i], wl.dil[i]) for i in range(3)]
    return out, [wl.N, wl.G, wl.Cg, wl.Kg, *wl.inp, *out, *wl.ker, *wl.stride, *wl.pad, *wl.dil, wl.ndim]


def _run(exe, lines):
    r = subprocess.run([exe], input="\n".join(lines) + "\n", capture_output=True, text=True, check=True,
                       timeout=300)
    return [json.loads(ln) for ln in r.stdout.splitlines()]


def _problems(seed, n, **kw):
    rng = np.random.default_rng(seed)
    return [inputs.random_problem(rng, **kw) for _ in range(n)]


def _dw_candidates():
    probs = [wl for wl in inputs.all_workloads() if (wl.Cg == 1 and wl.Kg == 1) or
             (wl.Cg == 2 and wl.Kg == 2 and wl.ndim == 2)]
    rng2 = np.random.default_rng(78)
    for _ in range(40):  # groups of two channels (column form only)
        s, d = int(rng2.integers(1, 3)), int(rng2.integers(1, 3))
        hw = [int(rng2.integers(1, 60)), int(rng2.integers(1, 60))]
        wl = inputs.Workload("g2", 0, 0, 2, int(rng2.integers(1, 5)), 4 * int(rng2.integers(1, 80)), 2, 2,
                             (1, *hw), (1, 3, 3), (1, s, s), (0, d, d), (1, d, d),
                             str(rng2.choice(["f16", "bf16"])), True)
        if min(_geom(wl)[0]) >= 1:
            probs.append(wl)
    probs += [inputs.by_name("mbv2_dw_s1_f16").with_(N=4800)]
    rng = np.random.default_rng(77)
    for _ in range(300):
        dt = str(rng.choice(["f16", "bf16", "f32"]))
        vec = 4 if dt == "f32" else 8
        s, d = int(rng.integers(1, 3)), int(rng.integers(1, 3))
        nd = int(rng.choice([2, 2, 3]))
        hw = [int(rng.integers(1, 80)), int(rng.integers(1, 80))]
        z = int(rng.choice([1, 3])) if nd == 3 else 1
        dz = int(rng.integers(1, 3)) if nd == 3 else 1
        inp = (int(rng.integers(max(1, dz * (z - 1) + 1), 9)) if nd == 3 else 1, *hw)
        wl = inputs.Workload("r", 0, 0, nd, int(rng.integers(1, 9)), vec * int(rng.integers(1, 65)), 1, 1,
                             inp, (z, 3, 3), (1 if nd == 2 else int(rng.integers(1, 3)), s, s),
                             (0 if nd == 2 else int(rng.integers(0, 2)), d, d), (dz, d, d), dt, True)
        if min(_geom(wl)[0]) >= 1:
            probs.append(wl)
    return probs


def test_depthwise_plans(harness):
    probs = _dw_candidates()
    lines = []
    for wl in probs:
        es = 4 if wl.dtype == "f32" else 2
        lines.append(" ".join(map(str, _geom(wl)[1] + [es, 96, 0, 0, 0, 0])))  # 96 registers: above any build's
    res = _run(harness["plan_dw"], lines)
    assert len(res) == len(probs)
    planned = 0
    for wl, p in zip(probs, res):
        if p["ok"]:
            planned += 1
            _check_dw_plan(wl, p)
    assert planned >= 0.9 * len(probs)


@pytest.mark.parametrize("name", ["mbv2_dw_s1_f16", "mbv2_dw_s2_f16", "sweep_g512_d2_s1_bf16"])
def test_depthwise_overridden_plans(harness, name):
    """Tile overrides of the column form (TH x TW x stages x CTAs per SM): every
    plan they produce keeps the invariants, and the override is honoured."""
    wl = inputs.by_name(name)
    combos = [(th, tw, st, ct) for th in (0, 2, 4, 7, 14) for tw in (0, 7, 14, 28) for st in (0, 2, 3, 4)
              for ct in (0, 1, 2, 3)]
    lines = [" ".join(map(str, _geom(wl)[1] + [2, 96, th, tw, st, ct])) for th, tw, st, ct in combos]
    res = _run(harness["plan_dw"], lines)
    planned = 0
    for (th, tw, st, ct), p in zip(combos, res):
        if not p["ok"]:
            continue
        planned += 1
        assert (not th or p["TH"] == th) and (not tw or p["TW"] == tw), (th, tw, p)
        assert (not st or p["stages"] == st) and (not ct or p["ctas"] == ct), (st, ct, p)
        _check_dw_plan(wl, p)
    assert planned >= len(combos) // 4, planned


def _check_dw_plan(wl, p):
    """Invariants of one depthwise plan (see the module docstring)."""
    out = _geom(wl)[0]
    es = 4 if wl.dtype == "f32" else 2
    ctx = (wl, p)
    assert p["smem"] <= SMEM_BLOCK, ctx
    assert p["ctas"] * (p["smem"] + RESERVED) <= SMEM_SM, ctx
    assert p["threads"] % 32 == 0 and p["threads"] <= 1024, ctx
    if p["col"]:
        assert p["threads"] <= p["max_threads"], ctx
    assert p["TC"] <= 256 and (p["TC"] * es) % 16 == 0 and wl.C % p["TC"] == 0, ctx
    assert max(p["Wh"], p["Hh"], p["Dh"]) <= 256, ctx
    assert p["stage_off"] % 1024 == 0 and p["stage_stride"] % 1024 == 0, ctx
    assert p["stage_bytes"] == p["Dh"] * p["Hh"] * p["Wh"] * p["TC"] * es, ctx
    assert p["stage_bytes"] <= p["stage_stride"], ctx
    assert p["smem"] >= p["stage_off"] + p["stages"] * p["stage_stride"], ctx
    assert 2 <= p["stages"] <= 4, ctx
    assert p["Hh"] == (p["TH"] - 1) * wl.stride[1] + 2 * wl.dil[1] + 1, ctx
    assert p["tiles_h"] * p["TH"] >= out[1] and (p["tiles_h"] - 1) * p["TH"] < out[1], ctx
    assert p["tiles_w"] * p["TW"] >= out[2] and (p["tiles_w"] - 1) * p["TW"] < out[2], ctx
    assert p["num_tiles"] == p["tiles_c"] * p["tiles_w"] * p["tiles_h"] * out[0] * wl.N, ctx
    if p["col"]:
        assert p["h0"] == p["Hh"], ctx  # one copy per tile unless requested


def _tc_candidates():
    probs = [wl for wl in inputs.all_workloads() if wl.dtype != "f32" and not (wl.Cg == 1 and wl.Kg == 1)]
    probs += [inputs.by_name("sweep_g32_d1_s1_bf16").with_(N=5400)]
    # random shapes with a merge factor: per-group channels that 16-channel
    # MMA operands can pack, and enough groups to merge
    rng = np.random.default_rng(99)
    for wl in _problems(99, 400, max_c=64, max_hw=40):
        cg, kg = (int(rng.choice([2, 4, 8, 16, 32, 64])) for _ in range(2))
        G = int(rng.choice([1, 2, 4, 8, 16, 32])) * max(1, 16 // min(cg, kg))
        probs.append(wl.with_(Cg=cg, Kg=kg, G=G, N=int(rng.integers(1, 9)),
                              dtype="bf16" if wl.dtype == "f32" else wl.dtype))
    return [wl for wl in probs if wl.stride[1] == wl.stride[2] and wl.stride[1] <= 2 and min(_geom(wl)[0]) >= 1]


def _check_tc_plan(wl, p):
    """Invariants of one tensor-core plan (see the module docstring)."""
    out = _geom(wl)[0]
    ctx = (wl, p)
    G2 = p["sc"] * p["nmt"]
    assert p["smem"] <= SMEM_BLOCK, ctx
    assert p["tmem_cols"] in (32, 64, 128, 256, 512), ctx
    # 2..4 buffers of (partial) accumulators, all of them in the allocation
    assert 2 <= p["nbuf"] <= 4, ctx
    assert p["tmem_cols"] >= p["nbuf"] * p["np"] * G2 * p["Nn"], ctx
    # as many buffers as 512 columns hold
    assert p["nbuf"] == min(4, 512 // (p["np"] * G2 * p["Nn"])), ctx
    if p["tmem_cols"] > 256:  # a second CTA could not allocate beside it: keep it off the SM
        assert p["smem"] + RESERVED > SMEM_SM // 2, ctx
    assert 1 <= p["np"] <= max(1, wl.taps), ctx
    assert p["Nn"] % 16 == 0 and 16 <= p["Nn"] <= 256, ctx
    assert p["a_off"] % 1024 == 0 and p["b_off"] % 1024 == 0 and p["a_stage_bytes"] % 1024 == 0, ctx
    assert p["plane_stride"] % (128 if p["sw"] else 16) == 0, ctx
    assert p["a_off"] + p["stages"] * p["a_stage_bytes"] <= p["smem"], ctx
    assert p["tx_bytes"] <= p["a_stage_bytes"], ctx
    assert 2 <= p["stages"] <= 4, ctx
    # TMA boxes: (channels, P, Hh, Dh, 1) with at most 256 per dimension
    assert p["P"] <= 256 and p["Hh"] * wl.stride[1] <= 256 + 2 and p["Dh"] <= 256, ctx
    assert p["TH"] * p["tiles_h"] >= out[1] and p["TWo"] * p["tiles_w"] >= out[2], ctx
    assert p["spatial"] == wl.N * out[0] * p["tiles_h"] * p["tiles_w"], ctx
    assert p["grid"] == (p["n_gc"] // p["sc"]) * p["cpg"], ctx
    assert 0 <= p["ntab"] <= 2048, ctx
    # row shift: accumulator row f holds flattened output f + shift; the
    # tile's outputs still fit its M tiles, and the earliest A start (rows
    # before the plane, which feed only unstored rows) stays in shared memory
    assert -8 < p["shift"] <= 0, ctx
    assert p["TH"] * p["P"] - p["shift"] <= p["nmt"] * 128, ctx
    if p["ntab"]:
        assert p["a_off"] <= p["max_a"] < p["a_off"] + p["a_stage_bytes"], ctx
        assert p["a_off"] + 8 * p["shift"] * (128 if p["sw"] else 16) <= p["min_a"], ctx
        assert p["min_a"] >= 1024, ctx
        assert p["b_off"] <= p["max_b"] < p["a_off"], ctx
    assert p["bias_off"] < p["tab_off"] <= p["b_off"], ctx
    if p["epi_off"]:  # output box staged for TMA stores, one box per channel slice
        assert p["epi_off"] % 1024 == 0 and p["epi_slice_bytes"] % 1024 == 0, ctx
        assert p["epi_off"] >= p["a_off"] + p["stages"] * p["a_stage_bytes"], ctx
        assert p["epi_off"] + p["epi_slices"] * p["epi_slice_bytes"] <= p["smem"], ctx
        assert p["epi_w"] in (32, 64, 128) and p["epi_w"] * p["epi_slices"] == p["sc"] * p["Nn"] * 2, ctx
        assert p["TH"] * p["TWo"] * p["epi_w"] <= p["epi_slice_bytes"], ctx
        assert p["TWo"] <= 256 and p["TH"] <= 256, ctx


def test_tensor_core_plans(harness):
    probs = _tc_candidates()
    lines = [" ".join(map(str, _geom(wl)[1] + [int(wl.dtype == "bf16"), 0, 0, 0, 0, 0])) for wl in probs]
    res = _run(harness["plan_tc"], lines)
    assert len(res) == len(probs)
    planned = mergeable = 0
    for wl, p in zip(probs, res):
        mergeable += p["m"] > 0
        if p["ok"]:
            planned += 1
            _check_tc_plan(wl, p)
    assert mergeable >= 0.8 * len(probs)
    assert planned >= 0.9 * mergeable, (planned, mergeable)


@pytest.mark.parametrize("name", ["sweep_g8_d1_s1_bf16", "resnext_a_bf16", "resnext_b_bf16", "resnext3d_n8_f16"])
def test_tensor_core_overridden_plans(harness, name):
    """Tile overrides (M tiles per CTA x partial accumulators x stages): every
    combination whose accumulators fit tensor memory gets a plan, and every
    plan keeps the invariants."""
    wl = inputs.by_name(name)
    combos = [(nmt, np_, st) for nmt in (1, 2, 3, 4) for np_ in (1, 2, 4) for st in (0, 2, 3)]
    lines = [" ".join(map(str, _geom(wl)[1] + [int(wl.dtype == "bf16"), 0, nmt, st, np_, 0])) for nmt, np_, st in combos]
    res = _run(harness["plan_tc"], lines)
    auto = _run(harness["plan_tc"], [" ".join(map(str, _geom(wl)[1] + [int(wl.dtype == "bf16"), 0, 0, 0, 0, 0]))])[0]
    assert auto["ok"]
    G2_per_nmt = auto["sc"]  # accumulators per M tile
    for (nmt, np_, st), p in zip(combos, res):
        if p["ok"]:
            assert p["nmt"] == nmt and p["np"] == np_, (nmt, np_, p)
            if st:
                assert p["stages"] <= st
            _check_tc_plan(wl, p)
        elif np_ <= wl.taps and 2 * np_ * G2_per_nmt * nmt * auto["Nn"] <= 512 and nmt <= 2 and st == 0:
            # small tiles that fit tensor memory must be plannable
            raise AssertionError(f"{name}: no plan for nmt {nmt} np {np_}")


def _select_candidates():
    """Every workload family, random grouped problems in all dtypes, and the
    deep depthwise 3D filters whose smallest whole-pixel tile overflows a
    stage (fp32 C=256 3x3x3; fp16 C=256 depth 5 dilated 2)."""
    probs = [wl for wl in inputs.all_workloads()]
    probs += [inputs.Workload("dw3d_f32_c256", 0, 0, 3, 2, 256, 1, 1, (8, 28, 28), (3, 3, 3), (1, 1, 1),
                              (1, 1, 1), (1, 1, 1), "f32", True),
              inputs.Workload("dw3d_f16_c256_z5", 0, 0, 3, 2, 256, 1, 1, (12, 28, 28), (5, 3, 3), (1, 1, 1),
                              (4, 1, 1), (2, 1, 1), "f16", True)]
    probs += _dw_candidates()[:120]
    probs += _tc_candidates()[:200]
    return [wl for wl in probs if min(_geom(wl)[0]) >= 1]


@pytest.mark.parametrize("sms", [132, 148, 152, 160])
def test_selector_agrees_with_launch_planners(harness, sms):
    """The selector takes a specialised kernel only when that kernel's
    launcher finds a plan on a device with the same SM count and shared
    memory, so an auto-selected problem never fails for want of a plan."""
    probs = _select_candidates()
    code = {"f32": 0, "f16": 1, "bf16": 2}
    lines = [" ".join(map(str, _geom(wl)[1] + [code[wl.dtype], sms, SMEM_BLOCK, 96])) for wl in probs]
    res = _run(harness["plan_select"], lines)
    assert len(res) == len(probs)
    for wl, r in zip(probs, res):
        if r["dw_sel"]:
            assert r["dw_plan"], (wl, r)
        assert bool(r["tc_sel"]) == bool(r["tc_plan"]), (wl, r)
    by_name = {wl.name: r for wl, r in zip(probs, res)}
    # the deep 3D depthwise filters are planned with narrower channel tiles
    for name in ("dw3d_f32_c256", "dw3d_f16_c256_z5"):
        assert by_name[name]["dw_sel"] and by_name[name]["dw_plan"], by_name[name]
        assert by_name[name]["dw_TC"] < 256, by_name[name]


def _bwt_candidates():
    """Every 16-bit workload family and random grouped problems in the
    backward-weight tensor-core route's shape range (Cg == Kg dividing 64)."""
    probs = [wl for wl in inputs.all_workloads() if wl.dtype != "f32"]
    rng = np.random.default_rng(91)
    for i in range(300):
        Cg = int(rng.choice([1, 2, 4, 8, 16, 32, 64]))
        G = 64 // Cg * int(rng.integers(1, 5))
        nd = 3 if rng.random() < 0.2 else 2
        s = int(rng.integers(1, 3))
        k = int(rng.integers(1, 5))
        d = int(rng.integers(1, 3))
        hw = (int(rng.integers(2, 70)), int(rng.integers(2, 70)))
        inp = (int(rng.integers(2, 9)) if nd == 3 else 1, *hw)
        ker = (int(rng.integers(1, 4)) if nd == 3 else 1, k, k)
        pad = (int(rng.integers(0, 2)) if nd == 3 else 0, int(rng.integers(0, k)), int(rng.integers(0, k)))
        probs.append(inputs.Workload(f"bwt{i}", 0, i, nd, int(rng.integers(1, 4)), G, Cg, Cg, inp, ker,
                                     (1, s, s), pad, (1, d, d), "bf16" if i % 2 else "f16", False))
    return [wl for wl in probs if min(_geom(wl)[0]) >= 1]


def test_backward_weight_tc_plans(harness):
    """The tensor-core backward-weight plans keep every copy, MMA operand,
    accumulator column and workspace write inside its buffer, and their
    phase / offset tables reproduce the convolution's input coordinates."""
    probs = _bwt_candidates()
    lines = [" ".join(map(str, _geom(wl)[1] + [int(wl.dtype == "f16")])) for wl in probs]
    res = _run(harness["plan_bwt"], lines)
    assert len(res) == len(probs)
    n_ok = 0
    for wl, p in zip(probs, res):
        shape_ok = wl.Cg == wl.Kg and 64 % wl.Cg == 0 and (wl.G * wl.Cg) % 64 == 0 and \
            wl.stride[1] == wl.stride[2] and wl.stride[1] <= 2 and wl.ker[2] <= 4
        if not p["ok"]:
            continue
        n_ok += 1
        ctx = (wl, p)
        assert shape_ok, ctx
        s = wl.stride[1]
        out, _ = _geom(wl)
        Ho, Wo = out[1], out[2]
        X, Y, Z = wl.ker[2], wl.ker[1], wl.ker[0]
        # copies: boxes within TMA limits, landing inside their regions
        assert s * p["P"] <= 256 and s * p["TH"] <= 256 and p["P"] <= 256, ctx
        assert p["Kp"] % 16 == 0 and p["Kp"] >= 32 and p["TH"] * p["P"] <= p["Kp"], ctx
        assert p["tx_bytes"] == (1 + p["nplane"]) * p["TH"] * p["P"] * 128, ctx
        assert p["dy_bytes"] % 1024 == 0 and p["dy_bytes"] >= p["Kp"] * 128, ctx
        assert p["plane_bytes"] % 1024 == 0 and p["stage_bytes"] == p["dy_bytes"] + p["nplane"] * p["plane_bytes"]
        assert 2 <= p["stages"] <= 4, ctx
        assert 1024 + p["stages"] * p["stage_bytes"] <= p["smem"] <= SMEM_BLOCK, ctx
        # MMA operands: the last K step's B rows stay inside the x plane
        for r in p["runs"]:
            last = p["Kp"] - 16 + r["u0"] + (r["len"] - 1) * r["du"] + 15
            assert last < p["plane_bytes"] // 128, ctx
            assert r["idesc"] >> 24 == 4 and (r["idesc"] >> 17) & 63 == 64 * r["len"] // 8, ctx
            assert (r["idesc"] >> 15) & 3 == 3, ctx  # both operands MN-major
        # taps: every tap of the row exactly once, each at its input column
        kxs = sorted(k for r in p["runs"] for k in r["kx"])
        assert kxs == list(range(X)), ctx
        for r in p["runs"]:
            for b, kx in enumerate(r["kx"]):
                v = kx * wl.dil[2] - wl.pad[2]
                px = v % s
                qx = (v - px) // s
                assert px == p["plane_px"][r["plane"]], ctx
                assert qx - p["qx_min"] == r["u0"] + b * r["du"], ctx
                assert 0 <= r["u0"] + b * r["du"] <= p["P"] - Wo, ctx
        for kz in range(Z):
            for ky in range(Y):
                rr = kz * Y + ky
                assert s * p["row_qy"][rr] + p["row_py"][rr] == ky * wl.dil[1] - wl.pad[1], ctx
        # tensor memory: two accumulator sets of 64 columns per tap
        assert p["ncols"] == 64 * X and p["tmem_cols"] >= 2 * p["ncols"], ctx
        assert p["tmem_cols"] in (32, 64, 128, 256, 512), ctx
        if p["tmem_cols"] > 256:
            assert p["smem"] > SMEM_SM // 2, ctx
        # work split and workspace
        assert p["tiles_h"] * p["TH"] >= Ho and p["tiles"] == wl.N * out[0] * p["tiles_h"], ctx
        assert 1 <= p["S"] <= p["tiles"], ctx
        assert p["rows"] == Z * Y and p["chunks"] * 64 == wl.G * wl.Cg, ctx
        assert p["grid"] == p["rows"] * p["chunks"] * p["S"], ctx
        assert p["E"] == wl.G * wl.Kg * X * Y * Z * wl.Cg, ctx
    assert n_ok >= 150



def _fused_candidates():
    """MobileNetV2 layers, the fused kernel's GPU test shapes, and random
    shapes inside and just outside its rules."""
    probs = []
    for name in ("mbv2_dw_s1_f16", "mbv2_dw_s2_f16"):
        probs.append((inputs.by_name(name), 24, 2))
    for C, H, W, s, p in [(16, 13, 13, 1, 1), (32, 10, 9, 1, 0), (16, 7, 128, 1, 1), (48, 15, 21, 2, 1),
                          (32, 5, 253, 2, 1), (256, 6, 14, 1, 1), (64, 17, 19, 1, 1)]:
        for K in (8, 24, 32, 64, 256):
            probs.append((inputs.Workload("fz", 0, 0, 2, 3, C, 1, 1, (1, H, W), (1, 3, 3), (1, s, s), (0, p, p),
                                          (1, 1, 1), "bf16", True), K, 1))
    rng = np.random.default_rng(77)
    for i in range(400):
        C = int(rng.choice([8, 16, 24, 32, 48, 64, 96, 144, 160, 192, 240, 256, 272]))
        K = int(rng.choice([4, 8, 16, 24, 40, 64, 128, 200, 256, 264]))
        s = int(rng.choice([1, 1, 2, 3]))
        H, W = int(rng.integers(1, 300)), int(rng.integers(1, 300))
        p = int(rng.integers(0, 3))
        if H + 2 * p < 3 or W + 2 * p < 3:
            continue
        probs.append((inputs.Workload("fz", 0, i, 2, int(rng.integers(1, 5)), C, 1, 1, (1, H, W), (1, 3, 3),
                                      (1, s, s), (0, p, p), (1, 1, 1), "f16", True), K, int(rng.integers(0, 4))))
    return probs


def test_fused_block_plans(harness):
    probs = _fused_candidates()
    lines = [" ".join(map(str, _geom(wl)[1] + [int(wl.dtype == "bf16"), K, act])) for wl, K, act in probs]
    res = _run(harness["plan_fused"], lines)
    assert len(res) == len(probs)
    n_ok = 0
    for (wl, K, act), p in zip(probs, res):
        ctx = (wl, K, act, p)
        C, s = wl.G, wl.stride[1]
        rules = wl.ndim == 2 and C % 16 == 0 and C <= 256 and K % 8 == 0 and 8 <= K <= 256 and 0 <= act <= 2 \
            and s in (1, 2)
        assert p["ok"] == rules, ctx
        if not p["ok"]:
            continue
        n_ok += 1
        out, _ = _geom(wl)
        Ho, Wo = out[1], out[2]
        TH, TW = p["TH"], p["TW"]
        # tiles: at most 128 pixel rows of the MMA, covering the output
        assert 1 <= TW <= 16 and 1 <= TH <= Ho and TW <= Wo and TH * TW <= 128, ctx
        assert p["tiles_h"] == -(-Ho // TH) and p["tiles_w"] == -(-Wo // TW), ctx
        assert p["tiles"] == wl.N * p["tiles_h"] * p["tiles_w"], ctx
        # input box: the tile's halo; TMA box limits and a 16-byte inner extent
        assert p["Win"] == (TW - 1) * s + 3 and p["Hin"] == (TH - 1) * s + 3, ctx
        assert max(p["Win"], p["Hin"], p["CH"]) <= 256 and (2 * p["CH"]) % 16 == 0, ctx
        assert p["CH"] * p["chunks"] == C and p["GC"] * p["cpt"] == p["CH"] and p["GT"] * p["cpt"] == C, ctx
        assert p["cpt"] in (4, 8) and (2 * p["cpt"]) % 8 == 0, ctx
        assert p["x_stage_bytes"] == p["Hin"] * p["Win"] * p["CH"] * 2, ctx
        # the walk's last read (row (TH-1)s+2, column (TW-1)s+2, last group)
        # ends exactly at the end of the stage
        rowb, pixb = p["Win"] * p["CH"] * 2, p["CH"] * 2
        last = ((TH - 1) * s + 2) * rowb + ((TW - 1) * s + 2) * pixb + (p["GC"] - 1) * 2 * p["cpt"] + 2 * p["cpt"]
        assert last == p["x_stage_bytes"] <= p["x_stage_stride"], ctx
        assert p["x_stage_stride"] % 1024 == 0, ctx
        # a whole tile's copies fit the ring
        assert p["chunks"] <= p["stages"] <= p["max_stages"], ctx
        # compute items: every (row, column, group) of a tile in exactly one
        # segment of one column walk
        assert p["NS"] * p["rps"] >= TH and (p["NS"] - 1) * p["rps"] < TH, ctx
        assert p["G"] == C // 8, ctx
        # shared-memory regions: disjoint, in order, aligned, inside the block
        assert p["wdw_off"] >= 264 and p["bdw_off"] >= p["wdw_off"] + 18 * C, ctx
        assert p["bdw_off"] % 16 == 0 and p["bpw_off"] >= p["bdw_off"] + 2 * C and p["bpw_off"] % 4 == 0, ctx
        assert p["b_off"] >= p["bpw_off"] + 4 * p["Np"] and p["b_off"] % 1024 == 0, ctx
        assert p["a_off"] >= p["b_off"] + p["G"] * p["Np"] * 16 and p["a_off"] % 1024 == 0, ctx
        # A: whole 64-channel swizzled atoms, then the C % 64 tail in groups of
        # 2 KB + 16 B, the buffer rounded up to 1 KB
        tail = (C // 64) * p["atom"] + (C % 64) // 8 * 2064
        assert p["a_bytes"] == -(-tail // 1024) * 1024 and p["atom"] == 128 * 128, ctx
        assert p["a_bytes"] % 1024 == 0, ctx
        assert p["nA"] in (1, 2, 3) and p["x_off"] == p["a_off"] + p["nA"] * p["a_bytes"], ctx
        assert p["smem"] == p["x_off"] + p["stages"] * p["x_stage_stride"] <= SMEM_BLOCK, ctx
        # projection: N = K rounded up to 16; two accumulators in TMEM
        assert p["Np"] == -(-K // 16) * 16, ctx
        assert p["tmem_cols"] in (32, 64, 128, 256, 512) and p["tmem_cols"] >= 2 * p["Np"], ctx
        assert p["idesc"] >> 24 == 8 and (p["idesc"] >> 17) & 63 == p["Np"] // 8, ctx
        # 8 channels per thread with 8 compute warps, 4 with 16 (+ 6 warps of other roles)
        assert p["compute_threads"] == {8: 256, 4: 512}[p["cpt"]], ctx
        assert p["threads"] == p["compute_threads"] + 192, ctx
        # the compute warps issue the MMAs exactly when fewer than three A buffers fit
        assert p["inline_mma"] == (p["nA"] < 3), ctx
    assert n_ok > 100
    mb = {wl.name: p for (wl, _, _), p in zip(probs, res) if wl.name.startswith("mbv2")}
    # the MobileNetV2 layers get the plans measured best on GB300: 8 channels
    # per thread, 8 x 14 tiles with three A buffers and the issuing warp at
    # stride 1, 14 x 7 tiles with two A buffers and the compute warps issuing
    # the projection at stride 2
    s1, s2 = mb["mbv2_dw_s1_f16"], mb["mbv2_dw_s2_f16"]
    assert (s1["cpt"], s1["TH"], s1["TW"], s1["nA"], s1["inline_mma"]) == (8, 8, 14, 3, 0), s1
    assert (s2["cpt"], s2["TH"], s2["TW"], s2["nA"], s2["inline_mma"]) == (8, 14, 7, 2, 1), s2
