"""CUDA path vs the CPU oracle, element by element, through the C ABI.

* every workload family at reduced batch, compared on every output;
* every workload at its full benchmark size in the launch configuration the
  benchmark uses, compared on sampled outputs (random + padding borders);
* random small 2D/3D problems over all dtypes, auto-selected and forced onto
  each kernel that accepts them;
* edge cases: ragged tiles, odd sizes, 1x1 filters, channel counts that break
  16-byte vectors, misaligned input, integer inputs that must be bit-exact.
"""
import numpy as np
import pytest
import torch

import depthwise_convolution_forward_gb300 as gc
from depthwise_convolution_forward_gb300 import _binding as B
from depthwise_convolution_forward_gb300 import inputs
from gpu_util import assert_close, out_shape_of, require_gpu, run_gpu, sample_indices

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _reduced(wl):
    """Same family, small enough for a full oracle comparison in seconds."""
    if wl.cfg == 5:
        return wl.with_(N=2)
    if wl.cfg in (2, 3):
        return wl.with_(N=2)
    return wl.with_(N=min(wl.N, 2))


ALL = list(inputs.all_workloads())


@pytest.mark.parametrize("wl", ALL, ids=lambda w: w.name)
def test_reduced_batch_full_compare(orc, wl):
    r = _reduced(wl)
    x, w, b = inputs.make_inputs(r)
    y, sel = run_gpu(r, x, w, b)
    ref = orc.forward(r, x, w, b)
    assert_close(y.double().numpy(), ref, r.dtype, f"{r.name} (kernel {sel})")


@pytest.mark.parametrize("wl", ALL, ids=lambda w: w.name)
def test_full_size_sampled(orc, wl):
    x, w, b = inputs.make_inputs(wl)
    y, sel = run_gpu(wl, x, w, b)
    shape = out_shape_of(wl)
    idx = sample_indices(shape, 4000, seed=wl.variant + 17 * wl.cfg)
    ref = orc.points(wl, x, w, b, idx)
    got = y.reshape(-1)[torch.from_numpy(idx)].double().numpy()
    assert_close(got, ref, wl.dtype, f"{wl.name} (kernel {sel})")


def _forced_kernels(wl):
    ks = [B.KERNEL_DIRECT_GENERIC]
    if gc.grouped_conv_select(gc.problem_of(wl), gc.DTYPE_CODES[wl.dtype]) != B.KERNEL_DIRECT_GENERIC:
        ks.append(0)
    return ks


@pytest.mark.parametrize("seed", range(40))
def test_random_small_problems(orc, seed):
    rng = np.random.default_rng(1000 + seed)
    wl = inputs.random_problem(rng)
    x, w, b = inputs.make_inputs(wl)
    ref = orc.forward(wl, x, w, b)
    for k in _forced_kernels(wl):
        y, sel = run_gpu(wl, x, w, b, force=k)
        assert_close(y.double().numpy(), ref, wl.dtype, f"seed {seed} kernel {sel} {wl}")


DW_EDGE = [
    # (N, C, H, W, stride, pad, dil, dtype)
    (1, 8, 7, 7, 1, 1, 1, "f16"),
    (2, 16, 13, 11, 2, 1, 1, "bf16"),
    (1, 24, 9, 17, 2, 0, 1, "f16"),
    (1, 8, 12, 12, 1, 2, 2, "bf16"),
    (1, 8, 12, 12, 1, 0, 2, "f16"),
    (2, 16, 15, 15, 2, 2, 2, "bf16"),
    (1, 4, 10, 9, 1, 1, 1, "f32"),
    (1, 8, 10, 9, 2, 1, 1, "f32"),
    (1, 264, 9, 9, 1, 1, 1, "f16"),   # channels above one TMA box: channel tiles
    (1, 520, 6, 7, 2, 1, 1, "bf16"),  # channel tiles that do not divide C evenly
    (1, 16, 3, 300, 1, 1, 1, "f16"),  # wide rows: several column tiles
    (3, 32, 1, 1, 1, 1, 1, "bf16"),   # 1x1 input, padding only
    (1, 16, 3, 3, 2, 1, 2, "f16"),    # output 1x1, dilated
    # stride = dilation = 2 with padding a multiple of 2: every tap reads even
    # rows and columns, so the TMA forms run on the input subsampled by 2
    (1, 8, 14, 13, 2, 4, 2, "f16"),
    (1, 8, 11, 12, 2, 0, 2, "bf16"),
]


# depthwise kernel forms (tuning override slot 6): 1 row-blocked, 2 direct
# loads, 3 column form (the automatic choice for a depth filter of 1); slot 5
# selects the column form's operands: 1 split, 2 packed x4 (the automatic
# choice for 16-bit storage), 3 widened fp32x2, 4 packed x8
DW_FORMS = [(1, 0), (2, 0), (3, 0), (3, 1), (3, 3), (3, 4)]


@pytest.mark.parametrize("form", DW_FORMS, ids=lambda f: f"form{f[0]}-{f[1]}")
@pytest.mark.parametrize("case", DW_EDGE, ids=lambda c: "-".join(map(str, c)))
def test_depthwise_edges(orc, case, form):
    N, C, H, W, s, p, d, dt = case
    wl = inputs.Workload("dw_edge", 7, DW_EDGE.index(case), 2, N, C, 1, 1, (1, H, W), (1, 3, 3),
                         (1, s, s), (0, p, p), (1, d, d), dt, True)
    x, w, b = inputs.make_inputs(wl)
    y, sel = run_gpu(wl, x, w, b, force=B.KERNEL_DIRECT_DW, tile=[0, 0, 0, 0, 0, form[1], form[0]])
    assert sel == B.KERNEL_DIRECT_DW
    assert_close(y.double().numpy(), orc.forward(wl, x, w, b), dt, str(case))


# column form with explicit tiles (TH, TW, stages, CTAs per SM): ragged row
# and column tiles, one to three CTAs per SM, two to four stages.  Every tile
# set fits the shared memory of its workload.
COL_TILES = {
    "mbv2_dw_s1_f16": [(5, 3, 2, 1), (1, 1, 2, 2), (7, 13, 3, 1), (14, 8, 2, 2), (3, 5, 4, 3), (56, 2, 2, 1)],
    "mbv2_dw_s2_f16": [(5, 3, 2, 1), (1, 1, 2, 2), (7, 7, 2, 1), (3, 5, 2, 3), (28, 1, 2, 1)],
    "sweep_g512_d2_s1_bf16": [(5, 3, 2, 1), (1, 1, 2, 2), (7, 8, 2, 1), (3, 2, 2, 3)],
    "sweep_g512_d2_s2_bf16": [(5, 3, 2, 1), (1, 1, 2, 2), (3, 4, 2, 1), (2, 2, 2, 3), (14, 1, 2, 1)],
}
COL_CASES = [(n, t) for n, ts in COL_TILES.items() for t in ts]


@pytest.mark.parametrize("one_copy", [2, 0], ids=["split-copy", "one-copy"])
@pytest.mark.parametrize("name,tiles", COL_CASES, ids=lambda v: v if isinstance(v, str) else "-".join(map(str, v)))
def test_depthwise_column_tiles(orc, name, tiles, one_copy):
    """Explicit tiles; each CTA's first tile either as two copies on two
    barriers (slot 2 = 2, where the split point is aligned) or as one copy."""
    TH, TW, stages, ctas = tiles
    wl = inputs.by_name(name).with_(N=2)
    x, w, b = inputs.make_inputs(wl)
    ref = orc.forward(wl, x, w, b)
    y, sel = run_gpu(wl, x, w, b, force=B.KERNEL_DIRECT_DW, tile=[TH, TW, one_copy, stages, ctas, 0, 3])
    assert sel == B.KERNEL_DIRECT_DW
    assert_close(y.double().numpy(), ref, wl.dtype, f"{name} tiles {tiles}")


@pytest.mark.parametrize("name", ["resnext_b_bf16", "sweep_g8_d1_s1_bf16", "resnext3d_n1_f16", "sweep_g256_d2_s2_bf16",
                                  "resnext_a_bf16", "sweep_g64_d2_s1_bf16"])
@pytest.mark.parametrize("staged", [True, False], ids=["tma-store", "registers"])
def test_tensor_core_epilogue_paths(orc, name, staged):
    """Both epilogues of the tensor-core kernel: stores straight from
    registers (the default), and the output box staged in shared memory and
    written by TMA tensor stores (override slot 7 < 0).  The workloads cover
    128-, 64-byte channel slices, ragged bottom and right tile edges that the
    TMA store clips, and one to four partial accumulators."""
    wl = inputs.by_name(name).with_(N=min(inputs.by_name(name).N, 2))
    x, w, b = inputs.make_inputs(wl)
    ref = orc.forward(wl, x, w, b)
    tile = [0, 0, 0, 0, 0, 0, 0, -1] if staged else None
    y, sel = run_gpu(wl, x, w, b, force=B.KERNEL_IGEMM_TC, tile=tile)
    assert sel == B.KERNEL_IGEMM_TC
    assert_close(y.double().numpy(), ref, wl.dtype, f"{name} staged={staged}")


ALIGNED_CASES = [
    inputs.by_name("resnext_a_bf16").with_(N=2),
    inputs.by_name("sweep_g64_d1_s1_bf16").with_(N=2),
    inputs.by_name("sweep_g8_d1_s1_bf16").with_(N=2),
    inputs.by_name("sweep_g32_d2_s1_bf16").with_(N=2),
    inputs.by_name("sweep_g64_d2_s2_bf16").with_(N=2),
    # ragged: odd width (pitch padded 23 -> 24), rows not a multiple of the tile
    inputs.Workload("al_odd", 7, 2, 2, 2, 8, 16, 16, (1, 19, 23), (1, 3, 3), (1, 1, 1), (0, 1, 1), (1, 1, 1),
                    "bf16", True),
    inputs.Workload("al_f16", 7, 3, 2, 1, 16, 8, 8, (1, 17, 30), (1, 3, 3), (1, 1, 1), (0, 1, 1), (1, 2, 2),
                    "f16", True),
]


@pytest.mark.parametrize("wl", ALIGNED_CASES, ids=lambda w: w.name)
def test_tensor_core_aligned_copies(orc, wl):
    """Tensor-core kernel with one copy of the tile per column shift
    (override slot 5 = 2: every tap's A operand starts on an 8-row
    boundary) against the oracle, and slot 5 = 1 (shifted starts)."""
    x, w, b = inputs.make_inputs(wl)
    ref = orc.forward(wl, x, w, b)
    for mode in (2, 1):
        y, sel = run_gpu(wl, x, w, b, force=B.KERNEL_IGEMM_TC, tile=[0, 0, 0, 0, 0, mode, 0, 0])
        assert sel == B.KERNEL_IGEMM_TC
        assert_close(y.double().numpy(), ref, wl.dtype, f"{wl.name} plane mode {mode}")


def test_depthwise_3d(orc):
    wl = inputs.Workload("dw3d", 7, 1, 3, 2, 16, 1, 1, (5, 9, 10), (3, 3, 3), (2, 1, 1), (1, 1, 1),
                         (1, 1, 1), "f16", True)
    x, w, b = inputs.make_inputs(wl)
    y, sel = run_gpu(wl, x, w, b, force=B.KERNEL_DIRECT_DW)
    assert_close(y.double().numpy(), orc.forward(wl, x, w, b), "f16", "dw3d")


@pytest.mark.parametrize("wl", [
    # the smallest whole-pixel tile of these overflows a stage, so the planner
    # narrows the channel tile (fp32 C=256 3x3x3; fp16 C=256, depth 5 dilated 2)
    inputs.Workload("dw3d_f32_c256", 7, 2, 3, 2, 256, 1, 1, (8, 14, 14), (3, 3, 3), (1, 1, 1), (1, 1, 1),
                    (1, 1, 1), "f32", True),
    inputs.Workload("dw3d_f16_c256_z5", 7, 3, 3, 1, 256, 1, 1, (12, 10, 10), (5, 3, 3), (1, 1, 1), (4, 1, 1),
                    (2, 1, 1), "f16", True),
], ids=lambda w: w.name)
def test_depthwise_3d_channel_tiles(orc, wl):
    x, w, b = inputs.make_inputs(wl)
    assert gc.grouped_conv_select(gc.problem_of(wl), gc.DTYPE_CODES[wl.dtype]) == B.KERNEL_DIRECT_DW
    y, sel = run_gpu(wl, x, w, b)
    assert sel == B.KERNEL_DIRECT_DW
    assert_close(y.double().numpy(), orc.forward(wl, x, w, b), wl.dtype, wl.name)


G2_EDGE = [
    # (N, G, H, W, stride, pad, dil, dtype, tiles): groups of two channels on
    # the column kernel (Cg == Kg == 2), forced, with ragged and explicit tiles
    (2, 8, 13, 11, 1, 1, 1, "bf16", None),
    (1, 12, 9, 17, 2, 0, 1, "f16", None),
    (1, 8, 12, 12, 1, 2, 2, "bf16", None),
    (2, 16, 15, 15, 2, 2, 2, "f16", None),
    (1, 260, 6, 7, 1, 1, 1, "bf16", None),  # 520 channels: channel tiles
    (2, 64, 28, 28, 1, 1, 1, "bf16", (5, 3, 0, 2, 1, 0, 3)),
    (2, 64, 28, 28, 1, 1, 1, "f16", (3, 5, 0, 4, 2, 0, 3)),
    (1, 4, 1, 1, 1, 1, 1, "bf16", None),  # 1x1 input, padding only
]


@pytest.mark.parametrize("case", G2_EDGE, ids=lambda c: "-".join(map(str, c[:8])))
def test_group2_column_kernel(orc, case):
    N, G, H, W, s, p, d, dt, tiles = case
    wl = inputs.Workload("g2_edge", 7, G2_EDGE.index(case), 2, N, G, 2, 2, (1, H, W), (1, 3, 3), (1, s, s),
                         (0, p, p), (1, d, d), dt, True)
    x, w, b = inputs.make_inputs(wl)
    y, sel = run_gpu(wl, x, w, b, force=B.KERNEL_DIRECT_DW, tile=list(tiles) if tiles else None)
    assert sel == B.KERNEL_DIRECT_DW
    assert_close(y.double().numpy(), orc.forward(wl, x, w, b), dt, str(case))


def test_group2_selection():
    """Stride 1 runs on the column kernel, stride 2 on the tensor-core kernel."""
    s1 = gc.problem_of(inputs.by_name("sweep_g256_d1_s1_bf16"))
    s2 = gc.problem_of(inputs.by_name("sweep_g256_d1_s2_bf16"))
    assert gc.grouped_conv_select(s1, B.GCONV_BF16) == B.KERNEL_DIRECT_DW
    assert gc.grouped_conv_select(s2, B.GCONV_BF16) == B.KERNEL_IGEMM_TC


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
def test_integer_inputs_bit_exact(orc, dt):
    """Small integers: every product and partial sum is exact in fp32 and the
    result is representable, so GPU and oracle must agree exactly."""
    for wl in (inputs.Workload("int_dw", 8, 0, 2, 2, 32, 1, 1, (1, 11, 10), (1, 3, 3), (1, 1, 1),
                               (0, 1, 1), (1, 1, 1), dt, True),
               inputs.Workload("int_grp", 8, 1, 2, 1, 4, 3, 5, (1, 7, 6), (1, 3, 3), (1, 2, 1),
                               (0, 1, 1), (1, 1, 2), dt, True),
               inputs.Workload("int_g2", 8, 2, 2, 2, 16, 2, 2, (1, 9, 10), (1, 3, 3), (1, 1, 1),
                               (0, 1, 1), (1, 1, 1), dt, True)):
        g = torch.Generator().manual_seed(3)
        tdt = inputs.DTYPES[dt]
        x = torch.randint(-3, 4, wl.x_shape(), generator=g).to(tdt)
        w = torch.randint(-2, 3, wl.w_shape(), generator=g).to(tdt)
        b = torch.randint(-4, 5, (wl.K,), generator=g).to(tdt)
        ref = orc.forward(wl, x, w, b)
        for k in _forced_kernels(wl):
            y, _ = run_gpu(wl, x, w, b, force=k)
            assert np.array_equal(y.double().numpy(), ref), (wl.name, k)


def test_misaligned_input_falls_back(orc):
    wl = inputs.Workload("dw_mis", 7, 9, 2, 1, 16, 1, 1, (1, 8, 8), (1, 3, 3), (1, 1, 1), (0, 1, 1),
                         (1, 1, 1), "f16", True)
    x, w, b = inputs.make_inputs(wl)
    y, sel = run_gpu(wl, x, w, b, x_offset=1)
    assert sel == B.KERNEL_DIRECT_GENERIC
    assert_close(y.double().numpy(), orc.forward(wl, x, w, b), "f16", "misaligned")
    with pytest.raises(gc.GconvError) as e:
        run_gpu(wl, x, w, b, x_offset=1, force=B.KERNEL_DIRECT_DW)
    assert e.value.status == B.GCONV_ERR_UNSUPPORTED


def test_no_bias_and_groups_one(orc):
    for wl in (inputs.by_name("mbv2_dw_s1_f16").with_(N=1, bias=False),
               inputs.Workload("g1", 8, 2, 2, 1, 1, 12, 10, (1, 9, 9), (1, 3, 3), (1, 1, 1), (0, 1, 1),
                               (1, 1, 1), "bf16", False)):
        x, w, b = inputs.make_inputs(wl)
        y, _ = run_gpu(wl, x, w, None)
        assert_close(y.double().numpy(), orc.forward(wl, x, w, None), wl.dtype, wl.name)


def test_repeat_calls_and_streams(orc):
    wl = inputs.by_name("mbv2_dw_s2_f16").with_(N=2)
    x, w, b = inputs.make_inputs(wl)
    ref = orc.forward(wl, x, w, b)
    s = torch.cuda.Stream()
    for i in range(3):
        y, _ = run_gpu(wl, x, w, b, stream=s if i % 2 else None, debug=False)
        assert_close(y.double().numpy(), ref, wl.dtype, f"call {i}")
