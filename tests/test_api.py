"""Host-side C-ABI checks: library loads, exports what the header declares,
validates arguments and computes output shapes.  No GPU needed."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import depthwise_convolution_forward_gb300 as gc
from depthwise_convolution_forward_gb300 import _binding as B
from depthwise_convolution_forward_gb300 import build, inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return B.load_library()


def header_functions():
    src = open(os.path.join(ROOT, "include", "gconv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", src, flags=re.M)))


def test_header_symbols_exported(lib):
    names = header_functions()
    assert "grouped_conv_fwd" in names and len(names) >= 8, names
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    for n in names:
        assert n in exported, f"{n} declared in gconv.h but not exported"
        assert hasattr(lib, n)


def test_struct_layout():
    assert ctypes.sizeof(B.gconv_problem) == 88
    assert B.gconv_problem.N.offset == 8
    assert B.gconv_problem.dil.offset == 76
    assert ctypes.sizeof(B.gconv_options) == 64
    assert B.gconv_options.tile.offset == 24
    assert B.gconv_options.serial_launch.offset == 56


def good(**kw):
    base = dict(ndim=2, N=2, G=4, C=8, K=12, inp=(1, 9, 7), ker=(1, 3, 3), stride=(1, 1, 1),
                pad=(0, 1, 1), dil=(1, 1, 1))
    base.update(kw)
    return B.make_problem(**base)


@pytest.mark.parametrize("bad", [
    dict(C=9), dict(K=10), dict(G=0), dict(N=0), dict(ndim=4), dict(inp=(1, 0, 7)),
    dict(ker=(1, 0, 3)), dict(stride=(1, 0, 1)), dict(dil=(1, 1, 0)), dict(pad=(0, -1, 1)),
    dict(inp=(2, 9, 7)), dict(ker=(3, 3, 3)), dict(pad=(1, 1, 1)), dict(stride=(2, 1, 1)),
    dict(inp=(1, 2, 2), pad=(0, 0, 0)),  # 3x3 window does not fit: empty output
])
def test_invalid_problem_rejected(bad):
    p = good(**bad)
    with pytest.raises(gc.GconvError) as e:
        gc.grouped_conv_out_shape(p)
    assert e.value.status == B.GCONV_ERR_INVALID_ARG
    assert gc.gconv_last_error()


def test_reserved_must_be_zero():
    p = good()
    p.reserved = 1
    with pytest.raises(gc.GconvError):
        gc.grouped_conv_out_shape(p)


def test_null_pointers_rejected_before_launch():
    p = good()
    with pytest.raises(gc.GconvError) as e:
        gc.grouped_conv_fwd(None, 16, None, 32, p, B.GCONV_F32, None)
    assert e.value.status == B.GCONV_ERR_INVALID_ARG
    with pytest.raises(gc.GconvError) as e:
        gc.grouped_conv_fwd(16, 16, None, 32, p, 7, None)
    assert e.value.status == B.GCONV_ERR_UNSUPPORTED


def test_overlapping_output_rejected():
    p = good()
    base = 1 << 20
    with pytest.raises(gc.GconvError) as e:
        gc.grouped_conv_fwd(base, base + (1 << 16), None, base + 64, p, B.GCONV_F32, None)
    assert e.value.status == B.GCONV_ERR_INVALID_ARG
    assert "overlap" in gc.gconv_last_error()


def test_out_shape_matches_oracle(orc):
    rng = np.random.default_rng(5)
    for _ in range(300):
        wl = inputs.random_problem(rng)
        got = gc.grouped_conv_out_shape(gc.problem_of(wl))
        assert got == orc.out_shape(wl), wl


def test_status_strings():
    for s in range(5):
        assert gc.gconv_status_string(s)
    assert "unknown" in gc.gconv_status_string(42)


def test_selector_is_shape_based():
    sel = {wl.name: gc.grouped_conv_select(gc.problem_of(wl), gc.DTYPE_CODES[wl.dtype])
           for wl in inputs.all_workloads()}
    assert sel["mbv2_dw_s1_f16"] == B.KERNEL_DIRECT_DW
    assert sel["mbv2_dw_s2_f16"] == B.KERNEL_DIRECT_DW
    assert sel["sweep_g512_d2_s2_bf16"] == B.KERNEL_DIRECT_DW
    # groups of two channels: the direct kernel at stride 1 and dilation 1 only
    assert sel["sweep_g256_d1_s1_bf16"] == B.KERNEL_DIRECT_DW
    assert sel["sweep_g256_d2_s1_bf16"] == B.KERNEL_IGEMM_TC
    assert sel["sweep_g256_d1_s2_bf16"] == B.KERNEL_IGEMM_TC
    assert sel["grouped2d_f32_smoke"] == B.KERNEL_DIRECT_GENERIC  # fp32 never on tensor cores
    # depthwise with 3 channels breaks 16-byte vectors: generic path
    wl = inputs.by_name("mbv2_dw_s1_f16").with_(G=3)
    assert gc.grouped_conv_select(gc.problem_of(wl), B.GCONV_F16) == B.KERNEL_DIRECT_GENERIC


def test_epilogue_entry_validates():
    with pytest.raises(gc.GconvError) as e:
        gc.gconv_epilogue_apply(None, None, 16, 4, 4, B.GCONV_F16, None)
    assert e.value.status == B.GCONV_ERR_INVALID_ARG
    with pytest.raises(gc.GconvError):
        gc.gconv_epilogue_apply(16, None, 32, 4, 0, B.GCONV_F16, None)


# ---- backward data: host-side logic (nothing is launched on these errors) ----
def test_bwd_data_workspace_size():
    p = good()  # stride 1, pad 1 <= dil*(k-1) = 2: forward-kernel route, transposed weights
    w_bytes = 12 * 9 * 2 * 2  # K * taps * Cg * fp16
    assert gc.grouped_conv_bwd_data_workspace_size(p, B.GCONV_F16) == w_bytes
    assert gc.grouped_conv_bwd_data_workspace_size(p, B.GCONV_F32) == 2 * w_bytes
    assert gc.grouped_conv_bwd_data_workspace_size(good(stride=(1, 2, 2)), B.GCONV_F16) == 0  # direct kernel
    assert gc.grouped_conv_bwd_data_workspace_size(good(ker=(1, 1, 1)), B.GCONV_F16) == 0  # pad > dil*(k-1)
    assert gc.grouped_conv_bwd_data_workspace_size(good(ker=(1, 1, 1), pad=(0, 0, 0)), B.GCONV_F16) == 12 * 2 * 2


def test_bwd_data_workspace_required():
    p = good()
    need = gc.grouped_conv_bwd_data_workspace_size(p, B.GCONV_F16)
    base = 1 << 30
    for ws, nbytes in ((None, 0), (base + (1 << 24), need - 2), (base + (1 << 24) + 8, need)):
        with pytest.raises(gc.GconvError) as e:
            gc.grouped_conv_bwd_data(base, base + (1 << 20), base + (1 << 22), p, B.GCONV_F16, ws, nbytes)
        assert e.value.status == B.GCONV_ERR_INVALID_ARG
        assert "workspace" in gc.gconv_last_error()


def test_bwd_data_overlap_and_forced_route_rejected():
    p = good()
    base = 1 << 30
    with pytest.raises(gc.GconvError) as e:  # dx overlaps dy
        gc.grouped_conv_bwd_data(base, base + (1 << 20), base + 64, p, B.GCONV_F16, base + (1 << 24), 1 << 16)
    assert e.value.status == B.GCONV_ERR_INVALID_ARG and "overlap" in gc.gconv_last_error()
    opt = gc.gconv_options()
    opt.force_kernel = B.KERNEL_IGEMM_TC  # a forward kernel needs the stride-1 route
    with pytest.raises(gc.GconvError) as e:
        gc.grouped_conv_bwd_data_ex(base, base + (1 << 20), base + (1 << 22), good(stride=(1, 2, 2)), B.GCONV_F16,
                                    None, 0, None, opt)
    assert e.value.status == B.GCONV_ERR_UNSUPPORTED


# ---- backward weight: host-side logic (nothing is launched on these errors) ----
def test_bwd_weight_workspace_size():
    """fp32 partials of every dw element for a fixed number of pixel runs:
    a positive multiple of the dw element count, the same for every dtype's
    vector width choice of one shape, and at most 32 MB unless one run
    already needs more."""
    for p in (good(), good(stride=(1, 2, 2)), good(G=4, C=4, K=4),
              B.make_problem(3, 1, 32, 64, 128, (8, 28, 28), (3, 3, 3), (1, 1, 1), (1, 1, 1), (1, 1, 1))):
        E = p.K * p.ker[0] * p.ker[1] * p.ker[2] * (p.C // p.G)
        for dt in (B.GCONV_F16, B.GCONV_BF16, B.GCONV_F32):
            n = gc.grouped_conv_bwd_weight_workspace_size(p, dt)
            assert n > 0 and n % (4 * E) == 0, (n, E)
            assert n <= max(32 << 20, 4 * E)


def test_bwd_weight_argument_errors():
    p = good()
    need = gc.grouped_conv_bwd_weight_workspace_size(p, B.GCONV_F16)
    base = 1 << 30
    for ws, nbytes in ((None, 0), (base + (1 << 26), need - 4), (base + (1 << 26) + 8, need)):
        with pytest.raises(gc.GconvError) as e:
            gc.grouped_conv_bwd_weight(base, base + (1 << 20), base + (1 << 22), p, B.GCONV_F16, ws, nbytes)
        assert e.value.status == B.GCONV_ERR_INVALID_ARG and "workspace" in gc.gconv_last_error()
    with pytest.raises(gc.GconvError) as e:  # dw overlaps x
        gc.grouped_conv_bwd_weight(base, base + (1 << 20), base + 64, p, B.GCONV_F16, base + (1 << 26), need)
    assert e.value.status == B.GCONV_ERR_INVALID_ARG and "overlap" in gc.gconv_last_error()
    with pytest.raises(gc.GconvError) as e:  # NULL dy
        gc.grouped_conv_bwd_weight(base, None, base + (1 << 22), p, B.GCONV_F16, base + (1 << 26), need)
    assert e.value.status == B.GCONV_ERR_INVALID_ARG
    opt = gc.gconv_options()
    opt.force_kernel = B.KERNEL_DIRECT_DW
    with pytest.raises(gc.GconvError) as e:
        gc.grouped_conv_bwd_weight_ex(base, base + (1 << 20), base + (1 << 22), p, B.GCONV_F16,
                                      base + (1 << 26), need, None, opt)
    assert e.value.status == B.GCONV_ERR_UNSUPPORTED


def test_plain_c_program_uses_the_abi(tmp_path):
    """The header is plain C: a C99 program includes it, links libgconv.so and
    calls the host-only entry points (no GPU needed for these)."""
    import shutil
    import subprocess

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    lib = B.load_library()
    libdir = os.path.dirname(lib._name)
    src = tmp_path / "use_abi.c"
    src.write_text(r"""
#include <stdio.h>
#include "gconv.h"
int main(void) {
  gconv_problem p = {0};
  p.ndim = 2; p.N = 32; p.G = 144; p.C = 144; p.K = 144;
  p.in[0] = 1; p.in[1] = 56; p.in[2] = 56;
  p.ker[0] = 1; p.ker[1] = 3; p.ker[2] = 3;
  p.stride[0] = 1; p.stride[1] = 2; p.stride[2] = 2;
  p.pad[0] = 0; p.pad[1] = 1; p.pad[2] = 1;
  p.dil[0] = 1; p.dil[1] = 1; p.dil[2] = 1;
  int32_t out[3], kernel = -1;
  int64_t ws = -1;
  if (grouped_conv_out_shape(&p, out) != GCONV_OK) return 1;
  if (grouped_conv_select(&p, GCONV_F16, &kernel) != GCONV_OK) return 2;
  if (grouped_conv_bwd_data_workspace_size(&p, GCONV_F16, &ws) != GCONV_OK) return 3;
  p.C = 145;
  gconv_status bad = grouped_conv_out_shape(&p, out);
  printf("%d %d %d %d %lld %d %s\n", out[0], out[1], out[2], kernel, (long long)ws, (int)bad,
         gconv_status_string(bad));
  return 0;
}
""")
    exe = tmp_path / "use_abi"
    subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I" + os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                    "-L" + libdir, "-lgconv", "-Wl,-rpath," + libdir], check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    d, h, w, kernel, ws, bad, text = r.stdout.split(maxsplit=6)
    assert (int(d), int(h), int(w)) == (1, 28, 28)
    assert int(kernel) == B.KERNEL_DIRECT_DW
    assert int(ws) == 0  # stride 2: the direct backward kernel needs no workspace
    assert int(bad) == B.GCONV_ERR_INVALID_ARG and text.strip() == "invalid argument"
