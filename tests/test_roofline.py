"""The benchmark's work and traffic formulas against the numbers the TileOps
review prints for its 3D grouped case (tests/golden/resnext3d_n1_counts.json)."""
import json
import os

import depthwise_convolution_forward_gb300 as gc
from depthwise_convolution_forward_gb300 import build, inputs, roofline

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "resnext3d_n1_counts.json")


def test_printed_3d_counts():
    build.build()
    g = json.load(open(GOLDEN))["printed"]
    wl = inputs.by_name("resnext3d_n1_f16")
    out = gc.grouped_conv_out_shape(gc.problem_of(wl))
    assert roofline.outputs(wl, out) == g["output_elements"]
    assert wl.Cg * wl.taps == g["macs_per_output"]
    assert round(roofline.flops(wl, out) / 1e6, 1) == g["mflop_approx"]
    tb = roofline.tensor_bytes(wl, out)
    assert round(tb["x"] / 1e6, 1) == g["input_mb_approx"]
    assert round(tb["y"] / 1e6, 1) == g["output_mb_approx"]
    assert round(tb["w"] / 1e3) == g["weight_kb_approx"]
    assert round((tb["x"] + tb["y"] + tb["w"]) / 1e6, 1) == g["io_mb_approx"]


def test_flops_scale_with_per_group_channels():
    wl = inputs.by_name("sweep_g8_d1_s1_bf16")
    out = gc.grouped_conv_out_shape(gc.problem_of(wl))
    f8 = roofline.flops(wl, out)
    f512 = roofline.flops(inputs.by_name("sweep_g512_d1_s1_bf16"), out)
    assert f8 == 64 * f512


def test_input_bytes_count_touched_positions():
    """Stride 2 with dilation 2 and pad 2 reads only the even rows and
    columns: a quarter of x; stride 2 with pad 1 (3x3) and stride 1 read all."""
    for name, frac in (("sweep_g64_d2_s2_bf16", 0.25), ("sweep_g64_d1_s2_bf16", 1.0), ("mbv2_dw_s2_f16", 1.0),
                       ("sweep_g8_d2_s1_bf16", 1.0)):
        wl = inputs.by_name(name)
        out = gc.grouped_conv_out_shape(gc.problem_of(wl))
        full = wl.N * wl.inp[0] * wl.inp[1] * wl.inp[2] * wl.C * roofline.ES[wl.dtype]
        assert roofline.tensor_bytes(wl, out)["x"] == full * frac, name
    # brute force on a small odd case: positions o*s - p + t*d inside the input
    assert roofline.touched(7, 3, 3, 3, 0, 1) == 7 - 0  # windows [0,3), [3,6), [6,9) -> 0..6
    assert roofline.touched(7, 2, 2, 3, 0, 2) == 4      # {0, 2} and {3, 5}


def test_backward_data_bytes_count_all_of_dx():
    """Backward data writes every dx position (zeros where no output
    reaches), so its x term is the whole input even when the forward pass
    touches only a quarter of it."""
    wl = inputs.by_name("sweep_g8_d2_s2_bf16")
    out = [(wl.inp[i] + 2 * wl.pad[i] - wl.dil[i] * (wl.ker[i] - 1) - 1) // wl.stride[i] + 1 for i in range(3)]
    fwd = roofline.tensor_bytes(wl, out)
    bwd = roofline.tensor_bytes(wl, out, "bwd_data")
    full = wl.N * wl.inp[0] * wl.inp[1] * wl.inp[2] * wl.C * 2
    assert bwd["x"] == full and fwd["x"] == full // 4
    assert roofline.algorithmic_bytes(wl, out, "bwd_weight") == roofline.algorithmic_bytes(wl, out)



def test_fused_block_accounting():
    """Fused depthwise + 1x1 projection on the MobileNetV2 stride-1 layer
    (N=32, C=144, 56x56, K=24, f16), every tensor once, worked by hand."""
    wl = inputs.by_name("mbv2_dw_s1_f16")
    out = (1, 56, 56)
    pix = 32 * 56 * 56
    b = roofline.fused_block_bytes(wl, out, 24)
    assert b == {"x": pix * 144 * 2, "w_dw": 144 * 9 * 2, "b_dw": 144 * 2, "w_pw": 24 * 144 * 2, "b_pw": 24 * 2,
                 "y": pix * 24 * 2, "h_saved": 2 * pix * 144 * 2}
    assert roofline.fused_block_flops(wl, out, 24) == 2 * pix * 144 * 9 + 2 * pix * 144 * 24
    # stride 2, pad 1: every input row and column is read; y at 28 x 28
    w2 = inputs.by_name("mbv2_dw_s2_f16")
    b2 = roofline.fused_block_bytes(w2, (1, 28, 28), 32)
    assert b2["x"] == pix * 144 * 2 and b2["y"] == 32 * 28 * 28 * 32 * 2
