"""Backward-data oracle against its pins (adjoint identity with the pinned
forward oracle; torch's conv-input gradient), and mutants of its source
that the pins must catch."""
import pytest

import oracle
import oracle_pins as pins


@pytest.mark.parametrize("pin", pins.BWD_PINS, ids=lambda f: f.__name__)
def test_bwd_pin(orc, pin):
    pin(orc)


# textual edits of the backward-data function only (anchors unique to it)
BWD_MUTANTS = {
    "bwd_pad_sign": ("const long ih = oh * st[1] - pd[1]", "const long ih = oh * st[1] + pd[1]"),
    "bwd_drop_dilation_w": ("const long iw = ow * st[2] - pd[2] + xx * dl[2];",
                            "const long iw = ow * st[2] - pd[2] + xx;"),
    "bwd_dy_channel_transposed": ("const double d = dy[(((n * Do + od) * Ho + oh) * Wo + ow) * K + g * Kg + k];",
                                  "const double d = dy[(((n * Do + od) * Ho + oh) * Wo + ow) * K + k * G + g];"),
    "bwd_dx_group_uses_kg": ("* W + iw) * C + g * Cg);\n                                    const double *wp",
                             "* W + iw) * C + g * Kg);\n                                    const double *wp"),
    "bwd_kernel_flipped": ("const double *wp = w + ((((g * Kg + k) * Z + z) * Y + yy) * X + xx) * Cg;\n"
                           "                                    for",
                           "const double *wp = w + ((((g * Kg + k) * Z + z) * Y + (Y - 1 - yy)) * X + xx) * Cg;\n"
                           "                                    for"),
    "bwd_stride_ignored": ("const long id = od * st[0] - pd[0] + z * dl[0];\n"
                           "                            if (id < 0 || id >= D)",
                           "const long id = od * st[0] - pd[0] + z * dl[0];\n"
                           "                            if (id < 0 || id >= D || (st[1] > 1 && oh % 2))"),
}


@pytest.mark.parametrize("name", sorted(BWD_MUTANTS))
def test_bwd_mutant_is_caught(tmp_path, name):
    old, new = BWD_MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    cfile = tmp_path / "mut.c"
    cfile.write_text(src.replace(old, new))
    orc = oracle.load(oracle.compile_source(str(cfile), str(tmp_path / "libmut.so"), openmp=False))
    caught = []
    for pin in pins.BWD_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"


def test_stride1_backward_data_is_a_forward_pass(orc):
    """The identity the library's stride-1 backward-data route runs on, checked
    with the pinned oracles alone: for stride 1 and pad <= d*(k-1), backward
    data equals the forward convolution of dy with per-group transposed,
    spatially flipped weights wt[g, c, t', k] = w[g, k, flip(t'), c], Cg and
    Kg swapped and padding d*(k-1) - pad."""
    import numpy as np

    from depthwise_convolution_forward_gb300 import inputs

    rng = np.random.default_rng(11)
    checked = 0
    for _ in range(400):
        wl = inputs.random_problem(rng)
        if any(s != 1 for s in wl.stride) or any(p > d * (k - 1) for p, d, k in zip(wl.pad, wl.dil, wl.ker)):
            continue
        w = rng.normal(size=wl.w_shape())
        out = orc.out_shape(wl)
        dy = rng.uniform(-1, 1, size=(wl.N, *out, wl.G, wl.Kg))
        ref = orc.bwd_data(wl, dy, w).reshape(wl.N, *wl.inp, wl.G, wl.Cg)
        w6 = w.reshape(wl.G, wl.Kg, *wl.ker, wl.Cg)
        wt = np.ascontiguousarray(np.transpose(w6[:, :, ::-1, ::-1, ::-1, :], (0, 5, 2, 3, 4, 1)))
        f = wl.with_(Cg=wl.Kg, Kg=wl.Cg, inp=tuple(out), bias=False,
                     pad=tuple(d * (k - 1) - p for p, d, k in zip(wl.pad, wl.dil, wl.ker)))
        assert orc.out_shape(f) == tuple(wl.inp)
        got = orc.forward(f, dy, wt, None).reshape(ref.shape)
        assert np.allclose(got, ref, rtol=1e-12, atol=1e-12), wl
        checked += 1
    assert checked >= 20
