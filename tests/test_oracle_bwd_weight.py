"""Backward-weight oracle against its pins (the gradient identity with the
pinned forward oracle; torch's conv-weight gradient), and mutants of its
source that the pins must catch.  The GPU kernel for this operation is not
built yet: this is its oracle, pinned first."""
import pytest

import oracle
import oracle_pins as pins


@pytest.mark.parametrize("pin", pins.BWD_WEIGHT_PINS, ids=lambda f: f.__name__)
def test_bwd_weight_pin(orc, pin):
    pin(orc)


# textual edits of the backward-weight function only (anchors unique to it)
BWD_WEIGHT_MUTANTS = {
    "bww_pad_sign": ("const long hi = oh * st[1] - pd[1] + yy * dl[1];",
                     "const long hi = oh * st[1] + pd[1] + yy * dl[1];"),
    "bww_drop_dilation_w": ("const long wi = ow * st[2] - pd[2] + xx * dl[2];",
                            "const long wi = ow * st[2] - pd[2] + xx;"),
    "bww_dy_channel_transposed": ("* Wo + ow) * K + g * Kg + k];\n                                    const double *xp",
                                  "* Wo + ow) * K + k * G + g];\n                                    const double *xp"),
    "bww_x_group_uses_kg": ("* W + wi) * C + g * Cg);", "* W + wi) * C + g * Kg);"),
    "bww_filter_flipped": ("double *wp = dw + ((((g * Kg + k) * Z + z) * Y + yy) * X + xx) * Cg;",
                           "double *wp = dw + ((((g * Kg + k) * Z + z) * Y + (Y - 1 - yy)) * X + xx) * Cg;"),
    "bww_first_image_only": ("for (long n = 0; n < N; ++n)\n                        for (long od",
                             "for (long n = 0; n < 1; ++n)\n                        for (long od"),
}


@pytest.mark.parametrize("name", sorted(BWD_WEIGHT_MUTANTS))
def test_bwd_weight_mutant_is_caught(tmp_path, name):
    old, new = BWD_WEIGHT_MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    cfile = tmp_path / "mut.c"
    cfile.write_text(src.replace(old, new))
    orc = oracle.load(oracle.compile_source(str(cfile), str(tmp_path / "libmut.so"), openmp=False))
    caught = []
    for pin in pins.BWD_WEIGHT_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
