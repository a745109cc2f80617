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
