"""Plant mistakes in copies of the oracle and check that the pins catch each.

Every mutant is a textual edit of ``oracle/oracle.c`` compiled into a
temporary library; the real oracle is untouched.  A mutant that passes every
pin would mean the pins cannot tell that mistake from the definition.
"""
import os

import pytest

import oracle
import oracle_pins as pins

MUTANTS = {
    "flip_kernel_y": ("* Y + yy) * X + xx) * Cg", "* Y + (Y - 1 - yy)) * X + xx) * Cg"),
    "flip_kernel_x": ("* Y + yy) * X + xx) * Cg", "* Y + yy) * X + (X - 1 - xx)) * Cg"),
    "pad_sign": ("oh * st[1] - pd[1]", "oh * st[1] + pd[1]"),
    "drop_dilation_w": ("xx * dl[2]", "xx"),
    "group_channel_uses_kg": ("* C + g * Cg)", "* C + g * Kg)"),
    "drop_bias": ("acc += bias[g * Kg + k];", ";"),
    "bias_index_transposed": ("bias[g * Kg + k]", "bias[k * G + g]"),
    "extent_ceil": ("return room / s + 1;", "return (room + s - 1) / s + 1;"),
    "stride_axis_swap": ("ow * st[2]", "ow * st[1]"),
    "weight_k_cg_swap": ("(((g * Kg + k) * Z + z)", "(((g * Kg + (k % Kg)) * Z + z) + 0 * Cg"),
    "skip_first_depth_tap": ("for (long z = 0; z < Z; ++z)", "for (long z = (Z > 1); z < Z; ++z)"),
    "padding_not_zero": ("if (iw < 0 || iw >= W)\n                    continue;",
                         "if (iw < 0 || iw >= W) { acc += 1e-3; continue; }"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert old in src, f"mutation anchor for {name} not found"
    mutated = src.replace(old, new, 1)
    if name == "weight_k_cg_swap":
        # transposed operand: index the weight as [G][Cg][..][Kg] instead of [G][Kg][..][Cg]
        mutated = src.replace(
            "const double *wp = w + ((((g * Kg + k) * Z + z) * Y + yy) * X + xx) * Cg;\n"
            "                for (long cg = 0; cg < Cg; ++cg)\n"
            "                    acc += xp[cg] * wp[cg];",
            "for (long cg = 0; cg < Cg; ++cg)\n"
            "                    acc += xp[cg] * w[((((g * Cg + cg) * Z + z) * Y + yy) * X + xx) * Kg + k];")
        assert mutated != src
    cfile = tmp_path / "mut.c"
    cfile.write_text(mutated)
    lib = oracle.compile_source(str(cfile), str(tmp_path / "libmut.so"), openmp=False)
    orc = oracle.load(lib)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
