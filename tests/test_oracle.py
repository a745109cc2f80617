"""The CPU oracle against facts that do not come from the oracle itself."""
import json
import os

import numpy as np
import pytest

import oracle_pins as pins

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_printed_3d_case_geometry(orc):
    """The TileOps review prints 802,816 outputs and 54 MACs each for its 3D case."""
    g = json.load(open(os.path.join(GOLDEN, "resnext3d_n1_counts.json")))
    pr = g["problem"]
    p = pins.wl(3, pr["N"], pr["G"], pr["Cg"], pr["Kg"], pr["in"], pr["ker"], pr["stride"],
                pr["pad"], pr["dil"])
    Do, Ho, Wo = orc.out_shape(p)
    assert Do * Ho * Wo * p.N * p.K == g["printed"]["output_elements"]
    assert p.Cg * p.taps == g["printed"]["macs_per_output"]


def test_oracle_rejects_empty(orc):
    p = pins.wl(2, 1, 1, 1, 1, (2, 2), (5, 5), (1, 1), (0, 0), (1, 1))
    with pytest.raises(ValueError):
        orc.forward(p, np.zeros(p.x_shape()), np.zeros(p.w_shape()), None)
    p = pins.wl(2, 1, 1, 1, 1, (4, 4), (3, 3), (1, 1), (1, 1), (1, 1))
    with pytest.raises(ValueError):
        orc.points(p, np.zeros(p.x_shape()), np.zeros(p.w_shape()), None, [10**6])
