"""The oracle still reproduces its committed golden fixtures (CPU only).

The fixtures under tests/golden/ were written by tests/golden/make_golden.py,
which calls only the oracle and the seeded inputs.  A failure here means the
oracle's arithmetic (or the input recipe) changed: such a change must name the
page passage, or the reading of it, that justifies it.
"""
import os

import numpy as np

from tests.golden import make_golden

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read(name):
    rows = []
    shape = None
    with open(os.path.join(HERE, name)) as f:
        for line in f:
            if line.startswith("# shape"):
                shape = tuple(int(v) for v in line.split()[2:])
            elif not line.startswith("#"):
                rows.append([int(v, 16) for v in line.split()])
    return np.array(rows, dtype=np.uint16).reshape(shape)


def test_tiny_delta_golden(oracle):
    _, out, err = make_golden.tiny_delta()
    assert err == 0
    assert np.array_equal(out, read("tiny_delta_oracle.txt"))


def test_tiny_moe_golden(oracle):
    for mode, shared in (("regular", False), ("shared", True)):
        _, out, err = make_golden.tiny_moe(shared)
        assert np.array_equal(out, read(f"tiny_moe_{mode}_oracle.txt"))


def test_tiny_moe_in_place_golden(oracle):
    _, y, err = make_golden.tiny_w13()
    assert err == 0
    assert np.array_equal(y, read("tiny_moe_w13_oracle.txt"))
    _, y, err = make_golden.tiny_w2()
    assert err == 0
    assert np.array_equal(y, read("tiny_moe_w2_oracle.txt"))
