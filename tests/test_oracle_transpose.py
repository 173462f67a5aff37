"""Pins of the oracle's transpose (oracle/transpose.py): a hand-worked example
with row padding on both sides (tests/golden), index-encoded matrices whose
transpose has a closed form, the involution T(T(X)) = X, and padding columns
of the output left alone.  Planted mistakes each fail a pin."""
import json
import os

import numpy as np
import pytest

from oracle import transpose as ot

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden", "transpose_example.json")


def pin_hand_example(tr):
    g = json.load(open(GOLDEN))
    src = np.array(g["in"], dtype=np.uint32)
    out = tr(src, g["rows"], g["cols"], None, g["ld_out"])
    assert np.array_equal(out, np.array(g["out"], dtype=np.uint32))


def pin_index_encoding(tr):
    # value = i * 1000 + j in row i, column j, so out[j][i] must read i * 1000 + j
    for rows, cols in [(1, 1), (1, 7), (7, 1), (33, 65), (64, 64), (70, 129)]:
        src = (np.arange(rows)[:, None] * 1000 + np.arange(cols)[None, :]).astype(np.uint32)
        out = tr(src, rows, cols, None, None)
        for j in range(cols):
            for i in range(rows):
                assert out[j, i] == i * 1000 + j, (rows, cols, i, j)


def pin_involution(tr):
    rng = np.random.default_rng(7)
    for rows, cols in [(5, 9), (32, 32), (31, 47)]:
        x = rng.integers(0, 2 ** 16, size=(rows, cols), dtype=np.uint16)
        assert np.array_equal(tr(tr(x, rows, cols, None, None), cols, rows, None, None), x)


def pin_output_padding_untouched(tr):
    src = np.arange(12, dtype=np.uint16).reshape(3, 4)
    out = np.full((4, 6), 0xBEEF, dtype=np.uint16)
    tr(src, 3, 4, out, 6)
    assert np.all(out[:, 3:] == 0xBEEF)


PINS = [pin_hand_example, pin_index_encoding, pin_involution, pin_output_padding_untouched]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_transpose_pin(pin):
    pin(ot.transpose)


def _mutant(kind):
    def tr(src, rows, cols, out=None, ld_out=None):
        ld_out = rows if ld_out is None else ld_out
        if out is None:
            out = np.zeros((cols, ld_out), dtype=src.dtype)
        if kind == "copy_not_transpose":
            for i in range(min(rows, cols)):
                out[i, :min(rows, cols)] = src[i, :min(rows, cols)]
        elif kind == "off_by_one_column":
            for j in range(cols):
                out[j, :rows] = src[:rows, min(j + 1, cols - 1)]
        elif kind == "writes_padding":
            out[:, :] = 0
            for j in range(cols):
                out[j, :rows] = src[:rows, j]
        elif kind == "reads_padding":
            for j in range(cols):
                out[j, :rows] = src[:rows, src.shape[1] - cols + j]
        else:
            raise ValueError(kind)
        return out
    return tr


@pytest.mark.parametrize("kind", ["copy_not_transpose", "off_by_one_column", "writes_padding", "reads_padding"])
def test_every_planted_mistake_fails_a_pin(kind):
    failures = 0
    for pin in PINS:
        try:
            pin(_mutant(kind))
        except (AssertionError, IndexError, ValueError):
            failures += 1
    assert failures > 0, f"mutant {kind} passes every pin"
