"""Pins of the oracle's fused epilogue (oracle/epilogue.py) against facts it
does not compute itself: a hand-worked example (tests/golden), and relations
the definition fixes between outputs -- ReLU applied after the bias, beta = 0
never reading C, alpha = 0 and beta = 1 returning C exactly, K = 0 leaving
act(beta C + bias), and linearity in alpha.  The last test plants plausible
mistakes in copies of the epilogue and checks that each fails a pin.
"""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import epilogue
import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden", "epilogue_example.json")
FMTS = ["f32", "f16", "bf16"]


def bits_of(values, fmt):
    values = np.asarray(values, dtype=np.float64)
    assert np.array_equal(wl.round_to_format(values, fmt), values)
    return np.ascontiguousarray(wl.encode(values, fmt))


def product(A, B, fmt):
    A, B = np.asarray(A, dtype=np.float64), np.asarray(B, dtype=np.float64)
    D, _ = oracle.gemm(bits_of(A, fmt), bits_of(B, fmt), fmt, A.shape[0], B.shape[1], A.shape[1])
    return D


def random_case(seed, M=6, N=7, K=9):
    A = wl.round_to_format(wl.uniform_pm1(seed, M * K), "bf16").reshape(M, K)
    B = wl.round_to_format(wl.uniform_pm1(seed + 1, K * N), "bf16").reshape(K, N)
    Cin = wl.round_to_format(wl.uniform_pm1(seed + 2, M * N), "bf16").reshape(M, N)
    bias = wl.round_to_format(wl.uniform_pm1(seed + 3, N), "bf16")
    return product(A, B, "bf16"), Cin, bias


# ---------------------------------------------------------------- pin suite
# Each pin takes an epilogue implementation (the oracle's, or a planted
# mutant with the same signature) and raises AssertionError on failure.

def pin_hand_example(apply):
    g = json.load(open(GOLDEN))
    for fmt in FMTS:
        D = product(g["A"], g["B"], fmt)
        assert np.array_equal(D, np.array(g["D"], dtype=np.float64)), fmt
        for act in ("none", "relu"):
            out = apply(D, np.array(g["Cin"], dtype=np.float64), g["alpha"], g["beta"],
                        np.array(g["bias"], dtype=np.float64), act)
            assert np.array_equal(out, np.array(g[f"out_{act}"])), (fmt, act)


def pin_relu_after_bias(apply):
    D, Cin, bias = random_case(11)
    z = apply(D, Cin, 1.5, -0.5, bias, "none")
    r = apply(D, Cin, 1.5, -0.5, bias, "relu")
    assert np.array_equal(r, np.where(z < 0, 0.0, z))
    assert (z < 0).any() and (z > 0).any()  # the case exercises both sides


def pin_beta_zero_never_reads_c(apply):
    D, Cin, bias = random_case(12)
    poisoned = np.full_like(Cin, np.nan)
    a = apply(D, poisoned, 2.0, 0.0, bias, "none")
    b = apply(D, None, 2.0, 0.0, bias, "none")
    assert np.isfinite(a).all() and np.array_equal(a, b)


def pin_alpha_zero_returns_c(apply):
    D, Cin, _ = random_case(13)
    assert np.array_equal(apply(D, Cin, 0.0, 1.0, None, "none"), Cin)


def pin_empty_sum(apply):
    _, Cin, bias = random_case(14)
    D = np.zeros_like(Cin)  # K = 0: the product is the empty sum
    out = apply(D, Cin, 3.0, 0.25, bias, "none")
    # beta = 1/4 and bias values in bf16 make every term exact in float64
    for i in range(Cin.shape[0]):
        for j in range(Cin.shape[1]):
            assert out[i, j] == 0.25 * Cin[i, j] + bias[j]
    relu = apply(D, Cin, 3.0, 0.25, bias, "relu")
    assert (relu >= 0).all()


def pin_linear_in_alpha(apply):
    D, Cin, _ = random_case(15)
    a3 = apply(D, Cin, 3.0, 0.0, None, "none")
    a1 = apply(D, Cin, 1.0, 0.0, None, "none")
    assert np.allclose(a3 - a1, 2.0 * D, rtol=0, atol=1e-12)
    assert np.array_equal(apply(D, Cin, 1.0, 0.0, None, "none"), D)


def pin_nan_propagates_through_relu(apply):
    D = np.array([[np.nan, -1.0, 2.0]])
    out = apply(D, None, 1.0, 0.0, None, "relu")
    assert np.isnan(out[0, 0]) and out[0, 1] == 0.0 and out[0, 2] == 2.0


PINS = [pin_hand_example, pin_relu_after_bias, pin_beta_zero_never_reads_c, pin_alpha_zero_returns_c,
        pin_empty_sum, pin_linear_in_alpha, pin_nan_propagates_through_relu]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_epilogue_pin(pin):
    pin(epilogue.apply)


def test_magnitude_bounds_every_term():
    D, Cin, bias = random_case(16)
    S = np.abs(D) + 1.0
    T = epilogue.magnitude(S, Cin, -2.0, 0.5, bias)
    assert (T >= 2.0 * S).all() and (T >= np.abs(0.5 * Cin)).all() and (T >= np.abs(bias)[None, :]).all()


# ------------------------------------------------------- planted mistakes

def _mutant(kind):
    def apply(D, Cin=None, alpha=1.0, beta=0.0, bias=None, act="none"):
        D = np.asarray(D, dtype=np.float64)
        M, N = D.shape
        b = np.zeros(N) if bias is None else np.asarray(bias, dtype=np.float64)
        c = np.zeros((M, N)) if (beta == 0.0 or Cin is None) else np.asarray(Cin, dtype=np.float64)
        if kind == "relu_before_bias":
            Z = alpha * D + beta * c
            if act == "relu":
                Z = np.where(Z < 0, 0.0, Z)
            return Z + b[None, :]
        if kind == "bias_per_row":
            bb = np.resize(b, M)[:, None]
            Z = alpha * D + beta * c + bb
        elif kind == "beta_on_product":
            Z = alpha * D + beta * D + b[None, :]
        elif kind == "alpha_scales_bias":
            Z = alpha * (D + b[None, :]) + beta * c
        elif kind == "beta_sign":
            Z = alpha * D - beta * c + b[None, :]
        elif kind == "reads_c_when_beta_zero":
            cc = np.zeros((M, N)) if Cin is None else np.asarray(Cin, dtype=np.float64)
            Z = alpha * D + (beta if beta != 0 else 1e-300) * cc + b[None, :]
        elif kind == "relu_drops_nan":
            Z = alpha * D + beta * c + b[None, :]
            return np.fmax(Z, 0.0) if act == "relu" else Z
        elif kind == "clamps_positive":
            Z = alpha * D + beta * c + b[None, :]
            return np.where(Z > 0, 0.0, Z) if act == "relu" else Z
        else:
            raise ValueError(kind)
        if act == "relu":
            Z = np.where(Z < 0, 0.0, Z)
        return Z
    return apply


MUTANTS = ["relu_before_bias", "bias_per_row", "beta_on_product", "alpha_scales_bias", "beta_sign",
           "reads_c_when_beta_zero", "relu_drops_nan", "clamps_positive"]


@pytest.mark.parametrize("kind", MUTANTS)
def test_every_planted_mistake_fails_a_pin(kind):
    failures = 0
    for pin in PINS:
        try:
            pin(_mutant(kind))
        except AssertionError:
            failures += 1
    assert failures > 0, f"mutant {kind} passes every pin"
