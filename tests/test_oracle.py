"""Pins of the CPU oracle against facts it does not compute itself.

The oracle restates the definition C[i][j] = sum_k A[i][k] B[k][j] ("CUDA tile",
section 2.1).  Each pin below is a fact fixed by the mathematics or by a
library routine: exact integer products (numpy int64 matmul), the all-ones
product (C = K), identity and permutation matrices, the transpose identity
(AB)^T = B^T A^T, rank-1 outer products, and the correctly rounded exact sum
(math.fsum) within the oracle's error bound K * 2^-53 * S.  The last test
plants mistakes in a copy of the oracle source and checks that every mutant
fails at least one pin.
"""
import json
import math
import os
import shutil
import subprocess
import sys
import tempfile

import numpy as np
import pytest

import oracle
import workloads as wl

FMTS = ["f32", "f16", "bf16"]
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def bits_of(values: np.ndarray, fmt: str) -> np.ndarray:
    r = wl.round_to_format(values, fmt)
    assert np.array_equal(r, values), "pin inputs must be exact in the storage format"
    return np.ascontiguousarray(wl.encode(values, fmt))


# ---------------------------------------------------------------- pin suite
# Each pin takes the loaded oracle library and raises AssertionError on failure.

def pin_integer_brute_force(lib):
    for n in range(2, 9):
        for fmt in FMTS:
            A = wl.small_integer_matrix(n, n + 1, seed=100 + n)
            B = wl.small_integer_matrix(n + 1, n - 1, seed=200 + n)
            want = np.matmul(A.astype(np.int64), B.astype(np.int64)).astype(np.float64)
            C, S = oracle.gemm(bits_of(A, fmt), bits_of(B, fmt), fmt, n, n - 1, n + 1, lib=lib)
            assert np.array_equal(C, want), (n, fmt)
            want_s = np.matmul(np.abs(A).astype(np.int64), np.abs(B).astype(np.int64)).astype(np.float64)
            assert np.array_equal(S, want_s), (n, fmt)


def pin_all_ones(lib):
    for fmt in FMTS:
        for (M, N, K) in [(3, 5, 7), (8, 2, 64), (1, 1, 1)]:
            A = np.ones((M, K))
            B = np.ones((K, N))
            C, S = oracle.gemm(bits_of(A, fmt), bits_of(B, fmt), fmt, M, N, K, lib=lib)
            assert np.all(C == K) and np.all(S == K), (fmt, M, N, K)


def pin_identity_and_permutation(lib):
    rng_vals = wl.round_to_format(wl.uniform_pm1(77, 6 * 9), "bf16").reshape(6, 9)
    for fmt in FMTS:
        X = wl.round_to_format(rng_vals, fmt)
        I6, I9 = np.eye(6), np.eye(9)
        C, _ = oracle.gemm(bits_of(I6, fmt), bits_of(X, fmt), fmt, 6, 9, 6, lib=lib)
        assert np.array_equal(C, X), fmt
        C, _ = oracle.gemm(bits_of(X, fmt), bits_of(I9, fmt), fmt, 6, 9, 9, lib=lib)
        assert np.array_equal(C, X), fmt
        pr = np.array([3, 0, 5, 1, 4, 2])
        pc = np.array([8, 2, 0, 7, 1, 6, 3, 5, 4])
        P = I6[pr]                      # (P X)[r] = X[pr[r]]
        C, _ = oracle.gemm(bits_of(P, fmt), bits_of(X, fmt), fmt, 6, 9, 6, lib=lib)
        assert np.array_equal(C, X[pr]), fmt
        Q = I9[:, pc]                   # (X Q)[:, c] = X[:, pc[c]]
        C, _ = oracle.gemm(bits_of(X, fmt), bits_of(Q, fmt), fmt, 6, 9, 9, lib=lib)
        assert np.array_equal(C, X[:, pc]), fmt


def pin_transpose_identity(lib):
    M, N, K = 5, 7, 11
    for fmt in FMTS:
        A = wl.round_to_format(wl.uniform_pm1(31, M * K), fmt).reshape(M, K)
        B = wl.round_to_format(wl.uniform_pm1(32, K * N), fmt).reshape(K, N)
        C, S = oracle.gemm(bits_of(A, fmt), bits_of(B, fmt), fmt, M, N, K, lib=lib)
        Ct, St = oracle.gemm(bits_of(np.ascontiguousarray(B.T), fmt), bits_of(np.ascontiguousarray(A.T), fmt),
                             fmt, N, M, K, lib=lib)
        assert np.array_equal(C.T, Ct) and np.array_equal(S.T, St), fmt


def pin_rank_one(lib):
    for fmt in FMTS:
        u = wl.round_to_format(wl.uniform_pm1(41, 9), fmt).reshape(9, 1)
        v = wl.round_to_format(wl.uniform_pm1(42, 6), fmt).reshape(1, 6)
        C, S = oracle.gemm(bits_of(u, fmt), bits_of(v, fmt), fmt, 9, 6, 1, lib=lib)
        assert np.array_equal(C, u * v) and np.array_equal(S, np.abs(u * v)), fmt


def pin_exact_sum_bound(lib):
    """Random values: |C - fsum| <= K 2^-53 S and S = fsum of |terms| within the same bound."""
    M, N, K = 6, 5, 300
    for fmt in FMTS:
        A = wl.round_to_format(wl.uniform_pm1(51, M * K), fmt).reshape(M, K)
        B = wl.round_to_format(wl.normal01(52, K * N), fmt).reshape(K, N)
        C, S = oracle.gemm(bits_of(A, fmt), bits_of(B, fmt), fmt, M, N, K, lib=lib)
        for i in range(M):
            for j in range(N):
                terms = [A[i, k] * B[k, j] for k in range(K)]
                exact = math.fsum(terms)
                sabs = math.fsum(abs(t) for t in terms)
                assert abs(C[i, j] - exact) <= K * 2.0 ** -53 * sabs, (fmt, i, j)
                assert abs(S[i, j] - sabs) <= K * 2.0 ** -53 * sabs, (fmt, i, j)


def pin_decode_vectors(lib):
    f16 = {0x3C00: 1.0, 0xC000: -2.0, 0x7BFF: 65504.0, 0x0001: 2.0 ** -24, 0x0400: 2.0 ** -14,
           0x3555: (1 + 0x155 / 1024) * 0.25, 0x7C00: math.inf, 0x8000: -0.0}
    bf16 = {0x3F80: 1.0, 0xC040: -3.0, 0x7F7F: (2 - 2 ** -7) * 2.0 ** 127, 0x0001: 2.0 ** -133,
            0x3C00: 2.0 ** -7, 0x4049: 3.140625, 0xFF80: -math.inf}
    f32 = {0x3F800000: 1.0, 0x00000001: 2.0 ** -149, 0x7F7FFFFF: (2 - 2 ** -23) * 2.0 ** 127,
           0x40490FDB: 3.1415927410125732}
    for fmt, table, dt in (("f16", f16, np.uint16), ("bf16", bf16, np.uint16), ("f32", f32, np.uint32)):
        bits = np.array(list(table.keys()), dtype=dt).reshape(1, -1)
        got = oracle.decode(bits, fmt, lib=lib)[0]
        want = np.array(list(table.values()))
        assert np.array_equal(got, want), (fmt, got, want)
        assert np.array_equal(np.signbit(got), np.signbit(want)), fmt


def pin_leading_dimension(lib):
    """Padding columns hold NaN; the oracle must read only the logical matrix."""
    M, N, K = 4, 3, 5
    for fmt in FMTS:
        A = wl.small_integer_matrix(M, K, seed=61)
        B = wl.small_integer_matrix(K, N, seed=62)
        nan = {"f32": 0x7FC00000, "f16": 0x7E00, "bf16": 0x7FC0}[fmt]
        Ab = np.full((M, K + 3), nan, dtype=np.uint32 if fmt == "f32" else np.uint16)
        Bb = np.full((K, N + 2), nan, dtype=Ab.dtype)
        Ab[:, :K] = bits_of(A, fmt)
        Bb[:, :N] = bits_of(B, fmt)
        C, _ = oracle.gemm(Ab, Bb, fmt, M, N, K, lib=lib)
        assert np.array_equal(C, (A.astype(np.int64) @ B.astype(np.int64)).astype(float)), fmt


def pin_empty_k(lib):
    A = np.zeros((3, 1), dtype=np.uint16)
    B = np.zeros((1, 4), dtype=np.uint16)
    C, S = oracle.gemm(A, B, "bf16", 3, 4, 0, lib=lib)
    assert np.all(C == 0) and np.all(S == 0) and not np.any(np.signbit(C))


PINS = [pin_integer_brute_force, pin_all_ones, pin_identity_and_permutation, pin_transpose_identity,
        pin_rank_one, pin_exact_sum_bound, pin_decode_vectors, pin_leading_dimension, pin_empty_k]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(oracle.load())


# ------------------------------------------------------- properties of the oracle

def test_thread_count_invariance():
    w = wl.Workload("t", 37, 29, 45, wl.BF16, "uniform", 9)
    A, B = wl.make_inputs(w)
    C1, S1 = oracle.gemm(A, B, "bf16", w.M, w.N, w.K, threads=1)
    C7, S7 = oracle.gemm(A, B, "bf16", w.M, w.N, w.K, threads=7)
    assert np.array_equal(C1, C7) and np.array_equal(S1, S7)


def test_entries_match_full_product():
    w = wl.Workload("t", 33, 41, 70, wl.F16, "normal", 8)
    A, B = wl.make_inputs(w, lda=75, ldb=44)
    C, S = oracle.gemm(A, B, "f16", w.M, w.N, w.K)
    rows = np.array([0, 32, 17, 5])
    cols = np.array([40, 0, 13, 39])
    c, s = oracle.entries(A, B, "f16", w.K, rows, cols)
    assert np.array_equal(c, C[rows, cols]) and np.array_equal(s, S[rows, cols])


def test_blocked_variant_agrees():
    w = wl.Workload("t", 70, 300, 260, wl.BF16, "uniform", 7)
    A, B = wl.make_inputs(w, ldb=304)
    C, S = oracle.gemm(A, B, "bf16", w.M, w.N, w.K)
    Cb = oracle.gemm_blocked(A, B, "bf16", w.M, w.N, w.K, threads=3)
    assert np.all(np.abs(Cb - C) <= 2.0 ** -40 * S)


def test_decode_agrees_with_generator_encoding():
    for fmt in FMTS:
        x = wl.round_to_format(wl.normal01(5, 1000) * 3.0, fmt)
        bits = wl.encode(x, fmt).reshape(10, 100)
        assert np.array_equal(oracle.decode(np.ascontiguousarray(bits), fmt), x.reshape(10, 100))


# ------------------------------------------------------------- planted mistakes

MUTANTS = {
    "transposed_A": ("a = load_elem(A, fmt, i * lda + k)", "a = load_elem(A, fmt, k * lda + i)"),
    "transposed_B": ("p = a * load_elem(B, fmt, k * ldb + j)", "p = a * load_elem(B, fmt, j * ldb + k)"),
    "dropped_last_term": ("for (int64_t k = 0; k < K; ++k) {\n      double a", "for (int64_t k = 0; k + 1 < K; ++k) {\n      double a"),
    "dropped_first_term": ("for (int64_t k = 0; k < K; ++k) {\n      double a", "for (int64_t k = 1; k < K; ++k) {\n      double a"),
    "wrong_sign": ("c[j] += p;", "c[j] -= p;"),
    "abs_dropped": ("s[j] += fabs(p);", "s[j] += p;"),
    "f16_bias": ("e - 25", "e - 24"),
    "f16_subnormal": ("ldexp((double)f, -24)", "ldexp((double)f, -25)"),
    "bf16_shift": ("(uint32_t)h << 16", "(uint32_t)h << 15"),
    "row_index": ("double* c = C + i * N;", "double* c = C + i * N + (i > 0);"),
    "no_zero_init": ("      c[j] = 0.0;\n", "      c[j] = c[j];\n"),
}


def _run_pins_in_this_process(lib_path: str) -> list:
    lib = oracle.load(lib_path)
    failures = []
    for pin in PINS:
        try:
            pin(lib)
        except AssertionError:
            failures.append(pin.__name__)
    return failures


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    """A mutant may write out of bounds, so it runs in a child process; a crash
    of the child counts as caught only if it is not the clean oracle's."""
    if shutil.which("gcc") is None:
        pytest.skip("no host C compiler")
    src = open(oracle.SOURCE).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, name
    d = tempfile.mkdtemp(prefix="oracle_mutant_")
    try:
        path = os.path.join(d, "mutant.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        lib_path = oracle.compile_library(path, os.path.join(d, "libmutant.so"))
        code = ("import sys, json; sys.path.insert(0, %r); sys.path.insert(0, %r); "
                "import test_oracle as t; print(json.dumps(t._run_pins_in_this_process(%r)))"
                % (ROOT, os.path.dirname(__file__), lib_path))
        r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
        if r.returncode == 0:
            failures = json.loads(r.stdout.strip().splitlines()[-1])
            assert failures, f"mutant {name} passes every pin"
        # a non-zero exit (the mutant crashed the child) is a detected mistake
    finally:
        shutil.rmtree(d)


def test_clean_oracle_passes_in_child():
    """The child-process harness itself reports no failure for the real oracle."""
    code = ("import sys, json; sys.path.insert(0, %r); sys.path.insert(0, %r); "
            "import test_oracle as t, oracle; oracle.load(); print(json.dumps(t._run_pins_in_this_process(oracle.LIBRARY)))"
            % (ROOT, os.path.dirname(__file__)))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert json.loads(r.stdout.strip().splitlines()[-1]) == []
