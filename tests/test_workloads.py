"""The seeded input generator: stream, distributions and round-to-nearest-even."""
import numpy as np

import workloads as wl


def test_splitmix64_reference_vector():
    # first three outputs of splitmix64 seeded with 0 in the public reference implementation
    got = [int(x) for x in wl.splitmix64(0, 3)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    # a stream can be resumed at any offset
    assert np.array_equal(wl.splitmix64(12345, 10)[4:], wl.splitmix64(12345, 6, start=4))


def test_uniform_and_normal_moments():
    u = wl.uniform_pm1(wl.seed_for(2, "A"), 1 << 18)
    assert u.min() >= -1.0 and u.max() < 1.0
    assert abs(u.mean()) < 0.01 and abs(u.var() - 1 / 3) < 0.01
    n = wl.normal01(wl.seed_for(3, "B"), 1 << 18)
    assert abs(n.mean()) < 0.01 and abs(n.var() - 1.0) < 0.02
    assert abs(np.mean(n ** 4) - 3.0) < 0.1      # Gaussian kurtosis


def test_rounding_matches_ieee_casts():
    x = np.concatenate([
        wl.normal01(7, 20000) * 10.0 ** np.linspace(-9, 6, 20000),
        wl.uniform_pm1(8, 1000) * 2.0 ** -20,      # fp16 subnormal range
        np.array([65504.0, 65519.99, 65520.0, 1e6, -1e6, 0.0, -0.0, 2.0 ** -25, 2.0 ** -24 * 1.5]),
    ])
    with np.errstate(over="ignore"):
        assert np.array_equal(wl.round_to_format(x, "f16"), x.astype(np.float16).astype(np.float64))
    y = np.concatenate([wl.normal01(9, 20000) * 10.0 ** np.linspace(-44, 38, 20000),
                        np.array([3.4028235677973366e38, 3.4028235e38 * 1.0000001, 1e-46])])
    with np.errstate(over="ignore"):
        assert np.array_equal(wl.round_to_format(y, "f32"), y.astype(np.float32).astype(np.float64))


def test_bf16_rounding_vectors():
    e = 2.0 ** -7   # bf16 ulp at 1.0
    cases = {
        1.0 + e / 2: 1.0,               # tie -> even (1.0)
        1.0 + 3 * e / 2: 1.0 + 2 * e,   # tie -> even (mantissa ...10)
        1.0 + e / 2 + 2.0 ** -30: 1.0 + e,
        -(1.0 + e / 2): -1.0,
        3.14159265: 3.140625,
        2.0 ** -133: 2.0 ** -133,       # smallest subnormal
        2.0 ** -134: 0.0,               # tie -> even (zero)
        1.5 * 2.0 ** -134: 2.0 ** -133,
        (2 - 2 ** -8) * 2.0 ** 127: np.inf,   # max + half ulp overflows
        (2 - 2 ** -7) * 2.0 ** 127: (2 - 2 ** -7) * 2.0 ** 127,
    }
    xs = np.array(list(cases.keys()))
    want = np.array(list(cases.values()))
    assert np.array_equal(wl.round_to_format(xs, "bf16"), want)
    bits = wl.encode(wl.round_to_format(np.array([1.0, -2.0, 3.140625]), "bf16"), "bf16")
    assert list(bits) == [0x3F80, 0xC000, 0x4049]


def test_make_inputs_deterministic_and_padded():
    w = wl.Workload("t", 5, 6, 7, wl.BF16, "normal", 11)
    A1, B1 = wl.make_inputs(w)
    A2, B2 = wl.make_inputs(w, lda=9, ldb=8)
    assert np.array_equal(A1, A2[:, :7]) and np.array_equal(B1, B2[:, :6])
    assert np.all(A2[:, 7:] == 0x7FC0) and np.all(B2[:, 6:] == 0x7FC0)
    # values are representable and decode back exactly
    v = wl.decode(A1, "bf16")
    assert np.array_equal(wl.round_to_format(v, "bf16"), v)


def test_workload_table():
    names = [w.name for w in wl.WORKLOADS[:5]]
    assert names == ["f32_64x64x64", "f16_1024x1024x1024", "bf16_2048x2048x2048",
                     "bf16_4096x4096x4096_f32out", "bf16_1000x1500x4096_ragged"]
    h = wl.HEADLINE
    assert (h.M, h.N, h.K, h.dtype) == (4096, 4096, 4096, wl.BF16_F32OUT)
    assert h.flops == 2 * 4096 ** 3
    assert h.compulsory_bytes == (2 * 4096 * 4096) * 2 + 4096 * 4096 * 4


def test_batch_workload_inputs():
    """The batch benchmark's inputs: matrix 0 of the batch is the one-product
    workload's input (one seeded stream per operand), every matrix is distinct
    and every value is a bf16 value in [-1, 1] (rounding can reach 1)."""
    bw = wl.BATCH_BY_NAME["batch64_bf16_512x512x512"]
    A, B = wl.make_batch_inputs(bw)
    assert A.shape == (bw.batch * bw.M, bw.K) and B.shape == (bw.batch * bw.K, bw.N)
    A1, B1 = wl.make_inputs(bw.one())
    assert np.array_equal(A[:bw.M], A1) and np.array_equal(B[:bw.K], B1)
    assert not np.array_equal(A[:bw.M], A[bw.M:2 * bw.M])
    vals = wl.decode(A[: 4 * bw.M], "bf16")
    assert np.all(vals >= -1.0) and np.all(vals <= 1.0)
    assert bw.flops == 2 * 64 * 512 ** 3
