"""GPU parity of the fused epilogue, tgemm_gemm_epilogue:
C = act(alpha A.B + beta C_prior + bias), against the oracle's epilogue
(oracle/epilogue.py) on the oracle's exact product, within the epilogue bound
of tests/tolerance.py, on every kernel path: the swapped-operand pairs, the
pair kernel (also with the stream-K finisher),
the one-SM kernel with bulk-tensor or per-thread operands, the fp32 SIMT
kernel, and the K = 0 fill.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import epilogue as oepi
import workloads as wl
from tests import gpu_harness as H
from tests import tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    H.tg()
    torch.cuda.set_device(0)


EPILOGUES = {
    "bias_relu": dict(alpha=1.0, beta=0.0, activation=1, bias=True),
    "axpby": dict(alpha=0.5, beta=-2.0, activation=0, bias=False),
    "all": dict(alpha=2.0, beta=1.0, activation=1, bias=True),
}

PATHS = {
    "swapped_pairs": {"swap_ab": 2},
    "pairs": {"cta_group": 2, "swap_ab": 1},
    "pairs_per_thread_store": {"cta_group": 2, "swap_ab": 1, "store_mode": 2},
    "one_sm": {"cta_group": 1},
    "one_sm_copy_producers": {"kernel": 2},
    "pairs_copy_producers": {"kernel": 2, "cta_group": 2},
}


def run_case(M, N, K, dtype, epi_name, options, seed, workspace=None, lda=None, ldb=None, poison_prior=False):
    fin, fout = wl.IN_FORMAT[dtype], wl.OUT_FORMAT[dtype]
    if K == 0:  # the empty product: A and B are never read
        A = np.zeros((M, 1), dtype=H.NP_BITS[fin])
        B = np.zeros((1, N), dtype=H.NP_BITS[fin])
    else:
        A, B = wl.make_inputs(wl.Workload("epi", M, N, K, dtype, "uniform", seed), lda=lda, ldb=ldb)
    spec = EPILOGUES[epi_name]
    prior_vals = wl.round_to_format(wl.uniform_pm1(seed + 7, M * N), fout).reshape(M, N)
    prior_bits = wl.encode(prior_vals, fout)
    if poison_prior:
        prior_bits = np.full((M, N), H.CANARY[fout] ^ 1, dtype=H.NP_BITS[fout])  # a NaN pattern
    bias = wl.round_to_format(wl.uniform_pm1(seed + 8, N), "bf16").astype(np.float32) if spec["bias"] else None
    ep = {"alpha": spec["alpha"], "beta": spec["beta"], "activation": spec["activation"]}
    res = H.run_gpu(A, B, M, N, K, dtype, options=options, epilogue=ep, c_prior=prior_bits, bias=bias,
                    workspace=workspace)
    if K == 0:
        D, S = np.zeros((M, N)), np.zeros((M, N))
    else:
        D, S = oracle.gemm(np.ascontiguousarray(A), np.ascontiguousarray(B), fin, M, N, K)
    Cin = oracle.decode(np.ascontiguousarray(prior_bits), fout)
    b64 = None if bias is None else bias.astype(np.float64)
    act = "relu" if spec["activation"] == 1 else "none"
    Z = oepi.apply(D, Cin, spec["alpha"], spec["beta"], b64, act)
    T = oepi.magnitude(S, Cin, spec["alpha"], spec["beta"], b64)
    tol = tolerance.bound_epilogue(Z, S, T, spec["alpha"], fin, fout)
    ok, ratio, where = tolerance.check(res.got, Z, S, fin, fout, tol=tol)
    assert res.guard_ok and res.pad_ok, "guard band or ldc padding of C overwritten"
    assert ok, f"{epi_name} {options}: error/bound {ratio:.3g} at {where}: got {res.got[where]} want {Z[where]}"
    return res


@pytest.mark.parametrize("epi_name", list(EPILOGUES))
@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("dtype", [wl.BF16, wl.F16, wl.BF16_F32OUT], ids=lambda d: wl.DTYPE_NAMES[d])
def test_epilogue_every_tensor_core_path(dtype, path, epi_name):
    """Ragged M, N and K (300 x 520 x 200) on each tensor-core kernel."""
    res = run_case(300, 520, 200, dtype, epi_name, PATHS[path], seed=80)
    if path == "swapped_pairs":
        assert res.plan.swap_ab == 1


@pytest.mark.parametrize("epi_name", list(EPILOGUES))
def test_epilogue_copy_pairs_unaligned_rows(epi_name):
    """B rows of 1048 bytes (8-byte granules): CTA pairs copying B per thread."""
    res = run_case(300, 520, 200, wl.BF16, epi_name, {"cta_group": 2}, seed=81, ldb=524)
    assert res.plan.cta_group == 2 and res.plan.kernel == 2 and res.plan.b_copy_bytes == 8


@pytest.mark.parametrize("epi_name", list(EPILOGUES))
def test_epilogue_stream_k_finisher(epi_name):
    """Tiles split along K: the finishing pair applies the epilogue after
    adding the other pairs' partial sums."""
    opts = {"cta_group": 2, "tile_n": 256, "max_ctas": 16, "stream_k": 2}
    res = run_case(1100, 1304, 640, wl.BF16, epi_name, opts, seed=81, workspace=True)
    assert res.plan.sk_iters > 0


@pytest.mark.parametrize("epi_name", list(EPILOGUES))
def test_epilogue_copy_pairs_stream_k(epi_name):
    """Unaligned B rows on CTA pairs with the stream-K split: the pair that
    finishes a tile applies the epilogue once, to the sum of all partials."""
    opts = {"cta_group": 2, "tile_n": 128, "max_ctas": 16, "stream_k": 2, "repack": 1}
    res = run_case(1100, 1300, 640, wl.BF16, epi_name, opts, seed=86, workspace=True, ldb=1302)
    assert res.plan.kernel == 2 and res.plan.sk_iters > 0


@pytest.mark.parametrize("split", [0, 2], ids=["auto", "split_requested"])
@pytest.mark.parametrize("epi_name", list(EPILOGUES))
@pytest.mark.parametrize("shape", [(300, 520, 200), (129, 257, 33)], ids=lambda s: "x".join(map(str, s)))
def test_epilogue_simt(shape, epi_name, split):
    """With an epilogue the SIMT kernel computes every tile whole, even where
    the plan of the plain product splits tiles into K halves."""
    M, N, K = shape
    run_case(M, N, K, wl.F32, epi_name, {"simt_split": split} if split else None, seed=82)


@pytest.mark.parametrize("epi_name", list(EPILOGUES))
@pytest.mark.parametrize("dtype", [wl.BF16, wl.F16, wl.BF16_F32OUT, wl.F32], ids=lambda d: wl.DTYPE_NAMES[d])
def test_epilogue_k_zero(dtype, epi_name):
    """The empty product: C = act(beta C_prior + bias)."""
    run_case(70, 90, 0, dtype, epi_name, None, seed=83)


def test_beta_zero_never_reads_c():
    """C holding NaN everywhere before the call: with beta = 0 the result is
    finite (and correct), so C was not read."""
    res = run_case(300, 520, 200, wl.BF16, "bias_relu", {"swap_ab": 2}, seed=84, poison_prior=True)
    assert np.isfinite(res.got).all()


def test_headline_shape_with_bias_relu():
    """bf16 4096^3 -> fp32 with bias and ReLU in the benchmark's launch
    configuration, every element."""
    w = wl.BY_NAME["bf16_4096x4096x4096_f32out"]
    A, B, D, S = H.workload_reference(w.name)
    bias = wl.round_to_format(wl.uniform_pm1(85, w.N), "bf16").astype(np.float32)
    ep = {"alpha": 1.0, "beta": 0.0, "activation": 1}
    res = H.run_gpu(A, B, w.M, w.N, w.K, w.dtype, epilogue=ep, bias=bias)
    b = bias.astype(np.float64)
    Z = oepi.apply(D, None, 1.0, 0.0, b, "relu")
    T = oepi.magnitude(S, None, 1.0, 0.0, b)
    tol = tolerance.bound_epilogue(Z, S, T, 1.0, "bf16", "f32")
    ok, ratio, where = tolerance.check(res.got, Z, S, "bf16", "f32", tol=tol)
    assert res.guard_ok and res.pad_ok
    assert ok, f"error/bound {ratio:.3g} at {where}"
