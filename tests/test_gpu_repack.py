"""GPU parity of operand repacking (tgemm_options.repack, tgemm_gemm_ws).

An operand whose rows are not 16-byte aligned is copied into the caller's
workspace with its pitch rounded up to 8 elements, and the bulk-tensor
kernels read the copy.  Elements move as raw bits, so every result is checked
against the oracle under the usual tolerance, with the guard bands and ldc
padding of C intact; the original operands are never written.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    H.tg()
    torch.cuda.set_device(0)


def case(M, N, K, dtype, seed, lda=None, ldb=None, ldc=None, options=None, workspace=True):
    w = wl.Workload("repack", M, N, K, dtype, "uniform", seed)
    A, B = wl.make_inputs(w, lda=lda, ldb=ldb)
    return A, B, H.run_gpu(A, B, M, N, K, dtype, ldc=ldc, options=options, workspace=workspace)


def test_ragged_workload_repacks_b():
    """bf16 1000 x 1500 x 4096 (3000-byte B rows): with a workspace, B is
    copied to a 3008-byte pitch and the bulk-tensor kernels run; every
    element against the oracle."""
    w = wl.BY_NAME["bf16_1000x1500x4096_ragged"]
    A, B = wl.make_inputs(w)
    res = H.run_gpu(A, B, w.M, w.N, w.K, w.dtype, workspace=True)
    assert res.plan.packed == 2 and res.plan.kernel == 1 and res.plan.b_copy_bytes == 0
    H.check_full(res, A, B, w.M, w.N, w.K, w.dtype, "ragged, B repacked")


# (pad of lda past K, pad of ldb past N): source granules 8, 4 and 2 bytes
PADS = [(0, 4), (2, 2), (1, 1), (0, 0)]


@pytest.mark.parametrize("pads", PADS, ids=lambda p: f"lda+{p[0]}_ldb+{p[1]}")
@pytest.mark.parametrize("dtype", [wl.BF16, wl.F16, wl.BF16_F32OUT, wl.F16_F32OUT], ids=lambda d: wl.DTYPE_NAMES[d])
@pytest.mark.parametrize("shape", [(300, 520, 204), (600, 1000, 1030), (129, 77, 35)],
                         ids=lambda s: "x".join(map(str, s)))
def test_repack_any_operand(shape, dtype, pads):
    """repack = 2 on ragged shapes whose K and N are not multiples of 8, so
    rows of A and/or B (and C) are off the 16-byte grid; whatever stays
    aligned is read in place."""
    M, N, K = shape
    lda, ldb = K + pads[0], N + pads[1]
    A, B, res = case(M, N, K, dtype, seed=140, lda=lda, ldb=ldb, ldc=N + 3, options={"repack": 2})
    want = (0 if (lda * 2) % 16 == 0 else 1) | (0 if (ldb * 2) % 16 == 0 else 2)
    assert res.plan.packed == want
    if want == 3:
        assert res.plan.kernel == 1  # both operands now go through bulk-tensor copies
    H.check_full(res, A, B, M, N, K, dtype, f"repack {shape} pads {pads}")


@pytest.mark.parametrize("options", [{"repack": 2, "stream_k": 2, "cta_group": 2, "swap_ab": 1, "tile_n": 128},
                                     {"repack": 2, "swap_ab": 2, "tile_m": 128},
                                     {"repack": 2, "cta_group": 1}],
                         ids=["pairs_stream_k", "swapped_pairs", "one_sm"])
def test_repack_on_every_bulk_tensor_kernel(options):
    """The copies feed each bulk-tensor kernel; with the stream-K split the
    workspace holds flags, partial sums and the copy of B at once."""
    M, N, K = 1100, 1302, 1000
    A, B, res = case(M, N, K, wl.BF16, seed=141, lda=1000, ldb=1302, options=options)
    assert res.plan.packed == 2
    if options.get("stream_k") == 2:
        assert res.plan.sk_iters > 0
    H.check_full(res, A, B, M, N, K, wl.BF16, f"repack {options}")


def test_workspace_reused_across_shapes_and_splits():
    """One workspace serves, in turn, a repacking product, a stream-K product
    whose flags take the first 4 KiB, and the repacking product again: flags
    only ever land on flags, so no call reads another's leftovers."""
    M, N, K = 1000, 1500, 2048
    A1, B1 = wl.make_inputs(wl.Workload("reuse", M, N, K, wl.BF16, "uniform", 142))
    need = 64 << 20
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    r1 = H.run_gpu(A1, B1, M, N, K, wl.BF16, workspace=ws)
    assert r1.plan.packed == 2
    H.check_full(r1, A1, B1, M, N, K, wl.BF16, "repack, first")
    A2, B2 = wl.make_inputs(wl.Workload("reuse", 1100, 1304, 640, wl.BF16, "uniform", 143))
    opts = {"cta_group": 2, "tile_n": 256, "max_ctas": 16, "stream_k": 2}
    r2 = H.run_gpu(A2, B2, 1100, 1304, 640, wl.BF16, options=opts, workspace=ws)
    assert r2.plan.sk_iters > 0
    H.check_full(r2, A2, B2, 1100, 1304, 640, wl.BF16, "stream-K between")
    r3 = H.run_gpu(A1, B1, M, N, K, wl.BF16, workspace=ws)
    assert np.array_equal(r1.raw, r3.raw)


@pytest.mark.parametrize("epi", [{"alpha": 2.0, "beta": 1.0, "activation": 1}, {"alpha": 0.5, "beta": 0.0,
                                                                                  "activation": 0}],
                         ids=["all", "scale"])
def test_repack_with_epilogue(epi):
    from oracle import epilogue as oepi
    import oracle
    from tests import tolerance
    M, N, K = 600, 1000, 520
    A, B = wl.make_inputs(wl.Workload("repack_epi", M, N, K, wl.BF16, "uniform", 144), ldb=N + 2)
    prior = wl.round_to_format(wl.uniform_pm1(145, M * N), "bf16").reshape(M, N)
    bias = wl.round_to_format(wl.uniform_pm1(146, N), "bf16").astype(np.float32)
    res = H.run_gpu(A, B, M, N, K, wl.BF16, epilogue=epi, c_prior=wl.encode(prior, "bf16"), bias=bias,
                    workspace=True, options={"repack": 2})
    assert res.plan.packed == 2
    D, S = oracle.gemm(np.ascontiguousarray(A), np.ascontiguousarray(B), "bf16", M, N, K)
    act = "relu" if epi["activation"] == 1 else "none"
    b64 = bias.astype(np.float64)
    Z = oepi.apply(D, prior, epi["alpha"], epi["beta"], b64, act)
    T = oepi.magnitude(S, prior, epi["alpha"], epi["beta"], b64)
    tol = tolerance.bound_epilogue(Z, S, T, epi["alpha"], "bf16", "bf16")
    ok, ratio, where = tolerance.check(res.got, Z, S, "bf16", "bf16", tol=tol)
    assert ok and res.guard_ok and res.pad_ok, f"error/bound {ratio:.3g} at {where}"
