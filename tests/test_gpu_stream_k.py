"""GPU parity of the stream-K tail of the CTA-pair kernel (tgemm_gemm_ws).

Tiles left over after the last full round of CTA pairs are split along K over
all pairs; partial fp32 sums go through the caller's workspace and the pair
holding a tile's last k-stage adds them in a fixed order.  Checked against the
oracle, for determinism, and for reuse of one workspace by consecutive calls.
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


def case(M, N, K, dtype, options, seed, lda=None, ldb=None, ldc=None, workspace=True):
    w = wl.Workload("sk", M, N, K, dtype, "uniform", seed)
    A, B = wl.make_inputs(w, lda=lda, ldb=ldb)
    return A, B, H.run_gpu(A, B, M, N, K, dtype, ldc=ldc, options=options, workspace=workspace)


@pytest.mark.parametrize("tile_k", [64, 128])
@pytest.mark.parametrize("tile_n", [128, 192, 224, 256])
@pytest.mark.parametrize("dtype", [wl.BF16, wl.BF16_F32OUT, wl.F16, wl.F16_F32OUT], ids=lambda d: wl.DTYPE_NAMES[d])
def test_stream_k_tail(dtype, tile_n, tile_k):
    """8 pairs over 5 x ceil(1300/tile_n) pair tiles: the remainder is split
    along K (several workers per tile, finishing pairs add 1..3 partials)."""
    M, N, K = 1100, 1304, 640
    opts = {"cta_group": 2, "tile_n": tile_n, "tile_k": tile_k, "max_ctas": 16, "stream_k": 2}
    A, B, res = case(M, N, K, dtype, opts, seed=70)
    assert res.plan.cta_group == 2 and res.plan.sk_iters > 0 and res.plan.ctas == 16
    H.check_full(res, A, B, M, N, K, dtype, f"stream-K tile_n {tile_n} tile_k {tile_k}")


@pytest.mark.parametrize("max_ctas,K", [(6, 1024), (8, 1024), (14, 512), (0, 4096)])
def test_stream_k_more_workers_than_tiles(max_ctas, K):
    """10 pair tiles on 3, 4, 7 and all pairs: remainders of 1..10 tiles, up
    to every tile split across ~8 pairs."""
    M, N = 512, 1280
    opts = {"cta_group": 2, "tile_n": 256, "max_ctas": max_ctas, "stream_k": 2}
    A, B, res = case(M, N, K, wl.BF16_F32OUT, opts, seed=71)
    H.check_full(res, A, B, M, N, K, wl.BF16_F32OUT, f"stream-K ctas {max_ctas} K {K}")


@pytest.mark.parametrize("tile_k", [64, 128])
@pytest.mark.parametrize("dtype", [wl.BF16, wl.BF16_F32OUT], ids=lambda d: wl.DTYPE_NAMES[d])
@pytest.mark.parametrize("M,N", [(256, 256), (512, 256)])
def test_stream_k_many_contributors(M, N, dtype, tile_k):
    """One or two 256 x 256 tiles with a long K over every pair: each tile is
    split across dozens of pairs, more partial sums than the finishing warp's
    share of the ring holds, so they are added in several rounds."""
    K = 16384
    opts = {"cta_group": 2, "tile_n": 256, "tile_k": tile_k, "stream_k": 2}
    A, B, res = case(M, N, K, dtype, opts, seed=74)
    assert res.plan.sk_iters > 0 and res.plan.dp_tiles == 0
    H.check_full(res, A, B, M, N, K, dtype, f"stream-K {M}x{N} K {K} tile_k {tile_k}")


def test_stream_k_deterministic_and_workspace_reuse():
    """The same workspace serves consecutive calls without clearing; the
    fixed summation order makes repeated results bitwise equal."""
    M, N, K = 1100, 1304, 1024
    opts = {"cta_group": 2, "tile_n": 256, "max_ctas": 16, "stream_k": 2}
    A, B, r1 = case(M, N, K, wl.BF16, opts, seed=72)
    assert r1.plan.sk_iters > 0
    r2 = H.run_gpu(A, B, M, N, K, wl.BF16, options=opts, workspace=r1.workspace)
    assert np.array_equal(r1.raw, r2.raw)
    # different inputs through the same workspace
    A2, B2, _ = case(M, N, K, wl.BF16, opts, seed=73, workspace=False)
    r3 = H.run_gpu(A2, B2, M, N, K, wl.BF16, options=opts, workspace=r1.workspace)
    H.check_full(r3, A2, B2, M, N, K, wl.BF16, "reused workspace")


@pytest.mark.parametrize("name", ["bf16_4096x4096x4096_f32out", "bf16_2048x2048x2048"])
def test_stream_k_workloads(name):
    """Full-size workloads with the stream-K tail forced on (tile choice automatic)."""
    w = wl.BY_NAME[name]
    A, B, ref, S = H.workload_reference(name)
    res = H.run_gpu(A, B, w.M, w.N, w.K, w.dtype, workspace=True, options={"stream_k": 2})
    assert res.plan.sk_iters > 0
    H.check_full(res, A, B, w.M, w.N, w.K, w.dtype, name, reference=(ref, S))


def test_workspace_too_small_runs_whole_tiles():
    M, N, K = 1100, 1304, 640
    opts = {"cta_group": 2, "tile_n": 256, "max_ctas": 16, "stream_k": 2}
    ws = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    A, B, res = case(M, N, K, wl.BF16, opts, seed=74, workspace=ws)
    assert res.plan.sk_iters == 0
    H.check_full(res, A, B, M, N, K, wl.BF16, "small workspace")


# ------------------------------- CTA pairs copying B per thread (unaligned B rows)

@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("dtype", [wl.BF16, wl.BF16_F32OUT, wl.F16], ids=lambda d: wl.DTYPE_NAMES[d])
@pytest.mark.parametrize("max_ctas,ldb_pad", [(16, 0), (14, 6), (0, 1)], ids=["8_pairs_8B", "7_pairs_4B", "all_2B"])
def test_copy_pair_stream_k(dtype, tile_n, max_ctas, ldb_pad):
    """B rows off the 16-byte grid (ldb = N + pad = 1300, 1306, 1301: pitches of
    2600, 2612 and 2602 bytes, 8-, 4- and 2-byte granules) on CTA pairs that
    copy B per thread, with the tiles past the last full round of pairs split
    along K: ragged M, N and K, finishing pairs add one or more partial sums."""
    M, N, K = 1100, 1300, 1000
    opts = {"cta_group": 2, "tile_n": tile_n, "max_ctas": max_ctas, "stream_k": 2, "repack": 1}
    A, B, res = case(M, N, K, dtype, opts, seed=75, ldb=N + ldb_pad)
    assert res.plan.kernel == 2 and res.plan.cta_group == 2 and res.plan.sk_iters > 0
    assert res.plan.b_copy_bytes == {0: 8, 6: 4, 1: 2}[ldb_pad]
    H.check_full(res, A, B, M, N, K, dtype, f"copy-pair stream-K tile_n {tile_n} ctas {max_ctas}")


def test_copy_pair_stream_k_ragged_workload():
    """The ragged bf16 1000 x 1500 x 4096 workload (3000-byte B rows): 48 pair
    tiles spread over every pair, every element against the oracle, and a
    second call through the same workspace gives the same bits."""
    w = wl.BY_NAME["bf16_1000x1500x4096_ragged"]
    A, B = wl.make_inputs(w)
    opts = {"stream_k": 2, "repack": 1}
    r1 = H.run_gpu(A, B, w.M, w.N, w.K, w.dtype, workspace=True, options=opts)
    assert r1.plan.kernel == 2 and r1.plan.cta_group == 2 and r1.plan.sk_iters == 48 * 64
    assert r1.plan.dp_tiles == 0
    H.check_full(r1, A, B, w.M, w.N, w.K, w.dtype, "ragged workload, stream-K")
    r2 = H.run_gpu(A, B, w.M, w.N, w.K, w.dtype, workspace=r1.workspace, options=opts)
    assert np.array_equal(r1.raw, r2.raw)


@pytest.mark.parametrize("K", [200, 257, 448, 1000])
def test_copy_pair_stream_k_short_k(K):
    """Few k-stages per tile over every pair (24 pair tiles of 4 to 16 stages
    on 76 pairs): ranges of one or two stages, tiles finished by pairs that
    hold a single stage; B rows of 1804 bytes (4-byte granules)."""
    M, N = 600, 900
    opts = {"cta_group": 2, "tile_n": 128, "stream_k": 2, "repack": 1}
    A, B, res = case(M, N, K, wl.BF16, opts, seed=76, lda=(K + 7) // 8 * 8, ldb=N + 2)
    assert res.plan.kernel == 2 and res.plan.sk_iters > 0 and res.plan.b_copy_bytes == 4
    H.check_full(res, A, B, M, N, K, wl.BF16, f"copy-pair stream-K K {K}")
