"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Tolerance (tests/tolerance.py): |C_gpu - C_ref| <= 2^-10 S + ulp_out(C_ref)/2
for fp16/bf16 inputs and <= 2^-20 S for fp32, S = sum_k |a_ik b_kj|.
Every case also checks the guard bands around C and the ldc padding.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu

TC_DTYPES = [wl.F16, wl.BF16, wl.BF16_F32OUT, wl.F16_F32OUT]


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    H.tg()
    torch.cuda.set_device(0)


def case(M, N, K, dtype, dist="uniform", seed=20, lda=None, ldb=None, ldc=None, **kw):
    w = wl.Workload("case", M, N, K, dtype, dist, seed)
    A, B = wl.make_inputs(w, lda=lda, ldb=ldb)
    res = H.run_gpu(A, B, M, N, K, dtype, ldc=ldc, **kw)
    return A, B, res


# ------------------------------------------------------------------ workloads

@pytest.mark.parametrize("name", ["f32_64x64x64", "f16_1024x1024x1024", "bf16_2048x2048x2048",
                                  "bf16_1000x1500x4096_ragged", "f16_512x512x512"])
def test_workload_full_product(name):
    w = wl.BY_NAME[name]
    A, B = wl.make_inputs(w)
    res = H.run_gpu(A, B, w.M, w.N, w.K, w.dtype)
    H.check_full(res, A, B, w.M, w.N, w.K, w.dtype, name)


@pytest.mark.parametrize("name", ["bf16_4096x4096x4096_f32out", "f32_4096x4096x4096", "f32_2048x2048x2048"])
def test_workload_full_size_every_element(name):
    """Full-size products in the launch configuration the benchmark times,
    every element against the oracle's full product."""
    w = wl.BY_NAME[name]
    A, B, ref, S = H.workload_reference(name)
    res = H.run_gpu(A, B, w.M, w.N, w.K, w.dtype)
    H.check_full(res, A, B, w.M, w.N, w.K, w.dtype, name, reference=(ref, S))


def test_workload_f16_8192_bands():
    """f16 8192^3 in the benchmark's launch configuration: every element of one
    whole 256-row band of tiles and one whole 256-column band (about 4.2 M
    outputs, every tile the band crosses), plus the border rows and columns
    and random samples."""
    w = wl.BY_NAME["f16_8192x8192x8192"]
    A, B = wl.make_inputs(w)
    res = H.run_gpu(A, B, w.M, w.N, w.K, w.dtype)
    H.check_block(res, A, B, w.K, w.dtype, 17 * 256, 18 * 256, 0, w.N, "tile row 17")
    H.check_block(res, A, B, w.K, w.dtype, 0, w.M, 23 * 256, 24 * 256, "tile column 23")
    rows, cols = H.sample_positions(w.M, w.N, 4096, seed=99)
    H.check_sampled(res, A, B, w.K, w.dtype, rows, cols, "f16 8192^3")


# ---------------------------------------------- fp32 tiles split into K halves

def slots():
    return 2 * torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("shape,lds", [
    ((300, 200, 1000), (None, None, None)),   # every tile split; 16-byte rows: vector adds
    ((300, 200, 1000), (1003, 205, 211)),     # rows off the 16-byte grid: scalar loads and adds
    ((130, 129, 40), (None, None, 133)),      # three 16-deep stages: halves of one and two stages
], ids=["aligned", "unaligned", "short_k"])
def test_simt_split_all_tiles(shape, lds):
    """simt_split = 2 on a product whose tiles all fit in half of the CTA
    slots: each tile is two CTAs, one per half of its k-stages, adding into
    rows of C the call zeroes; ldc padding and guard bands keep their NaN
    canaries (a missed zero would leave NaN in the sum)."""
    (M, N, K), (lda, ldb, ldc) = shape, lds
    A, B, res = case(M, N, K, wl.F32, seed=120, lda=lda, ldb=ldb, ldc=ldc, options={"simt_split": 2})
    tiles = res.plan.tiles_m * res.plan.tiles_n
    assert res.plan.dp_tiles == 0 and res.plan.ctas == 2 * tiles
    H.check_full(res, A, B, M, N, K, wl.F32, "simt split")


def test_simt_split_off_matches_oracle_too():
    A, B, res = case(300, 200, 1000, wl.F32, seed=120, options={"simt_split": 1})
    assert res.plan.ctas == res.plan.tiles_m * res.plan.tiles_n == res.plan.dp_tiles
    H.check_full(res, A, B, 300, 200, 1000, wl.F32, "simt whole tiles")


def test_simt_split_last_round_auto():
    """20 x 17 tiles on 2 x SMs slots: the last round's tiles are split by
    default (K >= 256), starting in the middle of a tile row whose first
    tiles are computed whole after the zero fill."""
    M, N, K = 20 * 128 - 37, 17 * 128 - 5, 300
    A, B, res = case(M, N, K, wl.F32, seed=121, ldc=N + 3)
    tiles = 20 * 17
    tail = tiles % slots()
    if 0 < tail <= slots() // 2:
        assert res.plan.dp_tiles == tiles - tail and res.plan.ctas == tiles + tail
        assert res.plan.dp_tiles % 17 != 0
    H.check_full(res, A, B, M, N, K, wl.F32, "simt split tail")


@pytest.mark.parametrize("group_m", [1, 3, 7, 16, 40])
def test_simt_raster_groups_with_split_tail(group_m):
    """Tiles in groups of group_m tile rows (column by column within a group),
    with the last round split into K halves: the split tiles of grouped order
    are not a suffix of rows, so the call zeroes their bounding box and any
    whole tile inside it is stored over the zeros.  C starts as NaN canaries,
    so a split tile outside the zeroed box would come back NaN."""
    M, N, K = 20 * 128 - 37, 17 * 128 - 5, 300
    A, B, res = case(M, N, K, wl.F32, seed=123, ldc=N + 3, options={"group_m": group_m, "simt_split": 2})
    assert res.plan.group_m == min(group_m, 20)
    H.check_full(res, A, B, M, N, K, wl.F32, f"simt group {group_m}")


@pytest.mark.parametrize("K", [1, 31, 32, 33, 96, 97, 128, 129, 640, 2048])
@pytest.mark.parametrize("vec", [True, False], ids=["vec", "scalar"])
def test_simt_small_kernel(K, vec):
    """The small-product kernel (32 x 32 tiles, 32-deep stages, 4-stage ring):
    K around the stage and ring depths (every chunk in flight at once up to
    K = 96), ragged M and N; 16-byte copies where every row is 16-byte aligned,
    4-byte copies where none is (padding holds NaN, never read)."""
    M, N = 70, 90
    lda, ldb, ldc = ((K + 3) // 4 * 4, 92, 92) if vec else (K + 5, 93, 91)
    A, B, res = case(M, N, K, wl.F32, seed=124, lda=lda, ldb=ldb, ldc=ldc)
    assert res.plan.tile_m == 32 and res.plan.ctas == 3 * 3
    assert res.plan.store_bytes == (16 if vec else 4)
    H.check_full(res, A, B, M, N, K, wl.F32, f"simt small K {K}")


def test_simt_split_is_deterministic():
    """Two additions onto zero commute: repeated calls give the same bits."""
    A, B, r1 = case(300, 200, 1000, wl.F32, seed=122, options={"simt_split": 2})
    for _ in range(3):
        _, _, r2 = case(300, 200, 1000, wl.F32, seed=122, options={"simt_split": 2})
        assert np.array_equal(r1.raw, r2.raw)


def test_headline_on_plain_pairs():
    """The bf16 4096^3 -> fp32 product on CTA pairs without the operand
    exchange (256 x BN tiles), every element."""
    w = wl.BY_NAME["bf16_4096x4096x4096_f32out"]
    A, B, ref, S = H.workload_reference(w.name)
    res = H.run_gpu(A, B, w.M, w.N, w.K, w.dtype, options={"cta_group": 2, "swap_ab": 1})
    assert res.plan.cluster_ctas == 2 and res.plan.swap_ab == 0
    H.check_full(res, A, B, w.M, w.N, w.K, w.dtype, "plain pairs", reference=(ref, S))


# ------------------------------------------------------------ shape sweeps

SHAPES = [(1, 1, 1), (7, 9, 5), (63, 65, 127), (128, 256, 64), (129, 257, 255), (300, 520, 200),
          (257, 129, 64), (513, 300, 1000)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", TC_DTYPES + [wl.F32], ids=lambda d: wl.DTYPE_NAMES[d])
def test_shape_sweep_auto(shape, dtype):
    M, N, K = shape
    A, B, res = case(M, N, K, dtype, seed=21)
    H.check_full(res, A, B, M, N, K, dtype, f"{shape} {wl.DTYPE_NAMES[dtype]}")


@pytest.mark.parametrize("tile_n", [64, 128, 192, 224, 256])
@pytest.mark.parametrize("store_mode", [1, 2])
@pytest.mark.parametrize("dtype", TC_DTYPES, ids=lambda d: wl.DTYPE_NAMES[d])
def test_tile_widths_and_store_modes(tile_n, store_mode, dtype):
    M, N, K = 300, 520, 200   # 3 row tiles with a 44-row tail, ragged N, K tail of 8
    A, B, res = case(M, N, K, dtype, seed=22, options={"tile_n": tile_n, "store_mode": store_mode})
    assert res.plan.tile_n == tile_n
    assert (res.plan.store_bytes == 0) == (store_mode == 1)
    H.check_full(res, A, B, M, N, K, dtype, f"tile_n {tile_n} store {store_mode}")


@pytest.mark.parametrize("tile_n", [64, 128, 192, 224, 256])
@pytest.mark.parametrize("dtype", [wl.BF16, wl.F16_F32OUT], ids=lambda d: wl.DTYPE_NAMES[d])
def test_copy_producer_on_aligned_rows(tile_n, dtype):
    """Force the per-thread-copy producer (16-byte granules) on aligned data."""
    M, N, K = 260, 390, 300
    # padded pitches (304 and 392 elements = 608 and 784 bytes) keep every row 16-byte aligned
    A, B, res = case(M, N, K, dtype, seed=23, lda=304, ldb=392, ldc=392,
                     options={"kernel": 2, "tile_n": tile_n})
    assert res.plan.kernel == 2 and res.plan.a_copy_bytes == 16 and res.plan.b_copy_bytes == 16
    H.check_full(res, A, B, M, N, K, dtype, f"copy tile_n {tile_n}")


# ------------------------------------------- CTA pairs copying B per thread

@pytest.mark.parametrize("ldb,b_off,granule", [(300, 0, 8), (302, 0, 4), (301, 0, 2), (304, 8, 8)],
                         ids=["pitch600", "pitch604", "pitch602", "base_plus_8"])
@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("dtype", [wl.BF16, wl.F16_F32OUT], ids=lambda d: wl.DTYPE_NAMES[d])
def test_copy_pair_kernel(tile_n, dtype, ldb, b_off, granule):
    """B rows off the 16-byte grid, A rows on it: CTA pairs whose CTAs copy
    their halves of B per thread.  Ragged M (the third pair tile has 8 rows),
    ragged N and a K tail, for each copy granule."""
    M, N, K = 520, 300, 200
    A, B, res = case(M, N, K, dtype, seed=26, lda=208, ldb=ldb, b_off=b_off,
                     options={"cta_group": 2, "tile_n": tile_n})
    p = res.plan
    assert (p.kernel, p.cta_group, p.tile_n, p.a_copy_bytes, p.b_copy_bytes) == (2, 2, tile_n, 0, granule)
    H.check_full(res, A, B, M, N, K, dtype, f"copy pair {tile_n} ldb {ldb}+{b_off}")


@pytest.mark.parametrize("tile_n", [128, 256])
def test_copy_pair_forced_on_aligned_rows(tile_n):
    """kernel = copy with cta_group = 2 on aligned rows: 16-byte copies of B,
    bulk-tensor loads of A, per-thread stores of C."""
    M, N, K = 600, 392, 328
    A, B, res = case(M, N, K, wl.BF16, seed=27, lda=336, ldb=392, ldc=400,
                     options={"kernel": 2, "cta_group": 2, "tile_n": tile_n})
    assert (res.plan.cta_group, res.plan.a_copy_bytes, res.plan.b_copy_bytes) == (2, 0, 16)
    H.check_full(res, A, B, M, N, K, wl.BF16, f"copy pair aligned {tile_n}")


@pytest.mark.parametrize("max_ctas,group_m", [(4, 1), (6, 3), (2, 2)])
def test_copy_pair_persistent(max_ctas, group_m):
    """Few pairs walking many tiles: every ring and accumulator phase turns
    over many times (1100 x 700 in 256 x 128 tiles = 30 tiles)."""
    M, N, K = 1100, 700, 264
    A, B, res = case(M, N, K, wl.BF16, seed=28, lda=264, ldb=700, ldc=700,
                     options={"cta_group": 2, "tile_n": 128, "max_ctas": max_ctas, "group_m": group_m})
    assert res.plan.cta_group == 2 and res.plan.ctas == max_ctas and res.plan.b_copy_bytes == 8
    H.check_full(res, A, B, M, N, K, wl.BF16, f"copy pair persistent {max_ctas}")


@pytest.mark.parametrize("offsets", [(2, 0, 0), (4, 4, 4), (8, 8, 8), (0, 2, 2), (6, 10, 12)])
@pytest.mark.parametrize("dtype", [wl.BF16, wl.F16], ids=lambda d: wl.DTYPE_NAMES[d])
def test_misaligned_pointers(offsets, dtype):
    """Bases off the 16-byte grid take the copy producer / per-thread stores."""
    a_off, b_off, c_off = offsets
    M, N, K = 200, 333, 150
    A, B, res = case(M, N, K, dtype, seed=24, lda=152, ldb=336, ldc=340, a_off=a_off, b_off=b_off, c_off=c_off)
    H.check_full(res, A, B, M, N, K, dtype, f"offsets {offsets}")


@pytest.mark.parametrize("lds", [(70, 90, 95), (72, 88, 96), (71, 83, 83), (65, 81, 81), (80, 96, 96)])
@pytest.mark.parametrize("dtype", [wl.BF16, wl.BF16_F32OUT, wl.F32], ids=lambda d: wl.DTYPE_NAMES[d])
def test_leading_dimensions(lds, dtype):
    """ld > dim: A/B padding holds NaN (must never be read), C padding a canary
    (must never be written)."""
    lda, ldb, ldc = lds
    M, N, K = 150, 81, 65
    A, B, res = case(M, N, K, dtype, seed=25, lda=lda, ldb=ldb, ldc=ldc)
    H.check_full(res, A, B, M, N, K, dtype, f"lds {lds}")


# ------------------------------------------------------------ CTA-pair kernel

@pytest.mark.parametrize("store_mode", [1, 2])
@pytest.mark.parametrize("tile_n", [128, 192, 224, 256])
@pytest.mark.parametrize("dtype", TC_DTYPES, ids=lambda d: wl.DTYPE_NAMES[d])
def test_pair_kernel(tile_n, dtype, store_mode):
    """256 x tile_n tiles on CTA pairs: ragged M (two pair tiles, the second
    44 rows), ragged N and a K tail; staged bulk-tensor stores (store_mode 1)
    and the unstaged variant with a deeper ring (store_mode 2)."""
    M, N, K = 300, 520, 200
    A, B, res = case(M, N, K, dtype, seed=34, options={"cta_group": 2, "tile_n": tile_n, "store_mode": store_mode,
                                                             "swap_ab": 1})
    assert res.plan.cta_group == 2 and res.plan.tile_m == 256 and res.plan.tile_n == tile_n
    assert res.plan.cluster_ctas == 2
    H.check_full(res, A, B, M, N, K, dtype, f"pair tile_n {tile_n}")


@pytest.mark.parametrize("tile_k", [64, 128])
@pytest.mark.parametrize("store_mode", [1, 2])
@pytest.mark.parametrize("max_ctas", [2, 6, 0])
def test_pair_kernel_persistent(store_mode, max_ctas, tile_k):
    """One or three pairs walking many 256 x 256 tiles (every ring and
    accumulator phase), and the full grid."""
    M, N, K = 1100, 1300, 330
    A, B, res = case(M, N, K, wl.BF16_F32OUT, seed=35, lda=336, ldb=1304,
                     options={"cta_group": 2, "tile_n": 256, "max_ctas": max_ctas, "store_mode": store_mode,
                              "tile_k": tile_k, "swap_ab": 1})
    assert res.plan.cta_group == 2 and res.plan.cluster_ctas == 2
    if max_ctas:
        assert res.plan.ctas == max_ctas
    H.check_full(res, A, B, M, N, K, wl.BF16_F32OUT, f"pair ctas {max_ctas} store {store_mode}")


@pytest.mark.parametrize("tile_k", [64, 128])
@pytest.mark.parametrize("K", [16, 64, 65, 128, 129, 384, 385, 448])
def test_pair_kernel_k_depths(K, tile_k):
    """K around multiples of the stage depth (64, or 128 = two sub-blocks per
    stage, where the last stage may hold a sub-block entirely past K)."""
    M, N = 257, 260
    lda = (K + 7) // 8 * 8   # 16-byte rows for the bulk-tensor loads of the pair kernel
    A, B, res = case(M, N, K, wl.BF16, seed=36, lda=lda, ldb=264,
                     options={"cta_group": 2, "tile_n": 128, "tile_k": tile_k, "swap_ab": 1})
    assert res.plan.tile_k == tile_k and res.plan.cluster_ctas == 2
    H.check_full(res, A, B, M, N, K, wl.BF16, f"pair K {K}")


# ------------------------------- pairs with the MMA's operands exchanged

@pytest.mark.parametrize("store_mode", [1, 2])
@pytest.mark.parametrize("tile_m", [128, 192, 224, 256])
@pytest.mark.parametrize("dtype", TC_DTYPES, ids=lambda d: wl.DTYPE_NAMES[d])
def test_swap_kernel(tile_m, dtype, store_mode):
    """tile_m x 256 tiles computed as tiles of C^T: ragged M (a partial
    second tile), ragged N (the second pair tile's upper CTA half lies past N),
    a K tail; bulk-tensor stores of 32 x 32 blocks (store_mode 1) and
    per-thread stores (store_mode 2)."""
    M, N, K = 300, 520, 200
    A, B, res = case(M, N, K, dtype, seed=40, options={"swap_ab": 2, "tile_m": tile_m, "store_mode": store_mode})
    assert res.plan.swap_ab == 1 and res.plan.tile_m == tile_m and res.plan.tile_n == 256
    assert (res.plan.store_bytes == 0) == (store_mode == 1)
    H.check_full(res, A, B, M, N, K, dtype, f"swap tile_m {tile_m} store {store_mode}")


@pytest.mark.parametrize("tile_k", [64, 128])
@pytest.mark.parametrize("max_ctas,group_m", [(2, 0), (6, 3), (0, 0)])
def test_swap_kernel_persistent(max_ctas, group_m, tile_k):
    """One and three pairs walking many 224 x 256 tiles, and the full grid."""
    M, N, K = 1100, 1300, 330
    A, B, res = case(M, N, K, wl.BF16_F32OUT, seed=41, lda=336, ldb=1304,
                     options={"swap_ab": 2, "tile_m": 224, "max_ctas": max_ctas, "group_m": group_m,
                              "tile_k": tile_k})
    assert res.plan.swap_ab == 1
    if max_ctas:
        assert res.plan.ctas == max_ctas
    H.check_full(res, A, B, M, N, K, wl.BF16_F32OUT, f"swap ctas {max_ctas} group {group_m}")


@pytest.mark.parametrize("tile_k", [64, 128])
@pytest.mark.parametrize("K", [16, 64, 65, 128, 129, 384, 385, 448])
def test_swap_kernel_k_depths(K, tile_k):
    M, N = 257, 264
    lda = (K + 7) // 8 * 8
    A, B, res = case(M, N, K, wl.BF16, seed=42, lda=lda,
                     options={"swap_ab": 2, "tile_m": 128, "tile_k": tile_k})
    assert res.plan.tile_k == tile_k and res.plan.swap_ab == 1
    H.check_full(res, A, B, M, N, K, wl.BF16, f"swap K {K}")


@pytest.mark.parametrize("tile_m", [192, 224, 256])
def test_swap_kernel_headline(tile_m):
    """bf16 4096^3 -> fp32 in tile_m x 256 swapped tiles, every element."""
    w = wl.BY_NAME["bf16_4096x4096x4096_f32out"]
    A, B, ref, S = H.workload_reference(w.name)
    res = H.run_gpu(A, B, w.M, w.N, w.K, w.dtype, options={"swap_ab": 2, "tile_m": tile_m})
    assert res.plan.swap_ab == 1 and res.plan.tile_m == tile_m
    H.check_full(res, A, B, w.M, w.N, w.K, w.dtype, f"swap {tile_m}", reference=(ref, S))


# ------------------------------------------------------- scheduler and edges

@pytest.mark.parametrize("max_ctas,group_m", [(1, 1), (3, 2), (5, 16), (7, 3)])
def test_persistent_scheduler(max_ctas, group_m):
    """Few CTAs walking many tiles exercises every phase of the stage ring and
    of the two accumulator buffers."""
    M, N, K = 1100, 1300, 300
    A, B, res = case(M, N, K, wl.BF16, seed=26, options={"max_ctas": max_ctas, "group_m": group_m, "tile_n": 128})
    assert res.plan.ctas == max_ctas
    H.check_full(res, A, B, M, N, K, wl.BF16, f"ctas {max_ctas} group {group_m}")


@pytest.mark.parametrize("K", [1, 16, 63, 64, 65, 128, 192, 320, 448, 640])
def test_k_block_counts(K):
    """K around multiples of the 64-wide stage and of the ring depth."""
    M, N = 130, 260
    for dtype, opts in ((wl.BF16_F32OUT, {"tile_n": 256}), (wl.F16, {"tile_n": 64}), (wl.BF16, {"tile_n": 224}),
                        (wl.F16_F32OUT, {"tile_n": 192}), (wl.F32, None)):
        A, B, res = case(M, N, K, dtype, seed=27, options=opts)
        H.check_full(res, A, B, M, N, K, dtype, f"K {K} {wl.DTYPE_NAMES[dtype]}")


@pytest.mark.parametrize("N,ldc", [(390, 392), (390, 400), (392, 400), (385, 392)])
def test_store_never_touches_row_padding(N, ldc):
    """The row end of C is not always on a 16-byte boundary: nothing past
    column N may change (bulk-tensor stores are used only when it is)."""
    M, K = 260, 304
    A, B, res = case(M, N, K, wl.BF16, seed=33, lda=304, ldb=400, ldc=ldc)
    assert (res.plan.store_bytes == 0) == ((N * 2) % 16 == 0)
    H.check_full(res, A, B, M, N, K, wl.BF16, f"N {N} ldc {ldc}")


def test_empty_dimensions_leave_c_untouched():
    for (M, N, K) in [(0, 5, 7), (5, 0, 7)]:
        A, B, res = case(M, N, K, wl.BF16, seed=28, lda=max(K, 1), ldb=max(N, 1), ldc=max(N, 1))
        assert res.guard_ok and res.pad_ok


@pytest.mark.parametrize("dtype", TC_DTYPES + [wl.F32], ids=lambda d: wl.DTYPE_NAMES[d])
def test_k_zero_writes_zeros(dtype):
    M, N = 37, 45
    w = wl.Workload("k0", M, 1, 1, dtype, "uniform", 29)
    fin = wl.IN_FORMAT[dtype]
    A = np.zeros((M, 1), dtype=H.NP_BITS[fin])
    B = np.zeros((1, N), dtype=H.NP_BITS[fin])
    res = H.run_gpu(A, B, M, N, 0, dtype, ldc=N + 3)
    assert res.guard_ok and res.pad_ok
    assert np.all(res.raw == 0)   # +0 in every format


def test_deterministic():
    A, B, r1 = case(700, 900, 777, wl.BF16, seed=30)
    r2 = H.run_gpu(A, B, 700, 900, 777, wl.BF16)
    assert np.array_equal(r1.raw, r2.raw)


def test_nan_poisons_only_its_row():
    M, N, K = 200, 300, 100
    w = wl.Workload("nan", M, N, K, wl.BF16, "uniform", 31)
    A, B = wl.make_inputs(w)
    A = A.copy()
    A[17, 50] = 0x7FC0   # NaN
    res = H.run_gpu(A, B, M, N, K, wl.BF16)
    assert np.all(np.isnan(res.got[17]))
    assert not np.any(np.isnan(np.delete(res.got, 17, axis=0)))


def test_simt_and_tensor_core_agree_with_oracle_on_same_values():
    """bf16-representable values run through the fp32 SIMT path and the bf16
    tensor-core path; both must meet their own bound against the oracle."""
    M, N, K = 256, 384, 512
    w = wl.Workload("x", M, N, K, wl.BF16, "uniform", 32)
    A16, B16 = wl.make_inputs(w)
    A32 = (A16.astype(np.uint32) << np.uint32(16))
    B32 = (B16.astype(np.uint32) << np.uint32(16))
    r16 = H.run_gpu(A16, B16, M, N, K, wl.BF16_F32OUT)
    r32 = H.run_gpu(A32, B32, M, N, K, wl.F32)
    H.check_full(r16, A16, B16, M, N, K, wl.BF16_F32OUT, "tc")
    H.check_full(r32, A32, B32, M, N, K, wl.F32, "simt")
