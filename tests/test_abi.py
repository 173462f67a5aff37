"""The C ABI on the host: the library loads, exports every declared entry
point, and its validation and dispatch planning behave as include/tgemm.h
states.  None of these calls reaches the GPU (validation errors are returned
before any CUDA call; tgemm_plan never touches the device)."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def tg():
    from tests.conftest import build_library
    build_library()
    import tiled_dense_gemm_02_gb300 as tg
    return tg


HEADER = os.path.join(ROOT, "include", "tgemm.h")


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*TGEMM_API\s+(?:const\s+)?\w+\s*\*?\s*(tgemm_\w+)\s*\(", text, re.M)))


def test_header_declares_the_abi():
    names = declared_functions()
    assert names == sorted(["tgemm_gemm", "tgemm_gemm_ex", "tgemm_gemm_ws", "tgemm_workspace_size", "tgemm_plan",
                            "tgemm_gemm_noalloc", "tgemm_gemm_epilogue", "tgemm_gemm_batched",
                            "tgemm_plan_batched", "tgemm_transpose", "tgemm_gemm_host", "tgemm_device_status",
                            "tgemm_status_string", "tgemm_version", "tgemm_host_counters"])


def test_library_exports_every_declared_symbol(tg):
    lib = tg.library()
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) == set(tg.EXPORTS)
    assert tg.version() == 10000


def test_host_counters_need_no_gpu(tg):
    """The counters are readable without a device; validation-only calls move
    none of them."""
    c0 = tg.host_counters()
    assert set(c0) == {"tc_launches", "map_hits", "map_encodes", "ns_prepare", "ns_launch"}
    assert tg.gemm(-1, 4, 4, 0, 4, 0, 4, 0, 4, tg.BF16) == tg.ERR_INVALID_VALUE
    assert tg.gemm(0, 4, 4, 0, 4, 0, 4, 0, 4, tg.BF16) == tg.OK
    assert tg.host_counters() == c0
    assert tg.library().tgemm_host_counters(None) == tg.ERR_INVALID_VALUE


def test_noalloc_scratch_size_matches_header(tg):
    """The binding's copy of TGEMM_NOALLOC_SCRATCH_BYTES is the header's value:
    4 KiB of stream-K flags and 20 MiB of partial sums, enough for every pair
    of 152 SMs at the widest tile."""
    text = open(HEADER).read()
    m = re.search(r"#define\s+TGEMM_NOALLOC_SCRATCH_BYTES\s+\(\(size_t\)(\d+)\s*\*\s*(\d+)\s*\*\s*(\d+)\s*\+\s*(\d+)\)",
                  text)
    assert m, "TGEMM_NOALLOC_SCRATCH_BYTES not found in the header"
    a, b, c, d = (int(g) for g in m.groups())
    assert a * b * c + d == tg.NOALLOC_SCRATCH_BYTES
    assert 4096 + 76 * 2 * 4 * 32 * 256 * 4 <= tg.NOALLOC_SCRATCH_BYTES


def header_struct_fields(name):
    """(field, element count) of `typedef struct name {...} name;` in the header,
    which declares int fields only."""
    text = open(HEADER).read()
    body = re.search(r"typedef struct %s \{(.*?)\} %s;" % (name, name), text, re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = []
    for decl in body.split(";"):
        decl = decl.strip()
        if not decl:
            continue
        assert decl.startswith("int "), decl
        for part in decl[4:].split(","):
            m = re.fullmatch(r"\s*(\w+)\s*(?:\[(\d+)\])?\s*", part)
            fields.append((m.group(1), int(m.group(2) or 1)))
    return fields


def test_epilogue_struct_matches_header(tg):
    text = open(HEADER).read()
    body = re.search(r"typedef struct tgemm_epilogue \{(.*?)\} tgemm_epilogue;", text, re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    decls = [d.strip() for d in body.split(";") if d.strip()]
    assert decls == ["float alpha", "float beta", "const float* bias", "int activation", "int reserved[3]"]
    assert [f for f, _ in tg.Epilogue._fields_] == ["alpha", "beta", "bias", "activation", "reserved"]
    assert ctypes.sizeof(tg.Epilogue) == 32
    assert tg.Epilogue.bias.offset == 8 and tg.Epilogue.activation.offset == 16


def test_epilogue_validation_returns_before_the_device(tg):
    """Bad epilogue arguments are refused on the host (these calls would
    otherwise need a GPU)."""
    lib = tg
    C = 0x30000000
    def call(**e):
        ep = {"alpha": 1.0, "beta": 0.0, "bias": None, "activation": 0}
        ep.update(e)
        return lib.gemm_epilogue(64, 64, 64, 0x10000000, 64, 0x20000000, 64, C, 64, 2, ep)
    assert call(activation=2) == lib.ERR_INVALID_VALUE
    assert call(activation=-1) == lib.ERR_INVALID_VALUE
    assert call(bias=0x40000002) == lib.ERR_INVALID_VALUE          # not 4-byte aligned
    assert call(bias=C + 100) == lib.ERR_ALIAS                      # inside C
    e = lib.Epilogue(alpha=1.0, beta=0.0, bias=None, activation=0)
    e.reserved[1] = 7
    assert lib.gemm_epilogue(64, 64, 64, 0x10000000, 64, 0x20000000, 64, C, 64, 2, e) == lib.ERR_INVALID_VALUE
    # empty products return before looking at anything else
    assert lib.gemm_epilogue(0, 64, 64, 0x10000000, 64, 0x20000000, 64, C, 64, 2, {"activation": 1}) == lib.OK


def test_struct_layouts_match_header(tg):
    for cls, name in ((tg.Options, "tgemm_options"), (tg.PlanInfo, "tgemm_plan_info")):
        want = header_struct_fields(name)
        got = [(f, getattr(t, "_length_", 1)) for f, t in cls._fields_]
        assert got == want, name
        assert ctypes.sizeof(cls) == 4 * sum(n for _, n in want)
    assert ctypes.sizeof(tg.Options) == 16 * 4  # the options struct keeps its size as fields are added


def test_status_strings(tg):
    for code in range(9):
        assert tg.status_string(code)
    assert tg.status_string(0) == "success"
    assert tg.status_string(99) == "unknown status"


# fake, well-aligned device addresses: planning never dereferences them
A0, B0, C0 = 0x10000000, 0x20000000, 0x30000000


def plan(tg, M, N, K, lda=None, ldb=None, ldc=None, dtype=2, A=A0, B=B0, C=C0, sms=148, ws=0, **opt):
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    ldc = N if ldc is None else ldc
    return tg.plan(M, N, K, A, lda, B, ldb, C, ldc, dtype, opt or None, sm_count=sms, workspace_bytes=ws)


def test_validation_errors(tg):
    assert plan(tg, -1, 4, 4)[0] == tg.ERR_INVALID_VALUE
    assert plan(tg, 4, 4, 4, lda=3)[0] == tg.ERR_INVALID_VALUE
    assert plan(tg, 4, 4, 4, ldb=3)[0] == tg.ERR_INVALID_VALUE
    assert plan(tg, 4, 4, 4, ldc=3)[0] == tg.ERR_INVALID_VALUE
    assert plan(tg, 4, 4, 4, dtype=7)[0] == tg.ERR_UNSUPPORTED_DTYPE
    assert plan(tg, 4, 4, 4, A=A0 + 1)[0] == tg.ERR_MISALIGNED
    assert plan(tg, 4, 4, 4, dtype=0, C=C0 + 2)[0] == tg.ERR_MISALIGNED
    assert plan(tg, 4, 4, 4, A=0)[0] == tg.ERR_INVALID_VALUE
    assert plan(tg, 4, 4, 4, C=A0 + 8)[0] == tg.ERR_ALIAS
    assert plan(tg, 4, 4, 4, C=B0)[0] == tg.ERR_ALIAS
    assert plan(tg, 1 << 31, 4, 4)[0] == tg.ERR_TOO_LARGE
    assert plan(tg, 4, 4, 4, tile_n=96)[0] == tg.ERR_INVALID_VALUE
    assert plan(tg, 4, 4, 4, tile_n=160)[0] == tg.ERR_INVALID_VALUE
    assert plan(tg, 4, 4, 4, dtype=0, kernel=tg.KERNEL_TC_TMA)[0] == tg.ERR_INVALID_VALUE
    assert plan(tg, 4, 4, 4, dtype=2, kernel=tg.KERNEL_SIMT)[0] == tg.ERR_INVALID_VALUE
    # TMA forced on rows that are not 16-byte aligned
    assert plan(tg, 4, 4, 6, kernel=tg.KERNEL_TC_TMA)[0] == tg.ERR_INVALID_VALUE
    assert plan(tg, 4, 6, 8, store_mode=1)[0] == tg.ERR_INVALID_VALUE


def test_gemm_validation_never_touches_the_gpu(tg):
    # these return before any CUDA call, so they run on a machine without a GPU
    assert tg.gemm(-1, 4, 4, A0, 4, B0, 4, C0, 4, 2, 0) == tg.ERR_INVALID_VALUE
    assert tg.gemm(4, 4, 4, A0, 4, B0, 4, A0, 4, 2, 0) == tg.ERR_ALIAS
    assert tg.gemm(4, 4, 4, A0, 4, B0, 4, C0, 4, 9, 0) == tg.ERR_UNSUPPORTED_DTYPE
    assert tg.gemm(0, 4, 4, A0, 4, B0, 4, C0, 4, 2, 0) == tg.OK   # empty: nothing to do
    assert tg.gemm(4, 0, 4, 0, 4, 0, 4, 0, 1, 2, 0) == tg.OK


def test_dispatch_aligned_uses_bulk_tensor_copies(tg):
    st, p = plan(tg, 4096, 4096, 4096, dtype=3, sms=148)
    assert st == tg.OK
    assert p.kernel == tg.KERNEL_TC_TMA and p.a_copy_bytes == 0 and p.b_copy_bytes == 0 and p.store_bytes == 0
    assert p.tile_m in (128, 192, 224, 256) and p.tile_k in (64, 128)
    assert p.tiles_m * p.tile_m >= 4096 and p.tiles_n * p.tile_n >= 4096
    assert p.ctas == min(148, p.tiles_m * p.tiles_n)
    assert p.smem_bytes <= 232448


def test_dispatch_ragged_unaligned_rows(tg):
    # 1000 x 1500 x 4096 bf16: B and C rows are 3000 bytes (8-byte granules)
    st, p = plan(tg, 1000, 1500, 4096, dtype=2)
    assert st == tg.OK
    assert p.kernel == tg.KERNEL_TC_COPY
    assert p.a_copy_bytes == 0 and p.b_copy_bytes == 8 and p.store_bytes == 8
    st, p = plan(tg, 33, 17, 7, dtype=1)  # odd everything: 2-byte granules
    assert (p.a_copy_bytes, p.b_copy_bytes, p.store_bytes) == (2, 2, 2)
    st, p = plan(tg, 64, 64, 64, dtype=2, A=A0 + 4)
    assert p.a_copy_bytes == 4 and p.b_copy_bytes == 0


def test_bulk_store_needs_16_byte_row_extent(tg):
    # rows of 780 bytes inside a 784-byte pitch: per-thread stores
    assert plan(tg, 260, 390, 304, ldc=392, ldb=392)[1].store_bytes == 16
    assert plan(tg, 260, 392, 304, ldc=400, ldb=392)[1].store_bytes == 0
    assert plan(tg, 260, 388, 304, ldc=392, ldb=392, dtype=3)[1].store_bytes == 0   # fp32: 1552 bytes


def test_pair_planning(tg):
    st, p = plan(tg, 4096, 4096, 4096, dtype=3, sms=152, swap_ab=1)
    assert st == tg.OK and p.cta_group == 2 and p.tile_m == 256 and p.ctas % 2 == 0 and p.ctas <= 152
    st, p = plan(tg, 4096, 4096, 4096, dtype=3, sms=152, cta_group=1)
    assert p.cta_group == 1 and p.tile_m == 128
    st, p = plan(tg, 300, 520, 200, dtype=2, cta_group=2, tile_n=224)
    assert st == tg.OK and (p.tiles_m, p.tiles_n, p.ctas) == (2, 3, 12)
    # pairs need bulk-tensor A rows and a pair width; B rows that are not
    # 16-byte aligned go to the pair kernel that copies B per thread
    assert plan(tg, 1000, 1500, 4096, dtype=2, cta_group=2, A=A0 + 8)[0] == tg.ERR_INVALID_VALUE
    assert plan(tg, 512, 512, 512, dtype=2, cta_group=2, tile_n=64)[0] == tg.ERR_INVALID_VALUE
    assert plan(tg, 512, 512, 512, dtype=2, cta_group=3)[0] == tg.ERR_INVALID_VALUE
    st, p = plan(tg, 1100, 1300, 330, lda=336, ldb=1304, dtype=3, cta_group=2, tile_n=256, max_ctas=6)
    assert st == tg.OK and p.ctas == 6
    st, p = plan(tg, 4096, 4096, 4096, dtype=3, cta_group=2, tile_n=256, tile_k=128)
    assert st == tg.OK and p.tile_k == 128 and p.stages == 3 and p.smem_bytes <= 232448
    assert plan(tg, 4096, 4096, 4096, dtype=3, cta_group=1, tile_k=128)[0] == tg.ERR_INVALID_VALUE
    assert plan(tg, 4096, 4096, 4096, dtype=3, tile_k=96)[0] == tg.ERR_INVALID_VALUE


def test_copy_pair_planning(tg):
    """B rows that rule out bulk-tensor copies (3000-byte pitch) with bulk-tensor
    A rows: CTA pairs, each copying half of the tile's B columns per thread."""
    st, p = plan(tg, 1000, 1500, 4096, dtype=2, sms=152)
    assert st == tg.OK and p.kernel == tg.KERNEL_TC_COPY and p.cta_group == 2 and p.cluster_ctas == 2
    assert (p.tile_m, p.tile_n, p.tiles_m, p.tiles_n, p.ctas) == (256, 128, 4, 12, 96)
    assert (p.a_copy_bytes, p.b_copy_bytes, p.store_bytes, p.tile_k) == (0, 8, 8, 64)
    assert p.smem_bytes <= 232448 and p.stages >= 3
    # forced: the one-SM copy kernel stays reachable, the pair takes 128 or 256 only
    st, p = plan(tg, 1000, 1500, 4096, dtype=2, cta_group=1)
    assert st == tg.OK and p.cta_group == 1 and p.kernel == tg.KERNEL_TC_COPY
    st, p = plan(tg, 1000, 1500, 4096, dtype=2, cta_group=2, tile_n=256)
    assert st == tg.OK and (p.tile_n, p.tiles_n, p.ctas) == (256, 6, 48)
    assert plan(tg, 1000, 1500, 4096, dtype=2, cta_group=2, tile_n=192)[0] == tg.ERR_INVALID_VALUE
    assert plan(tg, 1000, 1500, 4096, dtype=2, cta_group=2, tile_k=128)[0] == tg.ERR_INVALID_VALUE
    assert plan(tg, 1000, 1500, 4096, dtype=2, cta_group=2, store_mode=1)[0] == tg.ERR_INVALID_VALUE
    # aligned operands forced through copies in pairs: A keeps bulk-tensor loads
    st, p = plan(tg, 512, 512, 512, dtype=2, kernel=tg.KERNEL_TC_COPY, cta_group=2, tile_n=128)
    assert st == tg.OK and p.cta_group == 2 and (p.a_copy_bytes, p.b_copy_bytes) == (0, 16) and p.store_bytes != 0
    # a CTA cap bounds the pairs
    st, p = plan(tg, 1000, 1500, 4096, dtype=2, cta_group=2, max_ctas=10)
    assert st == tg.OK and p.ctas == 10


def test_copy_pair_stream_k_planning(tg):
    """The ragged product's 48 pair tiles on 76 pairs: with stream_k = 2 and a
    workspace, all 48 x 64 k-stages are spread over every pair; without a
    workspace (or with stream_k 0 / 1) whole tiles on 48 pairs."""
    need = 4096 + 76 * 2 * 4 * 32 * 128 * 4
    st, p = plan(tg, 1000, 1500, 4096, dtype=2, sms=152, stream_k=2, ws=need)
    assert st == tg.OK and p.kernel == tg.KERNEL_TC_COPY and p.cta_group == 2 and p.tile_n == 128
    assert (p.dp_tiles, p.sk_iters, p.ctas, p.workspace_bytes) == (0, 48 * 64, 152, need)
    for kw in ({"stream_k": 2, "ws": need - 1}, {"stream_k": 2}, {"stream_k": 1, "ws": need}, {"ws": need}):
        st, p = plan(tg, 1000, 1500, 4096, dtype=2, sms=152, **kw)
        assert st == tg.OK and (p.dp_tiles, p.sk_iters, p.ctas) == (48, 0, 96), kw
    # more tiles than pairs: the whole rounds stay whole, the remainder is split
    st, p = plan(tg, 4000, 3000, 4096, dtype=2, ldb=3004, sms=152, stream_k=2, cta_group=2, tile_n=128, ws=need)
    tiles = 16 * 24
    assert (p.dp_tiles, p.sk_iters, p.ctas) == (tiles - tiles % 76, (tiles % 76) * 64, 152)


def test_tuned_shape_table(tg):
    """Calls that leave every tuned option at 0 and match a measured shape take
    the table's options; any tuned option set, another shape, or pointers the
    entry cannot serve keep the heuristics."""
    st, p = plan(tg, 1024, 1024, 1024, dtype=1, sms=152)
    assert st == tg.OK and p.tuned == 1 and (p.cta_group, p.tile_n, p.group_m) == (1, 64, 8)
    st, p = plan(tg, 1024, 1024, 1024, dtype=1, sms=152, group_m=8)
    assert st == tg.OK and p.tuned == 0 and p.group_m == 8
    st, p = plan(tg, 1024, 1024, 1000, dtype=1, sms=152)
    assert p.tuned == 0
    st, p = plan(tg, 4096, 4096, 4096, dtype=3, sms=152)
    assert p.tuned == 1 and p.swap_ab == 1 and p.tile_m == 224
    # the 2048^3 bf16 entry asks for the swapped kernel, which needs bulk-tensor rows:
    # with 2-byte-misaligned A the table is skipped and the heuristics pick a copy kernel
    st, p = plan(tg, 2048, 2048, 2048, dtype=2, sms=152, A=A0 + 2)
    assert st == tg.OK and p.tuned == 0 and p.kernel == tg.KERNEL_TC_COPY


def test_swapped_pair_planning(tg):
    """Pairs with the MMA's operands exchanged: tile_m x 256 tiles; auto takes
    them for large bulk-tensor products and picks the height by rounds."""
    st, p = plan(tg, 4096, 4096, 4096, dtype=3, sms=152)
    assert st == tg.OK and p.swap_ab == 1 and (p.tile_m, p.tile_n) == (224, 256)
    assert (p.tiles_m, p.tiles_n, p.ctas, p.cta_group, p.cluster_ctas) == (19, 16, 152, 2, 2)
    st, p = plan(tg, 8192, 8192, 8192, dtype=2, sms=152)
    assert st == tg.OK and p.swap_ab == 1 and p.tile_m == 256 and p.group_m == 8
    st, p = plan(tg, 3072, 4096, 4096, dtype=2, sms=152)
    assert p.tuned == 0 and p.group_m == 4   # operands within half of L2
    st, p = plan(tg, 4096, 4096, 4096, dtype=2, sms=152)
    assert p.tuned == 1 and p.group_m == 4    # the table's measured raster group
    st, p = plan(tg, 4096, 4096, 4096, dtype=3, sms=152)
    assert p.tuned == 1 and p.group_m == 2 and p.tile_m == 224
    for tm in (128, 192, 224, 256):
        st, p = plan(tg, 300, 520, 200, dtype=2, swap_ab=2, tile_m=tm)
        assert st == tg.OK and p.swap_ab == 1 and p.tile_m == tm and p.tile_n == 256
    # off when asked, or when another option excludes it
    assert plan(tg, 4096, 4096, 4096, dtype=3, sms=152, swap_ab=1)[1].swap_ab == 0
    assert plan(tg, 4096, 4096, 4096, dtype=3, sms=152, tile_n=224)[1].swap_ab == 0
    # refused combinations
    for bad in ({"swap_ab": 2, "stream_k": 2}, {"swap_ab": 2, "cta_group": 1},
                {"swap_ab": 2, "tile_n": 224}, {"swap_ab": 2, "tile_m": 160}, {"tile_m": 224}, {"swap_ab": 3}):
        assert plan(tg, 4096, 4096, 4096, dtype=3, **bad)[0] == tg.ERR_INVALID_VALUE, bad
    assert plan(tg, 1000, 1500, 4096, dtype=2, swap_ab=2)[0] == tg.ERR_INVALID_VALUE  # per-thread copies


def test_batched_planning(tg):
    """A strided batch: one launch of the swapped kernel over all matrices when
    every matrix starts on a 16-byte boundary, else one launch per product."""
    A, B, C = 0x10000000, 0x40000000, 0x80000000
    M = N = K = 512
    st, p, n = tg.plan_batched(64, M, N, K, A, K, M * K, B, N, K * N, C, N, M * N, 2, sm_count=152)
    assert st == tg.OK and n == 1 and p.swap_ab == 1 and p.tile_n == 256
    assert p.dp_tiles == 64 * p.tiles_m * p.tiles_n and p.ctas == 152
    # B shared by every product (stride 0)
    st, p, n = tg.plan_batched(8, M, N, K, A, K, M * K, B, N, 0, C, N, M * N, 3, sm_count=152)
    assert st == tg.OK and n == 1
    # a stride that breaks 16-byte alignment of the later matrices: one launch each
    st, p, n = tg.plan_batched(8, M, N, K, A, K, M * K + 4, B, N, K * N, C, N, M * N, 2, sm_count=152)
    assert st == tg.OK and n == 8
    # fp32 runs the SIMT kernel once per product; batch 1 and 0
    assert tg.plan_batched(5, 64, 64, 64, A, 64, 4096, B, 64, 4096, C, 64, 4096, 0, sm_count=152)[2] == 5
    # fp32 products whose tiles are split into K halves: a zero fill and the product each
    assert tg.plan_batched(3, 1024, 1024, 1024, A, 1024, 1 << 20, B, 1024, 1 << 20, C, 1024, 1 << 20, 0,
                           sm_count=152)[2] == 6
    assert tg.plan_batched(1, M, N, K, A, K, 0, B, N, 0, C, N, 0, 2, sm_count=152)[2] == 1
    assert tg.plan_batched(0, M, N, K, A, K, 0, B, N, 0, C, N, 0, 2, sm_count=152)[2] == 0
    # options that exclude the swapped kernel loop over the products
    assert tg.plan_batched(4, M, N, K, A, K, M * K, B, N, K * N, C, N, M * N, 2, {"swap_ab": 1},
                           sm_count=152)[2] == 4
    # refused: overlapping C windows, C overlapping A's batch, negative values
    assert tg.plan_batched(4, M, N, K, A, K, M * K, B, N, K * N, C, N, M * N - 1, 2)[0] == tg.ERR_ALIAS
    assert tg.plan_batched(4, M, N, K, A, K, M * K, B, N, K * N, A + 3 * M * K * 2, N, M * N, 2)[0] == tg.ERR_ALIAS
    assert tg.plan_batched(-1, M, N, K, A, K, 0, B, N, 0, C, N, 0, 2)[0] == tg.ERR_INVALID_VALUE
    assert tg.plan_batched(2, M, N, K, A, K, -1, B, N, 0, C, N, M * N, 2)[0] == tg.ERR_INVALID_VALUE
    # the call validates on the host as well (no GPU here)
    assert tg.gemm_batched(4, M, N, K, A, K, M * K, B, N, K * N, C, N, 5, 2) == tg.ERR_ALIAS
    assert tg.gemm_batched(0, M, N, K, A, K, 0, B, N, 0, C, N, 0, 2) == tg.OK


def test_transpose_validation_returns_before_the_device(tg):
    S, D = 0x10000000, 0x20000000
    assert tg.transpose(-1, 4, S, 4, D, 4, 4) == tg.ERR_INVALID_VALUE
    assert tg.transpose(4, 4, S, 3, D, 4, 4) == tg.ERR_INVALID_VALUE     # ld_src < cols
    assert tg.transpose(4, 5, S, 5, D, 3, 4) == tg.ERR_INVALID_VALUE     # ld_dst < rows
    assert tg.transpose(4, 4, S, 4, D, 4, 8) == tg.ERR_UNSUPPORTED_DTYPE
    assert tg.transpose(4, 4, S + 2, 4, D, 4, 4) == tg.ERR_MISALIGNED
    assert tg.transpose(64, 64, S, 64, S + 4 * 64 * 10, 64, 4) == tg.ERR_ALIAS
    assert tg.transpose(4, 4, 0, 4, D, 4, 4) == tg.ERR_INVALID_VALUE
    assert tg.transpose(0, 4, S, 4, D, 1, 4) == tg.OK
    assert tg.transpose(1 << 31, 4, S, 4, D, 1 << 31, 2) == tg.ERR_TOO_LARGE


def test_gemm_host_validation_returns_before_the_device(tg):
    """Argument errors of the host-buffer product come back before any CUDA
    call (this machine has no GPU, so a call that reached CUDA would fail
    with ERR_LAUNCH or ERR_UNSUPPORTED_DEVICE instead)."""
    AH, BH, CH = 0x7000_0000, 0x7100_0000, 0x7200_0000
    DA, DB, DC = 0x1000_0000, 0x2000_0000, 0x3000_0000
    g = tg.gemm_host
    assert g(-1, 4, 4, AH, 4, BH, 4, CH, 4, 2, DA, DB, DC) == tg.ERR_INVALID_VALUE
    assert g(4, 4, 4, AH, 3, BH, 4, CH, 4, 2, DA, DB, DC) == tg.ERR_INVALID_VALUE       # lda < K
    assert g(4, 4, 4, AH, 4, BH, 4, CH, 3, 2, DA, DB, DC) == tg.ERR_INVALID_VALUE       # ldc < N
    assert g(4, 4, 4, AH, 4, BH, 4, CH, 4, 9, DA, DB, DC) == tg.ERR_UNSUPPORTED_DTYPE
    assert g(4, 4, 4, AH, 4, BH, 4, CH, 4, 2, DA, DB, DC, panels=-1) == tg.ERR_INVALID_VALUE
    assert g(4, 4, 4, 0, 4, BH, 4, CH, 4, 2, DA, DB, DC) == tg.ERR_INVALID_VALUE        # no A
    assert g(4, 4, 4, AH, 4, BH, 4, CH, 4, 2, DA, 0, DC) == tg.ERR_INVALID_VALUE        # no device B
    assert g(4, 4, 4, AH, 4, BH, 4, CH, 4, 2, DA, DB, 0) == tg.ERR_INVALID_VALUE        # no device C
    assert g(4, 4, 4, AH + 1, 4, BH, 4, CH, 4, 2, DA, DB, DC) == tg.ERR_MISALIGNED
    assert g(4, 4, 4, AH, 4, BH, 4, CH, 4, 0, DA, DB, DC + 2) == tg.ERR_MISALIGNED      # fp32 C
    assert g(64, 64, 64, AH, 64, BH, 64, CH, 64, 2, DA, DA + 64 * 64, DC) == tg.ERR_ALIAS   # dB inside dA
    assert g(64, 64, 64, AH, 64, BH, 64, CH, 64, 3, DA, DB, DB + 8) == tg.ERR_ALIAS         # dC over dB
    assert g(0, 4, 4, AH, 4, BH, 4, CH, 4, 2, DA, DB, DC) == tg.OK                      # empty: nothing to do
    assert g(1 << 31, 4, 4, AH, 4, BH, 4, CH, 4, 2, DA, DB, DC) == tg.ERR_TOO_LARGE


def test_cluster_planning(tg):
    """Tensor-core pairs run in 2-CTA clusters, one-SM tiles and the SIMT
    kernel in none; the reserved option field must stay 0."""
    st, p = plan(tg, 4096, 4096, 4096, dtype=3, sms=152)
    assert st == tg.OK and p.cluster_ctas == 2
    st, p = plan(tg, 4096, 4096, 4096, dtype=3, sms=152, cta_group=2, swap_ab=1)
    assert st == tg.OK and p.cluster_ctas == 2 and p.swap_ab == 0
    st, p = plan(tg, 4096, 4096, 4096, dtype=3, sms=152, cta_group=1)
    assert st == tg.OK and p.cluster_ctas == 1
    st, p = plan(tg, 300, 300, 300, dtype=0)
    assert st == tg.OK and p.cluster_ctas == 1
    for v in (1, 2, -1):
        assert plan(tg, 4096, 4096, 4096, dtype=3, reserved0=v)[0] == tg.ERR_INVALID_VALUE


def test_simt_split_planning(tg):
    """fp32: a last round of 128 x 128 tiles that fills at most half of the
    2 x SMs resident CTA slots is split into K halves (two CTAs per tile)."""
    # 4096^3 on 152 SMs: 1024 tiles, 3 full rounds of 304, 112 left -> 224 halves
    st, p = plan(tg, 4096, 4096, 4096, dtype=0, sms=152)
    assert st == tg.OK and p.kernel == tg.KERNEL_SIMT
    assert (p.tiles_m, p.tiles_n, p.dp_tiles, p.ctas) == (32, 32, 912, 1136)
    # 2048^3: 256 tiles in one round of 304 slots; halves would not fit in one round
    st, p = plan(tg, 2048, 2048, 2048, dtype=0, sms=152)
    assert (p.dp_tiles, p.ctas) == (256, 256)
    # 1024^3: 64 tiles, all split
    st, p = plan(tg, 1024, 1024, 1024, dtype=0, sms=152)
    assert (p.dp_tiles, p.ctas) == (0, 128)
    # auto needs K >= 256 (16 stages); simt_split = 2 needs two stages
    assert plan(tg, 64, 64, 64, dtype=0, sms=2)[1].ctas == 1
    assert plan(tg, 64, 64, 64, dtype=0, sms=152, simt_split=2)[1].ctas == 2
    assert plan(tg, 64, 64, 16, dtype=0, sms=152, simt_split=2)[1].ctas == 1
    assert plan(tg, 4096, 4096, 4096, dtype=0, sms=152, simt_split=1)[1].ctas == 1024
    # a remainder above half of the slots stays whole: 3072^3 -> 576 = 304 + 272
    st, p = plan(tg, 3072, 3072, 3072, dtype=0, sms=152, simt_split=2)
    assert (p.dp_tiles, p.ctas) == (576, 576)
    assert plan(tg, 64, 64, 64, dtype=0, simt_split=3)[0] == tg.ERR_INVALID_VALUE
    assert plan(tg, 64, 64, 64, dtype=0, simt_split=-1)[0] == tg.ERR_INVALID_VALUE
    assert plan(tg, 256, 256, 256, dtype=2, simt_split=2)[0] == tg.ERR_INVALID_VALUE


def test_simt_small_product_planning(tg):
    """fp32 products whose 128 x 128 tiles would fill at most an eighth of the
    SMs, with K <= 2048, take the small-product kernel: 32 x 32 tiles, 32-deep
    stages in a 4-stage ring, one CTA per tile."""
    st, p = plan(tg, 64, 64, 64, dtype=0, sms=152)
    assert st == tg.OK and p.kernel == tg.KERNEL_SIMT
    assert (p.tile_m, p.tile_n, p.tile_k, p.stages, p.ctas, p.dp_tiles) == (32, 32, 32, 4, 4, 4)
    assert plan(tg, 512, 512, 512, dtype=0, sms=152)[1].ctas == 256            # 16 big tiles x 8 <= 152
    assert plan(tg, 640, 640, 640, dtype=0, sms=152)[1].tile_m == 128          # 25 big tiles: throughput kernel
    assert plan(tg, 256, 256, 4096, dtype=0, sms=152)[1].tile_m == 128         # long K: throughput kernel
    assert plan(tg, 64, 64, 64, dtype=0, sms=152, simt_split=2)[1].tile_m == 128  # a forced split
    assert plan(tg, 70, 90, 33, dtype=0, sms=152)[1].ctas == 3 * 3
    assert plan(tg, 64, 64, 64, dtype=2, sms=152)[1].tile_m != 32              # tensor-core dtypes never


def test_simt_raster_group_planning(tg):
    """The SIMT kernel walks tiles in groups of 16 tile rows by default, fewer
    when the product has fewer rows; group_m overrides."""
    assert plan(tg, 4096, 4096, 4096, dtype=0, sms=152)[1].group_m == 16
    assert plan(tg, 300, 4096, 512, dtype=0, sms=152)[1].group_m == 3
    assert plan(tg, 4096, 4096, 4096, dtype=0, sms=152, group_m=5)[1].group_m == 5


def test_simt_split_rule_on_random_shapes(tg):
    """For seeded random fp32 shapes and SM counts, the plan splits exactly the
    tiles of a last round that fills at most half of the 2 x SMs slots (auto:
    K >= 256), and the launch covers every tile once whole or twice as halves."""
    rng = np.random.default_rng(7)
    for _ in range(300):
        M, N = (int(v) for v in rng.integers(1, 6000, size=2))
        K = int(rng.integers(1, 1200))
        sms = int(rng.choice([1, 8, 76, 132, 148, 152]))
        st, p = plan(tg, M, N, K, dtype=0, sms=sms)
        assert st == tg.OK
        tiles = -(-M // 128) * -(-N // 128)
        if tiles * 8 <= sms and K <= 2048:  # the small-product kernel: one CTA per 32 x 32 tile
            small = -(-M // 32) * -(-N // 32)
            assert (p.tile_m, p.tiles_m * p.tiles_n, p.dp_tiles, p.ctas) == (32, small, small, small), (M, N, K, sms)
            continue
        slots = 2 * sms
        tail = tiles % slots
        split = 0 < tail and 2 * tail <= slots and -(-K // 16) >= 16
        assert (p.tiles_m * p.tiles_n, p.dp_tiles, p.ctas) == (
            (tiles, tiles - tail, tiles + tail) if split else (tiles, tiles, tiles)), (M, N, K, sms)


def test_dispatch_options(tg):
    st, p = plan(tg, 1024, 1024, 1024, dtype=1, tile_n=64, max_ctas=5, group_m=3, store_mode=2)
    assert st == tg.OK
    assert (p.tile_n, p.ctas, p.group_m, p.store_bytes) == (64, 5, 3, 16)
    st, p = plan(tg, 1024, 1024, 1024, dtype=1, kernel=tg.KERNEL_TC_COPY)
    assert p.kernel == tg.KERNEL_TC_COPY and p.a_copy_bytes == 16 and p.b_copy_bytes == 16
    st, p = plan(tg, 300, 300, 300, dtype=0, A=A0 + 4)
    assert p.kernel == tg.KERNEL_SIMT and p.a_copy_bytes == 4   # scalar loads
    st, p = plan(tg, 64, 64, 0, lda=1, dtype=2)
    assert st == tg.OK and p.kernel == 0   # K = 0: zero fill, no GEMM kernel


def test_tile_width_choice_fills_the_sms(tg):
    # small problems should not leave most SMs idle with 256-wide tiles
    st, p = plan(tg, 1024, 1024, 1024, dtype=1, sms=148)
    assert p.ctas >= 64
    st, p = plan(tg, 8192, 8192, 8192, dtype=2, sms=148)
    assert p.tile_n in (224, 256) and p.cta_group == 2
    # one SM per tile at 4096^3 on 152 SMs: 256-wide tiles (4 rounds) beat
    # 224-wide ones (4 full rounds of a less efficient tile) as measured
    st, p = plan(tg, 4096, 4096, 4096, dtype=3, sms=152, cta_group=1)
    assert p.tile_n == 256
    for bn in (64, 128, 192, 224, 256):
        st, p = plan(tg, 512, 512, 512, tile_n=bn)
        assert st == tg.OK and p.smem_bytes <= 232448 and p.stages >= 3


def test_stream_k_planning(tg):
    # 4096^3 on 152 SMs: 256 pair tiles on 76 pairs leave 28 tiles for the tail
    st, p = plan(tg, 4096, 4096, 4096, dtype=3, sms=152, cta_group=2, tile_n=256, stream_k=2)
    assert st == tg.OK and p.sk_iters == 0 and p.workspace_bytes == 0     # no workspace: whole tiles
    need = 4096 + 76 * 2 * 4 * 32 * 256 * 4    # the flag region, then the partial sums
    st, p = plan(tg, 4096, 4096, 4096, dtype=3, sms=152, cta_group=2, tile_n=256, ws=need)
    assert p.sk_iters == 0                                                # auto: off
    st, p = plan(tg, 4096, 4096, 4096, dtype=3, sms=152, cta_group=2, tile_n=256, ws=need, stream_k=2)
    assert st == tg.OK and p.workspace_bytes == need
    assert p.dp_tiles == 228 and p.sk_iters == 28 * (4096 // p.tile_k)
    assert p.ctas == 152
    st, p = plan(tg, 4096, 4096, 4096, dtype=3, sms=152, cta_group=2, tile_n=256, ws=need - 1, stream_k=2)
    assert p.sk_iters == 0                                                # too small: whole tiles
    st, p = plan(tg, 4096, 4096, 4096, dtype=3, sms=152, cta_group=2, tile_n=256, ws=need, stream_k=1)
    assert p.sk_iters == 0
    # fewer tiles than pairs: every tile is split, all 76 pairs work
    st, p = plan(tg, 2048, 2048, 2048, dtype=2, sms=152, cta_group=2, tile_n=256, ws=need, stream_k=2)
    assert p.dp_tiles == 0 and p.sk_iters == 64 * (2048 // p.tile_k) and p.ctas == 152
    assert plan(tg, 64, 64, 64, stream_k=3)[0] == tg.ERR_INVALID_VALUE


def _units(dp_tiles, sk_iters, kb, workers, w):
    """Python restatement of the device unit list, for the partition invariants."""
    units = [(t, 0, kb, "full") for t in range(w, dp_tiles, workers)]
    if sk_iters:
        b, e = w * sk_iters // workers, (w + 1) * sk_iters // workers
        if e > b:
            tb, te = b // kb, (e - 1) // kb
            lo, hi = b - tb * kb, min(e, (tb + 1) * kb) - tb * kb
            first = (dp_tiles + tb, lo, hi, "partial" if hi < kb else ("full" if lo == 0 else "finish"))
            if te == tb:
                units.append(first)
            else:
                last = (dp_tiles + te, 0, e - te * kb, "partial" if e - te * kb < kb else "full")
                units += [last, first]
    return units


@pytest.mark.parametrize("tiles,kb,workers", [(256, 32, 76), (64, 16, 76), (100, 7, 76), (5, 64, 3), (300, 3, 76)])
def test_stream_k_partition_covers_every_stage_once(tiles, kb, workers):
    rem = tiles % workers
    dp = tiles - rem
    sk = rem * kb
    seen = {}
    for w in range(workers):
        us = _units(dp, sk, kb, workers, w)
        assert sum(1 for u in us if u[0] >= dp) <= 2
        roles = [u[3] for u in us if u[0] >= dp]
        if "finish" in roles:
            assert roles[-1] == "finish"   # finishing last: its partial sums exist, its ring is idle
        for (t, lo, hi, role) in us:
            for k in range(lo, hi):
                assert (t, k) not in seen
                seen[(t, k)] = w
    assert len(seen) == tiles * kb
    # every split tile has exactly one finishing worker, the owner of its last stage
    for t in range(dp, tiles):
        owners = sorted({seen[(t, k)] for k in range(kb)})
        assert seen[(t, kb - 1)] == owners[-1]


def test_repack_planning(tg):
    """Operands whose rows rule out bulk-tensor copies are repacked into the
    workspace (when it holds them) and the bulk-tensor kernels read the copy;
    the first 4 KiB stay reserved for stream-K flags."""
    M, N, K = 1000, 1500, 4096
    b_bytes = K * 1504 * 2                      # pitch 1500 -> 1504 elements
    need = 4096 + (b_bytes + 255) // 256 * 256
    st, p = plan(tg, M, N, K, dtype=2, sms=152, ws=need)
    assert st == tg.OK and p.packed == 2 and p.kernel == tg.KERNEL_TC_TMA and p.b_copy_bytes == 0
    assert p.workspace_bytes == need
    # too small a workspace, repack = 1, or no workspace: the per-thread copy pairs
    for kw in ({"ws": need - 1}, {"ws": need, "repack": 1}, {}):
        st, p = plan(tg, M, N, K, dtype=2, sms=152, **kw)
        assert st == tg.OK and p.packed == 0 and p.kernel == tg.KERNEL_TC_COPY and p.b_copy_bytes == 8, kw
    # auto leaves B alone when the product reads it about once (M < 512); repack = 2 copies it
    st, p = plan(tg, 300, N, K, dtype=2, sms=152, ws=need)
    assert st == tg.OK and p.packed == 0
    st, p = plan(tg, 300, N, K, dtype=2, sms=152, ws=need, repack=2)
    assert st == tg.OK and p.packed == 2 and p.kernel == tg.KERNEL_TC_TMA
    # an unaligned A (K = 4100: 8200-byte rows) is repacked too, both in one workspace
    a_bytes = 1000 * 4104 * 2
    need2 = 4096 + (a_bytes + 255) // 256 * 256 + (4100 * 1504 * 2 + 255) // 256 * 256
    st, p = plan(tg, M, N, 4100, dtype=2, sms=152, ws=need2)
    assert st == tg.OK and p.packed == 3 and p.kernel == tg.KERNEL_TC_TMA and p.workspace_bytes == need2
    # with a stream-K split: flags, partial sums, then the copy
    st, p = plan(tg, M, N, K, dtype=2, sms=152, ws=64 << 20, stream_k=2, cta_group=2, swap_ab=1, tile_n=128)
    assert st == tg.OK and p.packed == 2 and p.sk_iters > 0
    assert p.workspace_bytes == 4096 + 76 * 2 * 4 * 32 * 128 * 4 + (b_bytes + 255) // 256 * 256
    # forced per-thread copies never repack; forced bulk-tensor copies need the copy
    st, p = plan(tg, M, N, K, dtype=2, sms=152, ws=need, kernel=tg.KERNEL_TC_COPY)
    assert st == tg.OK and p.packed == 0
    assert plan(tg, M, N, K, dtype=2, sms=152, ws=need, kernel=tg.KERNEL_TC_TMA)[1].packed == 2
    assert plan(tg, M, N, K, dtype=2, sms=152, kernel=tg.KERNEL_TC_TMA)[0] == tg.ERR_INVALID_VALUE
    for bad in ({"repack": 3}, {"repack": -1}):
        assert plan(tg, M, N, K, dtype=2, ws=need, **bad)[0] == tg.ERR_INVALID_VALUE
    # fp32 (SIMT) never repacks
    assert plan(tg, M, N, K, dtype=0, ldb=1501, ws=64 << 20)[1].packed == 0
