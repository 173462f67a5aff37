// Device helpers shared by the tensor-core kernels: bounded mbarrier waits,
// the tile scheduler's tile -> (m, n) map, shared-memory matrix descriptors of
// tcgen05, the 128-byte swizzle, the per-thread copy producers that write the
// swizzled operand layout, and epilogue conversion/store routines.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "tgemm_internal.h"

namespace tgemm {
namespace {

struct Ctl {
  volatile uint32_t* abort;
  unsigned long long timeout_ns;
  unsigned int* status;
};

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const Ctl& c, uint32_t site) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*c.abort) return false;
    if (ptx::globaltimer_ns() - t0 > c.timeout_ns) {
      *c.abort = 1u;
      atomicCAS(c.status, 0u, kTimeoutFlag | site);
      return false;
    }
  }
}

// Lane 0 waits, the warp follows its verdict.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const Ctl& c, uint32_t site) {
  int ok = 1;
  if (ptx::lane_id() == 0) ok = wait_bounded(bar, parity, c, site) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Tile id -> (m block, n block): groups of `group_m` block-rows are walked
// column by column, so CTAs running at the same time touch group_m A panels
// and few B panels.
__device__ __forceinline__ void tile_coords(int t, const TcArgs& a, int& mb, int& nb) {
  const int per_group = a.group_m * a.tiles_n;
  const int g = t / per_group;
  const int first_m = g * a.group_m;
  const int gsz = min(a.tiles_m - first_m, a.group_m);
  const int r = t - g * per_group;
  mb = first_m + r % gsz;
  nb = r / gsz;
}

// Shared-memory matrix descriptor of tcgen05 for a 128-byte-swizzled operand:
// start address, leading-dimension byte offset, stride-dimension byte offset
// (all >> 4), descriptor version 1 (bit 46) and swizzle mode 2 = 128 B.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(lbo >> 4) << 16) |
         (static_cast<uint64_t>(sbo >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// Offset of byte `cb` (0..127) of row `r` inside a 128-byte-swizzled block:
// 16-byte chunk index XOR (row mod 8).
__device__ __forceinline__ uint32_t sw128_offset(int r, int cb) {
  return static_cast<uint32_t>(r * 128 + ((((cb >> 4) ^ (r & 7)) << 4) | (cb & 15)));
}

// ---------------------------------------------------------- copy producers
// Every operand of these loops arrives as a value, so the pointers, leading
// dimensions and extents stay in registers across the copy instructions
// (read from the kernel's argument block inside the loop, they would be
// fetched again after every copy).  A thread issues ITERS copies per stage;
// where the number of granules per tile row divides the thread count, each
// thread keeps one column granule and walks rows a fixed distance apart.

// A tile: rows m0..m0+127, k0..k0+63 of row-major A -> K-major swizzled rows.
template <int G>
__device__ __forceinline__ void copy_a_tile(uint32_t sa, const uint16_t* __restrict__ A, int64_t lda, int M, int K,
                                            int m0, int k0, int ct) {
  constexpr int PER_ROW = 128 / G;  // granules per 64-element row
  constexpr int STEP = kCopyWarps * 32;
  constexpr int RS = STEP / PER_ROW;  // rows between a thread's copies
  constexpr int ITERS = kTileM / RS;
  static_assert(STEP % PER_ROW == 0, "copy layout");
  const int cb = (ct % PER_ROW) * G, r0 = ct / PER_ROW;
  const int gk = k0 + cb / 2;
  const int vcol = max(0, min(G / 2, K - gk));
  const uint16_t* src = A + static_cast<int64_t>(m0 + r0) * lda + gk;
  const int64_t step = RS * lda;
#pragma unroll 8
  for (int j = 0; j < ITERS; ++j) {
    const int r = r0 + j * RS;
    const int valid = m0 + r < M ? vcol : 0;
    const uint32_t off = sw128_offset(r, cb);
    if constexpr (G >= 4) {
      ptx::cp_async<G>(sa + off, valid ? src : A, static_cast<uint32_t>(valid * 2));
    } else {
      ptx::st_shared_u16(sa + off, valid ? *src : uint16_t(0));
    }
    src += step;
  }
}

// B tile: rows k0..k0+63, columns n0..n0+BN-1 of row-major B -> N-major
// swizzled atoms of 64 columns (8 KB each).
template <int G, int BN>
__device__ __forceinline__ void copy_b_tile(uint32_t sb, const uint16_t* __restrict__ B, int64_t ldb, int K, int N,
                                            int k0, int n0, int ct) {
  constexpr int PER_ROW = BN * 2 / G;  // granules per k-row of the tile
  constexpr int STEP = kCopyWarps * 32;
  constexpr int ITERS = kTileK * PER_ROW / STEP;
  static_assert(kTileK * PER_ROW % STEP == 0, "copy layout");
  if constexpr (STEP % PER_ROW == 0) {
    constexpr int RS = STEP / PER_ROW;
    const int cb = (ct % PER_ROW) * G, r0 = ct / PER_ROW;
    const int gn = n0 + cb / 2;
    const int vcol = max(0, min(G / 2, N - gn));
    const uint32_t atom = sb + static_cast<uint32_t>((cb >> 7) * 8192);
    const uint16_t* src = B + static_cast<int64_t>(k0 + r0) * ldb + gn;
    const int64_t step = RS * ldb;
#pragma unroll 8
    for (int j = 0; j < ITERS; ++j) {
      const int r = r0 + j * RS;
      const int valid = k0 + r < K ? vcol : 0;
      const uint32_t off = sw128_offset(r, cb & 127);
      if constexpr (G >= 4) {
        ptx::cp_async<G>(atom + off, valid ? src : B, static_cast<uint32_t>(valid * 2));
      } else {
        ptx::st_shared_u16(atom + off, valid ? *src : uint16_t(0));
      }
      src += step;
    }
  } else {
#pragma unroll 4
    for (int j = 0; j < ITERS; ++j) {
      const int idx = ct + j * STEP;
      const int r = idx / PER_ROW, cb = (idx % PER_ROW) * G;
      const int gk = k0 + r, gn = n0 + cb / 2;
      const int valid = gk < K ? max(0, min(G / 2, N - gn)) : 0;
      const uint16_t* src = valid ? B + static_cast<int64_t>(gk) * ldb + gn : B;
      const uint32_t off = static_cast<uint32_t>((cb >> 7) * 8192) + sw128_offset(r, cb & 127);
      if constexpr (G >= 4) {
        ptx::cp_async<G>(sb + off, src, static_cast<uint32_t>(valid * 2));
      } else {
        ptx::st_shared_u16(sb + off, valid ? *src : uint16_t(0));
      }
    }
  }
}

// The copy side of one stage, with the operands already in registers.
struct CopyOps {
  const uint16_t* A;
  const uint16_t* B;
  int64_t lda, ldb;
  int M, N, K;
  int a_copy, b_copy;  // granule in bytes, 0 = not copied per thread
};

__device__ __forceinline__ void copy_a_dispatch(uint32_t sa, const CopyOps& o, int m0, int k0, int ct) {
  switch (o.a_copy) {
    case 16: copy_a_tile<16>(sa, o.A, o.lda, o.M, o.K, m0, k0, ct); break;
    case 8: copy_a_tile<8>(sa, o.A, o.lda, o.M, o.K, m0, k0, ct); break;
    case 4: copy_a_tile<4>(sa, o.A, o.lda, o.M, o.K, m0, k0, ct); break;
    default: copy_a_tile<2>(sa, o.A, o.lda, o.M, o.K, m0, k0, ct); break;
  }
}

template <int BN>
__device__ __forceinline__ void copy_b_dispatch(uint32_t sb, const CopyOps& o, int k0, int n0, int ct) {
  switch (o.b_copy) {
    case 16: copy_b_tile<16, BN>(sb, o.B, o.ldb, o.K, o.N, k0, n0, ct); break;
    case 8: copy_b_tile<8, BN>(sb, o.B, o.ldb, o.K, o.N, k0, n0, ct); break;
    case 4: copy_b_tile<4, BN>(sb, o.B, o.ldb, o.K, o.N, k0, n0, ct); break;
    default: copy_b_tile<2, BN>(sb, o.B, o.ldb, o.K, o.N, k0, n0, ct); break;
  }
}

// ------------------------------------------------------------- epilogue
__device__ __forceinline__ uint32_t pack_pair(float lo, float hi, int out_fmt) {
  if (out_fmt == OUT_BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ------------------------------------------------------- fused epilogue
// The prior C[row][col] in the output format (read before this kernel writes it:
// each element is read and then written by the same thread).
__device__ __forceinline__ float load_prior(const TcArgs& a, int row, int col, int64_t c_off = 0) {
  const int64_t idx = c_off + static_cast<int64_t>(row) * a.ldc + col;
  if (a.out_fmt == OUT_F32) return static_cast<const float*>(a.C)[idx];
  const uint16_t h = static_cast<const uint16_t*>(a.C)[idx];
  if (a.out_fmt == OUT_BF16) return __uint_as_float(static_cast<uint32_t>(h) << 16);
  return __half2float(__ushort_as_half(h));
}

// The epilogue on one row's 32 fp32 values v[i] = C[row][col0 + i].  The
// prior C elements and biases are all loaded before any is used, so the loads
// overlap; elements outside C are left alone (their stores are clipped).
__device__ __forceinline__ void epi_row(float (&v)[32], int row, int col0, const TcArgs& a) {
  float prior[32], bias[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const bool in = row < a.M && col0 + i < a.N;
    prior[i] = (in && a.epi.beta != 0.0f) ? load_prior(a, row, col0 + i) : 0.0f;
    bias[i] = (in && a.epi.bias) ? a.epi.bias[col0 + i] : 0.0f;
  }
#pragma unroll
  for (int i = 0; i < 32; ++i)
    if (row < a.M && col0 + i < a.N) v[i] = epi_combine(a.epi, v[i], prior[i], bias[i]);
}
__device__ __forceinline__ void epi_row(uint32_t (&v)[32], int row, int col0, const TcArgs& a) {
  float f[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
  epi_row(f, row, col0, a);
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(f[i]);
}

// Store a packed 128-byte row segment w[0..31] to global with the widest
// access `granule` (16/8/4/2 bytes) allows; only the first `valid_bytes`
// bytes are written (element size `es`).  Fully unrolled so w stays in
// registers.
__device__ __forceinline__ void store_segment(uint8_t* dst, const uint32_t (&w)[32], int valid_bytes, int granule,
                                              int es) {
  if (valid_bytes >= 128 && granule == 16) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      reinterpret_cast<uint4*>(dst)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
  } else if (valid_bytes >= 128 && granule == 8) {
#pragma unroll
    for (int i = 0; i < 16; ++i) reinterpret_cast<uint2*>(dst)[i] = make_uint2(w[2 * i], w[2 * i + 1]);
  } else if (granule >= 4) {
    // 4-byte words while they are whole, then a trailing half word
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if (4 * i + 4 <= valid_bytes) {
        reinterpret_cast<uint32_t*>(dst)[i] = w[i];
      } else if (es == 2 && 4 * i + 2 <= valid_bytes) {
        reinterpret_cast<uint16_t*>(dst)[2 * i] = static_cast<uint16_t>(w[i] & 0xFFFFu);
      }
    }
  } else {
    // 2-byte aligned rows (16-bit output only)
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if (4 * i + 2 <= valid_bytes) reinterpret_cast<uint16_t*>(dst)[2 * i] = static_cast<uint16_t>(w[i] & 0xFFFFu);
      if (4 * i + 4 <= valid_bytes) reinterpret_cast<uint16_t*>(dst)[2 * i + 1] = static_cast<uint16_t>(w[i] >> 16);
    }
  }
}


// Bounded wait that only records a timeout (teardown paths: no abort flag).
__device__ __forceinline__ void wait_teardown(uint32_t bar, uint32_t parity, const Ctl& c, uint32_t site) {
  if (ptx::mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > c.timeout_ns) {
      atomicCAS(c.status, 0u, kTimeoutFlag | site);
      return;
    }
  }
}


// ---------------------------------------------------------------- work units
// A persistent worker (a CTA, or a CTA pair) processes a list of units: k-stages
// [lo, hi) of one output tile.  Whole tiles [0, dp_tiles) go round-robin; the
// k-stages of the remaining tiles are split evenly over all workers (stream-K),
// so the last, partial round of tiles does not leave workers idle.  A tile
// split across workers is finished by the worker holding its last k-stage,
// which adds the others' fp32 partial sums in increasing worker order: the
// result does not depend on timing.
enum UnitRole : int { UNIT_FULL = 0, UNIT_PARTIAL = 1, UNIT_FINISH = 2 };
struct Unit {
  int tile, lo, hi, role;
};

__device__ __forceinline__ void sk_range(const TcArgs& a, int w, int workers, int& b, int& e) {
  b = static_cast<int>(static_cast<int64_t>(w) * a.sk_iters / workers);
  e = static_cast<int>(static_cast<int64_t>(w + 1) * a.sk_iters / workers);
}

// The idx-th unit of worker w; false when the list is exhausted.  The host
// keeps every stream-K range at most one tile long, so a worker has at most
// two stream-K units: the start of a tile (listed first since it waits for
// nobody) and the end of the previous tile (which it finishes, listed last).
__device__ __forceinline__ bool worker_unit(const TcArgs& a, int w, int workers, int idx, Unit& u) {
  const int ndp = a.dp_tiles > w ? (a.dp_tiles - 1 - w) / workers + 1 : 0;
  if (idx < ndp) {
    u = Unit{w + idx * workers, 0, a.k_blocks, UNIT_FULL};
    return true;
  }
  idx -= ndp;
  if (a.sk_iters == 0) return false;
  int b, e;
  sk_range(a, w, workers, b, e);
  if (e <= b) return false;
  const int KB = a.k_blocks;
  const int tb = b / KB, te = (e - 1) / KB;
  Unit first{a.dp_tiles + tb, b - tb * KB, min(e, (tb + 1) * KB) - tb * KB, UNIT_PARTIAL};
  if (first.hi == KB) first.role = first.lo == 0 ? UNIT_FULL : UNIT_FINISH;
  if (te == tb) {
    if (idx != 0) return false;
    u = first;
    return true;
  }
  Unit last{a.dp_tiles + te, 0, e - te * KB, UNIT_PARTIAL};
  if (last.hi == KB) last.role = UNIT_FULL;
  // the start of the later tile first (a partial sum or a whole tile, waiting
  // for nobody), the finishing unit last: its epilogue may then use the
  // worker's idle shared-memory ring
  if (idx == 0) {
    u = last;
    return true;
  }
  if (idx == 1) {
    u = first;
    return true;
  }
  return false;
}

// Workers whose partial sums a finishing unit of worker w must add: the
// contiguous range [*first, w) whose stream-K ranges reach into the tile.
__device__ __forceinline__ int sk_first_contributor(const TcArgs& a, int w, int workers, const Unit& u) {
  const int tile_begin = (u.tile - a.dp_tiles) * a.k_blocks;
  int f = w;
  while (f > 0) {
    int b, e;
    sk_range(a, f - 1, workers, b, e);
    if (e <= tile_begin) break;
    --f;
  }
  return f;
}

__device__ __forceinline__ void st_release_gpu(unsigned int* p, unsigned int v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Lane 0 waits (bounded) until every flag[k * stride], k < n, holds `epoch`;
// then every lane acquires them.  False if the wait gave up.
__device__ __forceinline__ bool warp_wait_flags(const unsigned int* flag0, int stride, int n, unsigned int epoch,
                                                const Ctl& c, uint32_t site) {
  int ok = 1;
  if (ptx::lane_id() == 0) {
    const uint64_t t0 = ptx::globaltimer_ns();
    for (int k = 0; k < n && ok; ++k) {
      while (ld_acquire_gpu(flag0 + k * stride) != epoch) {
        if (*c.abort || ptx::globaltimer_ns() - t0 > c.timeout_ns) {
          *c.abort = 1u;
          atomicCAS(c.status, 0u, kTimeoutFlag | site);
          ok = 0;
          break;
        }
      }
    }
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok)
    for (int k = 0; k < n; ++k) (void)ld_acquire_gpu(flag0 + k * stride);
  return ok != 0;
}

// Partial-sum layout of one warp's 32 rows: 32-column sub-chunk s holds
// 8 groups of 32 lanes x float4 (4 KB), so a warp's stores and loads are
// contiguous and a sub-chunk is one bulk copy.
// Write this warp's fp32 accumulator rows (BN columns) as a partial sum.
template <int BN>
__device__ __forceinline__ void epilogue_partial(uint32_t tbase, int lane, float* dst) {
#pragma unroll 1
  for (int s = 0; s < BN / 32; ++s) {
    uint32_t w[32];
    ptx::tmem_ld_32x32b_x32(tbase + s * 32, w);
    ptx::tmem_wait_ld();
    float4* d = reinterpret_cast<float4*>(dst) + s * 256 + lane;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      __stcg(d + i * 32, make_float4(__uint_as_float(w[4 * i]), __uint_as_float(w[4 * i + 1]),
                                     __uint_as_float(w[4 * i + 2]), __uint_as_float(w[4 * i + 3])));
  }
}

// Write one output chunk of a warp's 32 rows: 128 bytes per row (32 fp32 or
// 64 16-bit columns), already converted into w.  With `tma_store` and a whole
// chunk it goes through one of the warp's two 4 KB staging buffers and a
// bulk-tensor store; otherwise (no staging, or the 32-column last chunk of a
// 16-bit tile) by masked per-thread stores.
__device__ __forceinline__ void store_chunk(const uint32_t (&w)[32], int row0, int col0, bool half, bool tma_store,
                                            const TcArgs& args, const CUtensorMap* mapC, uint8_t* stage_base,
                                            int& sbuf, int lane) {
  const int es = args.out_fmt == OUT_F32 ? 4 : 2;
  const int row = row0 + lane;
  if (tma_store && !half) {
    uint8_t* buf = stage_base + sbuf * 4096;
    if (lane == 0) ptx::bulk_wait_group_read<1>();
    __syncwarp();
#pragma unroll
    for (int ch = 0; ch < 8; ++ch)
      *reinterpret_cast<uint4*>(buf + sw128_offset(lane, ch * 16)) =
          make_uint4(w[4 * ch], w[4 * ch + 1], w[4 * ch + 2], w[4 * ch + 3]);
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      ptx::tma_store_2d(mapC, col0, row0, ptx::smem_u32(buf));
      ptx::bulk_commit_group();
    }
    sbuf ^= 1;
  } else if (row < args.M && col0 < args.N) {
    uint8_t* dst = static_cast<uint8_t*>(args.C) + (static_cast<int64_t>(row) * args.ldc + col0) * es;
    const int width = half ? 32 : 128 / es;
    const int valid = min(args.N - col0, width) * es;
    // rows are 16-byte aligned whenever bulk stores are on
    store_segment(dst, w, valid, tma_store ? 16 : args.store_granule, es);
  }
}

// fp32 values of a chunk -> the output format, 128 bytes per row in w
__device__ __forceinline__ void pack_chunk(const float (&lo)[32], const float (&hi)[32], bool half, int out_fmt,
                                           uint32_t (&w)[32]) {
  if (out_fmt == OUT_F32) {
#pragma unroll
    for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(lo[i]);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      w[i] = pack_pair(lo[2 * i], lo[2 * i + 1], out_fmt);
      w[16 + i] = half ? 0u : pack_pair(hi[2 * i], hi[2 * i + 1], out_fmt);
    }
  }
}

// v += this lane's row of one 32 x 32 fp32 partial block in shared memory
__device__ __forceinline__ void add_partial(float (&v)[32], const uint8_t* block, int lane) {
  const float4* src = reinterpret_cast<const float4*>(block) + lane;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 q = src[i * 32];
    v[4 * i] += q.x;
    v[4 * i + 1] += q.y;
    v[4 * i + 2] += q.z;
    v[4 * i + 3] += q.w;
  }
}

// Epilogue of a finishing unit: the fp32 partial sums of `n_add` contributors
// (each 32 rows x BN, as epilogue_partial lays them out: 4 KB per 32 columns)
// are brought into this warp's `slots` 4 KB slots of the idle shared-memory
// ring by bulk copies, added in contributor order to the accumulator read from
// tensor memory, converted and stored like epilogue_tile.  A round of copies
// never exceeds `slots`: several whole chunks per round when all their
// contributors fit, else one chunk per round over groups of contributors.
// `bar` is this warp's mbarrier (count 1); `bar_phase` carries its phase from
// call to call.  False if a wait gave up.
template <int BN, bool kStaged>
__device__ __forceinline__ bool epilogue_finish(uint32_t tbase, int row0, int col_base, const TcArgs& args,
                                                const CUtensorMap* mapC, uint8_t* stage_base, int& sbuf, int lane,
                                                const float* add0, int64_t add_stride, int n_add, uint8_t* ring,
                                                int slots, uint32_t bar, uint32_t& bar_phase, const Ctl& ctl) {
  const int out_fmt = args.out_fmt;
  const int es = out_fmt == OUT_F32 ? 4 : 2;
  const bool tma_store = kStaged && args.store_granule == 0;
  const int cols_per_chunk = 128 / es;
  const int spc = cols_per_chunk / 32;  // 32-column partial blocks per chunk: 1 or 2
  const int chunks = (BN + cols_per_chunk - 1) / cols_per_chunk;
  const int per_chunk = spc * n_add;
  const int group = per_chunk <= slots ? n_add : max(1, slots / spc);  // contributors per round
  const int cb = per_chunk <= slots ? max(1, slots / per_chunk) : 1;    // chunks per round
  ptx::fence_proxy_async_all();  // partial sums written by generic stores, read by bulk copies
  float lo[32], hi[32];
#pragma unroll 1
  for (int c0 = 0; c0 < chunks; c0 += cb) {
    const int c1 = min(chunks, c0 + cb);
#pragma unroll 1
    for (int k0 = 0; k0 < n_add; k0 += group) {
      const int k1 = min(n_add, k0 + group);
      __syncwarp();
      if (lane == 0) {
        ptx::fence_proxy_async_smem();  // earlier reads of the slots precede the new copies
        int blocks = 0;
        for (int c = c0; c < c1; ++c) blocks += min(spc, BN / 32 - c * spc);
        ptx::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(blocks * (k1 - k0) * 4096));
        int slot = 0;
        for (int c = c0; c < c1; ++c)
          for (int sb = 0; sb < spc && c * spc + sb < BN / 32; ++sb)
            for (int k = k0; k < k1; ++k, ++slot)
              ptx::bulk_load_g2s(ptx::smem_u32(ring + slot * 4096),
                                 add0 + k * add_stride + static_cast<int64_t>(c * spc + sb) * 1024, 4096, bar);
      }
      if (!warp_wait(bar, bar_phase, ctl, SITE_SK_FLAG)) return false;
      bar_phase ^= 1u;
      int slot = 0;
#pragma unroll 1
      for (int c = c0; c < c1; ++c) {
        const int col_in_tile = c * cols_per_chunk;
        const bool half = col_in_tile + cols_per_chunk > BN;
        const int nsub = half ? 1 : spc;
        if (k0 == 0) {  // the accumulator, on the chunk's first round
          uint32_t t[32];
          ptx::tmem_ld_32x32b_x32(tbase + col_in_tile, t);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) lo[i] = __uint_as_float(t[i]);
          if (nsub == 2) {
            ptx::tmem_ld_32x32b_x32(tbase + col_in_tile + 32, t);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) hi[i] = __uint_as_float(t[i]);
          }
        }
        for (int k = k0; k < k1; ++k, ++slot) add_partial(lo, ring + slot * 4096, lane);
        if (nsub == 2)
          for (int k = k0; k < k1; ++k, ++slot) add_partial(hi, ring + slot * 4096, lane);
        if (k1 == n_add) {
          if (args.epi.on) {
            epi_row(lo, row0 + lane, col_base + col_in_tile, args);
            if (nsub == 2) epi_row(hi, row0 + lane, col_base + col_in_tile + 32, args);
          }
          uint32_t w[32];
          pack_chunk(lo, hi, half, out_fmt, w);
          store_chunk(w, row0, col_base + col_in_tile, half, tma_store, args, mapC, stage_base, sbuf, lane);
        }
      }
    }
  }
  return true;
}

// Epilogue of one warp for one tile: read the warp's 32 tensor-memory lanes
// (rows row0 .. row0+31) of the BN accumulator columns at `tbase`, convert to
// the output format and write C columns col_base .. col_base+BN-1, by
// bulk-tensor stores through the warp's two 4 KB staging buffers or by masked
// per-thread stores.  Chunks are 128 bytes of output per row (32 fp32 or 64
// 16-bit columns); with 16-bit output and BN % 64 == 32 the last chunk is 32
// columns wide and is stored per thread.
template <int BN, bool kStaged = true>
__device__ __forceinline__ void epilogue_tile(uint32_t tbase, int row0, int col_base, const TcArgs& args,
                                              const CUtensorMap* mapC, uint8_t* stage_base, int& sbuf, int lane) {
  const int out_fmt = args.out_fmt;
  const int es = out_fmt == OUT_F32 ? 4 : 2;
  // without staging buffers every chunk goes out by per-thread stores
  const bool tma_store = kStaged && args.store_granule == 0;
  const int cols_per_chunk = 128 / es;
  const int chunks = (BN + cols_per_chunk - 1) / cols_per_chunk;
#pragma unroll 1
  for (int c = 0; c < chunks; ++c) {
    const int col_in_tile = c * cols_per_chunk;
    const bool half = col_in_tile + cols_per_chunk > BN;
    uint32_t w[32];
    const int row = row0 + lane;
    if (out_fmt == OUT_F32) {
      ptx::tmem_ld_32x32b_x32(tbase + col_in_tile, w);
      ptx::tmem_wait_ld();
      if (args.epi.on) epi_row(w, row, col_base + col_in_tile, args);
    } else {
      uint32_t lo[32], hi[32];
      ptx::tmem_ld_32x32b_x32(tbase + col_in_tile, lo);
      if (!half) ptx::tmem_ld_32x32b_x32(tbase + col_in_tile + 32, hi);
      ptx::tmem_wait_ld();
      if (args.epi.on) {
        epi_row(lo, row, col_base + col_in_tile, args);
        if (!half) epi_row(hi, row, col_base + col_in_tile + 32, args);
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        w[i] = pack_pair(__uint_as_float(lo[2 * i]), __uint_as_float(lo[2 * i + 1]), out_fmt);
        w[16 + i] = half ? 0u : pack_pair(__uint_as_float(hi[2 * i]), __uint_as_float(hi[2 * i + 1]), out_fmt);
      }
    }
    store_chunk(w, row0, col_base + col_in_tile, half, tma_store, args, mapC, stage_base, sbuf, lane);
  }
}

}  // namespace
}  // namespace tgemm
