// fp32 SIMT tiled GEMM: C[M,N] = A[M,K] . B[K,N] on the CUDA cores.
//
// Register tiling as laid out in "寄存器Tiling" (sections 1.1-2.1): a warp is a
// 4 x 8 grid of threads, each thread owns an 8 x 8 block of C in registers
// (64 accumulators + 8 A values + 8 B values), so one warp covers 32 x 64
// outputs.  Eight warps (4 along M x 2 along N) make a 128 x 128 CTA tile.  K is
// walked in stages of BK ("矩阵乘法中的平铺", K-splitting), double-buffered in
// shared memory: while the CTA computes on one buffer it prefetches the next
// stage into registers and then into the other buffer (one barrier per stage,
// "Double Buffering / Multi-Stage Pipelining").  The FMAs are issued as paired
// fp32 FMAs (two columns per instruction), which halves the FMA instructions;
// measured on GB300 (fp32 4096^3) that is +20 % over scalar FMAs.  With two
// CTAs per SM the kernel is at the 128-register cap and spills a few words;
// that measured faster than the spill-free unroll-by-2 schedule.
//
// Shared-memory layout, chosen for conflict-free 16-byte reads
// ("Bank Conflict 与 Swizzling"):
//   As[k][m]  A stored transposed (k-major), rows padded to 132 floats; the two
//             threads sharing an A row store interleaved groups of 4 k, so a
//             warp's transposing stores hit 32 distinct banks;
//   Bs[k][n]  B as in global memory.
// A thread's 8 rows are two runs of 4 (m, m+16) and its 8 columns two runs of
// 4 (n, n+32), so each k step is 4 LDS.128 feeding 64 FMAs (32 paired FMA
// instructions, each a pair of columns).
//
// Which lane takes which (tm, tn) sets the cost of those reads.  A 16-byte
// shared load of a warp takes two wavefronts at best, one per half-warp.
// Measured on GB300: a half-warp takes one wavefront when its lanes read
// their chunks as adjacent runs (0,0,1,1,...) or at most two chunks per
// quarter-warp, and two when its quarter-warps repeat a spread pattern
// (0,1,..,7 in both).  With tn = lane % 8 the B reads were of the second
// kind (4 wavefronts each; 3 per load with A's).  Taking tm from lane bits 0 and 3
// and tn from bits 1, 2 and 4 makes every read 2 wavefronts (2.4 % faster at
// fp32 4096^3, same bits).  A warp's store instruction still writes four
// whole 128-byte row segments.  Edge tiles load
// zeros outside the matrix and mask their stores ("CUDA tile", section 四.4).
//
// Work units: the grid is one-dimensional.  Tiles are numbered in grouped
// order (simt_tile_coords: groups of tile rows, column by column within a
// group); tiles [0, full_tiles) are computed whole, and every later tile by
// two CTAs, one per half of its k-stages ("矩阵乘法中的平铺", K-splitting taken
// across CTAs).  The host plans that split only for a last round of tiles that
// fills at most half of the resident CTA slots: split, it ends in half the
// time.  The halves add their sums into C, which the host has zeroed; two
// additions onto zero give the same float whichever lands first
// (kSimtSplitWays).
#include "simt_sgemm.h"

namespace tgemm {
namespace {

constexpr int BM = kSimtBM, BN = kSimtBN;
constexpr int BK = kSimtBK;             // K depth of a shared-memory stage
constexpr int APAD = BM + 4;
constexpr int THREADS = 256;
constexpr int NV = BK / 8;              // float4 loads of A (and of B) per thread per stage
static_assert(BK == 8 || BK == 16, "stage depth");

struct Prefetch {
  float a[NV][4];  // A[m0 + tid/2][k0 + 4*(tid%2) + 8*j .. +3]
  float b[NV][4];  // B[k0 + tid/32 + 8*j][n0 + (tid%32)*4 .. +3]
};

// Per-thread global load positions; the k offset advances by BK per stage.
struct LoadPos {
  const float* a;   // &A[m0 + tid/2][4*(tid%2)]
  const float* b;   // &B[tid/32][n0 + (tid%32)*4]
  int a_k;          // 4*(tid%2)
  int b_k;          // tid/32
  bool a_row_ok;    // m0 + tid/2 < M
  int b_cols;       // N - (n0 + (tid%32)*4)
};

template <bool VEC>
__device__ __forceinline__ void load4(const float* src, bool ok, int left, float (&d)[4]) {
  if (VEC && ok && left >= 4) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(src));
    d[0] = v.x; d[1] = v.y; d[2] = v.z; d[3] = v.w;
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] = (ok && i < left) ? __ldg(src + i) : 0.0f;
  }
}

template <bool VEC>
__device__ __forceinline__ void load_stage(const SimtArgs& p, const LoadPos& q, int k0, Prefetch& f) {
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int ka = k0 + q.a_k + 8 * j;
    load4<VEC>(q.a + k0 + 8 * j, q.a_row_ok, p.K - ka, f.a[j]);
    const int kb = k0 + q.b_k + 8 * j;
    load4<VEC>(q.b + static_cast<int64_t>(k0 + 8 * j) * p.ldb, kb < p.K, q.b_cols, f.b[j]);
  }
}

__device__ __forceinline__ void store_stage(float (*As)[APAD], float (*Bs)[BN], int tid, const Prefetch& f) {
  const int r = tid >> 1, kq = (tid & 1) * 4;
  const int br = tid >> 5, nq = (tid & 31) * 4;
#pragma unroll
  for (int j = 0; j < NV; ++j) {
#pragma unroll
    for (int i = 0; i < 4; ++i) As[kq + 8 * j + i][r] = f.a[j][i];
    *reinterpret_cast<float4*>(&Bs[br + 8 * j][nq]) = make_float4(f.b[j][0], f.b[j][1], f.b[j][2], f.b[j][3]);
  }
}

struct Frag {
  float2 a[8];  // (a_i, a_i) for the thread's 8 rows
  float b[8];
};

__device__ __forceinline__ void load_frag(const float (*As)[APAD], const float (*Bs)[BN], int k, int m_in, int n_in,
                                          Frag& f) {
  const float4 a0 = *reinterpret_cast<const float4*>(&As[k][m_in]);
  const float4 a1 = *reinterpret_cast<const float4*>(&As[k][m_in + 16]);
  const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) f.a[i] = make_float2(a[i], a[i]);
  const float4 b0 = *reinterpret_cast<const float4*>(&Bs[k][n_in]);
  const float4 b1 = *reinterpret_cast<const float4*>(&Bs[k][n_in + 32]);
  f.b[0] = b0.x; f.b[1] = b0.y; f.b[2] = b0.z; f.b[3] = b0.w;
  f.b[4] = b1.x; f.b[5] = b1.y; f.b[6] = b1.z; f.b[7] = b1.w;
}

// acc[i][j] holds columns 2j and 2j+1 of row i of the thread's 8 x 8 tile.
// Each paired FMA is two fused multiply-adds, each rounded once as fmaf is.
__device__ __forceinline__ void fma_frag(const Frag& f, float2 (&acc)[8][4]) {
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
      acc[i][j] = __ffma2_rn(f.a[i], make_float2(f.b[2 * j], f.b[2 * j + 1]), acc[i][j]);
}

// EPI: the fused epilogue is compiled in (a separate instantiation, so the
// plain product keeps its register allocation)
template <bool VEC, bool EPI>
__global__ void __launch_bounds__(THREADS, 2) simt_sgemm_kernel(const SimtArgs p) {
  __shared__ __align__(16) float As[2][BK][APAD];
  __shared__ __align__(16) float Bs[2][BK][BN];

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int wm = warp >> 1, wn = warp & 1;       // 4 x 2 warps
  // 4 x 8 threads per warp: tm from lane bits 0 and 3, tn from bits 1, 2, 4
  const int tm = (lane & 1) | ((lane >> 2) & 2), tn = ((lane >> 1) & 3) | ((lane >> 2) & 4);
  const int m_in = wm * 32 + tm * 4;             // rows m_in..+3 and m_in+16..+19
  const int n_in = wn * 64 + tn * 4;             // cols n_in..+3 and n_in+32..+35
  int tile = blockIdx.x;
  int s_begin = 0, s_end = (p.K + BK - 1) / BK;
  bool half = false;
  if (!EPI && tile >= p.full_tiles) {
    const int h = tile - p.full_tiles;
    tile = p.full_tiles + h / kSimtSplitWays;
    half = true;
    if (h % kSimtSplitWays) s_begin = p.split_stage;
    else s_end = p.split_stage;
  }
  int tile_row, tile_col;
  simt_tile_coords(tile, p.tiles_m, p.tiles_n, p.group_m, tile_row, tile_col);
  const int m0 = tile_row * BM, n0 = tile_col * BN;

  LoadPos q;
  {
    const int ar = m0 + (tid >> 1);
    q.a_k = (tid & 1) * 4;
    q.a_row_ok = ar < p.M;
    q.a = p.A + static_cast<int64_t>(q.a_row_ok ? ar : 0) * p.lda + q.a_k;
    q.b_k = tid >> 5;
    const int bn = n0 + (tid & 31) * 4;
    q.b_cols = p.N - bn;
    q.b = p.B + static_cast<int64_t>(q.b_k) * p.ldb + (q.b_cols > 0 ? bn : 0);
  }

  float2 acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = make_float2(0.0f, 0.0f);

  Prefetch f;
  if (s_begin < s_end) {
    load_stage<VEC>(p, q, s_begin * BK, f);
    store_stage(As[0], Bs[0], tid, f);
  }
  __syncthreads();

#pragma unroll 1
  for (int s = s_begin; s < s_end; ++s) {
    const int buf = (s - s_begin) & 1;
    const bool more = s + 1 < s_end;
    if (more) load_stage<VEC>(p, q, (s + 1) * BK, f);
#pragma unroll
    for (int k = 0; k < BK; ++k) {
      Frag fr;
      load_frag(As[buf], Bs[buf], k, m_in, n_in, fr);
      fma_frag(fr, acc);
    }
    if (more) store_stage(As[buf ^ 1], Bs[buf ^ 1], tid, f);
    __syncthreads();
  }

  // masked store of the 8 x 8 register tile
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int gm = m0 + m_in + (i & 3) + (i >> 2) * 16;
    if (gm >= p.M) continue;
    float* crow = p.C + static_cast<int64_t>(gm) * p.ldc;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int gn = n0 + n_in + h * 32;
      float v[4] = {acc[i][2 * h].x, acc[i][2 * h].y, acc[i][2 * h + 1].x, acc[i][2 * h + 1].y};
      if (EPI) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (gn + j < p.N) v[j] = epi_apply(p.epi, v[j], gn + j, [&] { return crow[gn + j]; });
      }
      if (half) {
        // one K half of the tile: add into C (zeroed by the host)
        if (VEC && gn + 3 < p.N) {
          atomicAdd(reinterpret_cast<float4*>(crow + gn), make_float4(v[0], v[1], v[2], v[3]));
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (gn + j < p.N) atomicAdd(crow + gn + j, v[j]);
        }
      } else if (VEC && gn + 3 < p.N) {
        *reinterpret_cast<float4*>(crow + gn) = make_float4(v[0], v[1], v[2], v[3]);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (gn + j < p.N) crow[gn + j] = v[j];
      }
    }
  }
}

}  // namespace

cudaError_t launch_simt(const SimtArgs& args, int64_t units, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>(units));
  const bool epi = args.epi.on != 0;
  if (args.vec)
    epi ? simt_sgemm_kernel<true, true><<<grid, THREADS, 0, stream>>>(args)
        : simt_sgemm_kernel<true, false><<<grid, THREADS, 0, stream>>>(args);
  else
    epi ? simt_sgemm_kernel<false, true><<<grid, THREADS, 0, stream>>>(args)
        : simt_sgemm_kernel<false, false><<<grid, THREADS, 0, stream>>>(args);
  return cudaGetLastError();
}

}  // namespace tgemm
