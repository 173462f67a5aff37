// fp32 SIMT tiled GEMM: C[M,N] = A[M,K] . B[K,N] on the CUDA cores.
//
// Register tiling as laid out in "寄存器Tiling" (sections 1.1-2.1): a warp is a
// 4 x 8 grid of threads, each thread owns an 8 x 8 block of C in registers
// (64 accumulators + 8 A values + 8 B values), so one warp covers 32 x 64
// outputs.  Eight warps (4 along M x 2 along N) make a 128 x 128 CTA tile.  K is
// walked in stages of 8 ("矩阵乘法中的平铺", K-splitting), double-buffered in
// shared memory: while the CTA computes on one buffer it prefetches the next
// stage into registers and then into the other buffer (one barrier per stage,
// "Double Buffering / Multi-Stage Pipelining").
//
// Shared-memory layout, chosen for conflict-free 16-byte reads
// ("Bank Conflict 与 Swizzling"):
//   As[k][m]  A stored transposed (k-major), rows padded to 132 floats so the
//             transposing stores of a warp hit 32 distinct banks;
//   Bs[k][n]  B as in global memory.
// A thread's 8 rows are two runs of 4 (m, m+16) and its 8 columns two runs of
// 4 (n, n+32), so each k step is 4 LDS.128 feeding 64 FFMA.  Edge tiles load
// zeros outside the matrix and mask their stores ("CUDA tile", section 四.4).
#include "tgemm_internal.h"

namespace tgemm {
namespace {

constexpr int BM = kSimtBM, BN = kSimtBN, BK = kSimtBK;
constexpr int APAD = BM + 4;
constexpr int THREADS = 256;

struct Prefetch {
  float a[4];  // A[m0 + tid/2][k0 + (tid%2)*4 .. +3]
  float b[4];  // B[k0 + tid/32][n0 + (tid%32)*4 .. +3]
};

// Per-thread global load positions of one stage; the k offset advances by BK
// per stage (A: +BK columns, B: +BK rows).
struct LoadPos {
  const float* a;   // &A[m0 + tid/2][(tid%2)*4]
  const float* b;   // &B[tid/32][n0 + (tid%32)*4]
  int a_k;          // (tid%2)*4
  int b_k;          // tid/32
  bool a_row_ok;    // m0 + tid/2 < M
  int b_cols;       // N - (n0 + (tid%32)*4)
};

template <bool VEC>
__device__ __forceinline__ void load_stage(const SimtArgs& p, const LoadPos& q, int k0, Prefetch& f) {
  {
    const float* src = q.a + k0;
    const int left = p.K - k0 - q.a_k;  // valid columns starting at src
    if (VEC && q.a_row_ok && left >= 4) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(src));
      f.a[0] = v.x; f.a[1] = v.y; f.a[2] = v.z; f.a[3] = v.w;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) f.a[i] = (q.a_row_ok && i < left) ? __ldg(src + i) : 0.0f;
    }
  }
  {
    const bool row_ok = k0 + q.b_k < p.K;
    const float* src = q.b + static_cast<int64_t>(k0) * p.ldb;
    if (VEC && row_ok && q.b_cols >= 4) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(src));
      f.b[0] = v.x; f.b[1] = v.y; f.b[2] = v.z; f.b[3] = v.w;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) f.b[i] = (row_ok && i < q.b_cols) ? __ldg(src + i) : 0.0f;
    }
  }
}

__device__ __forceinline__ void store_stage(float (*As)[APAD], float (*Bs)[BN], int tid, const Prefetch& f) {
  const int r = tid >> 1, kq = (tid & 1) * 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) As[kq + i][r] = f.a[i];
  const int br = tid >> 5, nq = (tid & 31) * 4;
  *reinterpret_cast<float4*>(&Bs[br][nq]) = make_float4(f.b[0], f.b[1], f.b[2], f.b[3]);
}

template <bool VEC>
__global__ void __launch_bounds__(THREADS, 2) simt_sgemm_kernel(const SimtArgs p) {
  __shared__ __align__(16) float As[2][BK][APAD];
  __shared__ __align__(16) float Bs[2][BK][BN];

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int wm = warp >> 1, wn = warp & 1;       // 4 x 2 warps
  const int tm = lane >> 3, tn = lane & 7;       // 4 x 8 threads per warp
  const int m_in = wm * 32 + tm * 4;             // rows m_in..+3 and m_in+16..+19
  const int n_in = wn * 64 + tn * 4;             // cols n_in..+3 and n_in+32..+35
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;

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

  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

  const int kstages = (p.K + BK - 1) / BK;
  Prefetch f;
  if (kstages > 0) {
    load_stage<VEC>(p, q, 0, f);
    store_stage(As[0], Bs[0], tid, f);
  }
  __syncthreads();

#pragma unroll 1
  for (int s = 0; s < kstages; ++s) {
    const int buf = s & 1;
    const bool more = s + 1 < kstages;
    if (more) load_stage<VEC>(p, q, (s + 1) * BK, f);
#pragma unroll
    for (int k = 0; k < BK; ++k) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][k][m_in]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][k][m_in + 16]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][k][n_in]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][k][n_in + 32]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
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
      if (VEC && gn + 3 < p.N) {
        *reinterpret_cast<float4*>(crow + gn) =
            make_float4(acc[i][h * 4], acc[i][h * 4 + 1], acc[i][h * 4 + 2], acc[i][h * 4 + 3]);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (gn + j < p.N) crow[gn + j] = acc[i][h * 4 + j];
      }
    }
  }
}

}  // namespace

cudaError_t launch_simt(const SimtArgs& args, cudaStream_t stream) {
  dim3 grid((args.N + BN - 1) / BN, (args.M + BM - 1) / BM);
  if (args.vec)
    simt_sgemm_kernel<true><<<grid, THREADS, 0, stream>>>(args);
  else
    simt_sgemm_kernel<false><<<grid, THREADS, 0, stream>>>(args);
  return cudaGetLastError();
}

}  // namespace tgemm
