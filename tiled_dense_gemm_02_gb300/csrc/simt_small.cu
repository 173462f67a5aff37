// fp32 SIMT GEMM for small products: C[M,N] = A[M,K] . B[K,N], latency first.
//
// "GPU Kernel 的 Tile、Grid、Wave 与 Launch Overhead" (§1024², small matrices):
// a small product has too little work to fill the SMs, so fixed costs
// dominate.  The throughput kernel (simt_sgemm.cu, 128 x 128 tiles) would run
// a 64^3 product on one CTA that waits for DRAM once per 16-deep stage.  Here
// the block tile shrinks to 32 x 32 outputs, so the same product spreads over
// more SMs, and K is staged 32 deep through a 4-stage ring of asynchronous
// copies ("Tiling 策略与内存层次优化", §cp.async and §Double Buffering /
// Multi-Stage Pipelining): three stages are in flight before the first is
// used, so for K <= 96 the CTA waits for DRAM once.
//
// 256 threads as 16 x 16; thread (tx, ty) owns rows ty and ty + 16 and columns
// tx and tx + 16 of the tile (2 x 2 register tile, "寄存器Tiling" §1.1 at its
// smallest), so a warp's stores are two 64-byte row segments.  A is staged as
// loaded (A[m][k], rows padded to 36 floats: the two rows a warp reads at one
// k fall in different banks, each a broadcast), B as B[k][n] (16 consecutive
// floats per half-warp, the halves reading the same words).  Copies outside
// the matrix are zero-filled, so edge tiles need no masks in the K loop
// ("CUDA tile", section 四.4); stores are masked.  Each output is one fp32
// FMA chain in increasing k.
#include "simt_sgemm.h"
#include "ptx.cuh"

namespace tgemm {
namespace {

constexpr int T = kSimtSmallTile;  // 32 x 32 outputs per CTA
constexpr int KC = kSimtSmallK;    // K depth of a stage
constexpr int STAGES = 4;
constexpr int APITCH = KC + 4;     // floats per staged row of A (16-byte rows)
static_assert(T * KC == 256 * 4, "one 4-float copy of A and of B per thread per stage");

template <bool VEC, bool EPI>
__global__ void __launch_bounds__(256) simt_small_kernel(const SimtArgs p) {
  __shared__ __align__(16) float As[STAGES][T][APITCH];
  __shared__ __align__(16) float Bs[STAGES][KC][T];

  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int m0 = blockIdx.y * T, n0 = blockIdx.x * T;
  const int chunks = (p.K + KC - 1) / KC;
  // copy assignment: A row lr of the tile, k offset lc; B k-row lr, column offset lc
  const int lr = tid >> 3, lc = (tid & 7) * 4;

  auto issue = [&](int c) {
    const int st = c % STAGES;
    const int ak = c * KC + lc, am = m0 + lr;
    const int bk = c * KC + lr, bn = n0 + lc;
    const uint32_t da = ptx::smem_u32(&As[st][lr][lc]);
    const uint32_t db = ptx::smem_u32(&Bs[st][lr][lc]);
    if constexpr (VEC) {
      // 16-byte copies: rows and bases are 16-byte aligned, offsets are multiples of 4
      const int va = am < p.M ? max(0, min(4, p.K - ak)) : 0;
      ptx::cp_async<16>(da, va ? p.A + static_cast<int64_t>(am) * p.lda + ak : p.A, static_cast<uint32_t>(va * 4));
      const int vb = bk < p.K ? max(0, min(4, p.N - bn)) : 0;
      ptx::cp_async<16>(db, vb ? p.B + static_cast<int64_t>(bk) * p.ldb + bn : p.B, static_cast<uint32_t>(vb * 4));
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const bool oa = am < p.M && ak + i < p.K;
        ptx::cp_async<4>(da + 4 * i, oa ? p.A + static_cast<int64_t>(am) * p.lda + ak + i : p.A, oa ? 4u : 0u);
        const bool ob = bk < p.K && bn + i < p.N;
        ptx::cp_async<4>(db + 4 * i, ob ? p.B + static_cast<int64_t>(bk) * p.ldb + bn + i : p.B, ob ? 4u : 0u);
      }
    }
  };

#pragma unroll
  for (int c = 0; c < STAGES - 1; ++c) {
    if (c < chunks) issue(c);
    ptx::cp_async_commit();
  }
  float acc[2][2] = {{0.0f, 0.0f}, {0.0f, 0.0f}};
#pragma unroll 1
  for (int c = 0; c < chunks; ++c) {
    ptx::cp_async_wait<STAGES - 2>();  // stage c has landed (for this thread)
    __syncthreads();                   // ... for every thread; stage c - 1 is free
    if (c + STAGES - 1 < chunks) issue(c + STAGES - 1);
    ptx::cp_async_commit();
    const int st = c % STAGES;
#pragma unroll
    for (int k = 0; k < KC; ++k) {
      const float a0 = As[st][ty][k], a1 = As[st][ty + 16][k];
      const float b0 = Bs[st][k][tx], b1 = Bs[st][k][tx + 16];
      acc[0][0] = fmaf(a0, b0, acc[0][0]);
      acc[0][1] = fmaf(a0, b1, acc[0][1]);
      acc[1][0] = fmaf(a1, b0, acc[1][0]);
      acc[1][1] = fmaf(a1, b1, acc[1][1]);
    }
  }
  ptx::cp_async_wait<0>();  // no copy is left writing shared memory at exit

#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int gm = m0 + ty + 16 * i;
    if (gm >= p.M) continue;
    float* crow = p.C + static_cast<int64_t>(gm) * p.ldc;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int gn = n0 + tx + 16 * j;
      if (gn >= p.N) continue;
      float v = acc[i][j];
      if (EPI) v = epi_apply(p.epi, v, gn, [&] { return crow[gn]; });
      crow[gn] = v;
    }
  }
}

}  // namespace

cudaError_t launch_simt_small(const SimtArgs& args, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>((args.N + T - 1) / T), static_cast<unsigned>((args.M + T - 1) / T));
  const bool epi = args.epi.on != 0;
  if (args.vec)
    epi ? simt_small_kernel<true, true><<<grid, 256, 0, stream>>>(args)
        : simt_small_kernel<true, false><<<grid, 256, 0, stream>>>(args);
  else
    epi ? simt_small_kernel<false, true><<<grid, 256, 0, stream>>>(args)
        : simt_small_kernel<false, false><<<grid, 256, 0, stream>>>(args);
  return cudaGetLastError();
}

}  // namespace tgemm
