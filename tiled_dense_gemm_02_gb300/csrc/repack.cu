// Row repack of a 16-bit operand into a 16-byte-aligned row pitch.
//
// Bulk-tensor (TMA) copies need every row of a matrix to start on a 16-byte
// boundary ("Tiling 策略与内存层次优化", §约束一 and §cp.async: the staging
// copies want aligned, coalesced rows).  A matrix whose pitch breaks that (a
// 3000-byte row, say) is otherwise staged by per-thread copies, whose per-stage
// signalling between the two CTAs of a pair is slow.  When the caller lends a
// workspace, the library first copies the matrix, row by row, into the
// workspace with a pitch rounded up to 8 elements, and the bulk-tensor kernels
// then read that copy.  Each element is moved as raw bits, so the product is
// unchanged; elements past `cols` in a destination row are never written (the
// tensor maps stop at `cols`).
//
// This is bandwidth-bound work (each element read once and written once): a
// grid-stride loop over 16-byte chunks of destination rows, with the source
// read in the largest granule its alignment allows (8, 4 or 2 bytes) and the
// destination written as one 16-byte store per chunk.
#include "tgemm_internal.h"
#include "ptx.cuh"

namespace tgemm {
namespace {

constexpr int kRepackUnroll = 4;  // 16-byte chunks per thread per round, all loads issued first

// One 16-byte chunk of a source row, read in granules of G bytes.
template <int G>
__device__ __forceinline__ uint4 load_chunk(const uint8_t* s) {
  if constexpr (G == 8) {
    const uint2 lo = __ldg(reinterpret_cast<const uint2*>(s));
    const uint2 hi = __ldg(reinterpret_cast<const uint2*>(s + 8));
    return make_uint4(lo.x, lo.y, hi.x, hi.y);
  } else if constexpr (G == 4) {
    const uint32_t* s4 = reinterpret_cast<const uint32_t*>(s);
    return make_uint4(__ldg(s4), __ldg(s4 + 1), __ldg(s4 + 2), __ldg(s4 + 3));
  } else {
    const uint16_t* s2 = reinterpret_cast<const uint16_t*>(s);
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      w[j] = static_cast<uint32_t>(__ldg(s2 + 2 * j)) | (static_cast<uint32_t>(__ldg(s2 + 2 * j + 1)) << 16);
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
}

template <int G>  // source granule in bytes
__global__ void __launch_bounds__(256) repack_rows_kernel(const uint8_t* __restrict__ src, int64_t src_pitch,
                                                          uint8_t* __restrict__ dst, int64_t dst_pitch, int rows,
                                                          int row_bytes) {
  // the product that reads this copy may be scheduled now: its set-up overlaps
  // this kernel, and its producers wait for it to complete before loading
  ptx::griddep_launch_dependents();
  const int chunks = (row_bytes + 15) / 16;
  const int64_t total = static_cast<int64_t>(rows) * chunks;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t base = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; base < total;
       base += stride * kRepackUnroll) {
    uint4 v[kRepackUnroll];
    int64_t doff[kRepackUnroll];
    bool whole[kRepackUnroll];
#pragma unroll
    for (int u = 0; u < kRepackUnroll; ++u) {
      const int64_t i = base + u * stride;
      whole[u] = false;
      doff[u] = -1;
      if (i < total) {
        const int r = static_cast<int>(i / chunks);
        const int c = static_cast<int>(i - static_cast<int64_t>(r) * chunks) * 16;
        const uint8_t* s = src + r * src_pitch + c;
        doff[u] = r * dst_pitch + c;
        if (c + 16 <= row_bytes) {
          whole[u] = true;
          v[u] = load_chunk<G>(s);
        } else {
          // the row's last, partial chunk: element by element
          const uint16_t* s2 = reinterpret_cast<const uint16_t*>(s);
          uint16_t* d2 = reinterpret_cast<uint16_t*>(dst + doff[u]);
          for (int j = 0; 2 * j < row_bytes - c; ++j) d2[j] = __ldg(s2 + j);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kRepackUnroll; ++u)
      if (whole[u]) *reinterpret_cast<uint4*>(dst + doff[u]) = v[u];
  }
}

}  // namespace

cudaError_t launch_repack(const void* src, int64_t ld_src, void* dst, int64_t ld_dst, int rows, int cols,
                          int src_granule, int sms, cudaStream_t stream) {
  const int row_bytes = cols * 2;
  const int64_t total = static_cast<int64_t>(rows) * ((row_bytes + 15) / 16);
  // one round of kRepackUnroll chunks per thread where the matrix allows (so
  // every thread has that many loads in flight), at most 32 blocks per SM
  const int64_t want = (total + 256 * kRepackUnroll - 1) / (256 * kRepackUnroll);
  const int64_t cap = int64_t(32) * (sms > 0 ? sms : 1);
  const int blocks = static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
  const uint8_t* s = static_cast<const uint8_t*>(src);
  uint8_t* d = static_cast<uint8_t*>(dst);
  switch (src_granule) {
    case 8:
      repack_rows_kernel<8><<<blocks, 256, 0, stream>>>(s, ld_src * 2, d, ld_dst * 2, rows, row_bytes);
      break;
    case 4:
      repack_rows_kernel<4><<<blocks, 256, 0, stream>>>(s, ld_src * 2, d, ld_dst * 2, rows, row_bytes);
      break;
    default:
      repack_rows_kernel<2><<<blocks, 256, 0, stream>>>(s, ld_src * 2, d, ld_dst * 2, rows, row_bytes);
  }
  return cudaGetLastError();
}

}  // namespace tgemm
