// Tiled transpose: out[j][i] = in[i][j] for an in matrix of rows x cols.
//
// "CUDA tile", section 三, uses the transpose as the case where tiling settles
// the conflict between coalesced reads and coalesced writes: a block reads a
// tile along rows, keeps it in shared memory padded by one word per row so
// that column reads do not collide in a bank, and writes it back along the
// rows of the output.  Here the tile is 64 x 64 elements (4- or 2-byte), 256
// threads per block, and global accesses are 16-byte vectors when every row of
// both matrices starts on a 16-byte boundary (scalar otherwise, and at ragged
// edges).  The work is pure data movement: 2 * rows * cols * element bytes of
// HBM traffic, so the kernel is bound by HBM bandwidth, and several 16 KB
// tiles per SM keep enough bytes in flight.
#include "tgemm_internal.h"

namespace tgemm {
namespace {

constexpr int TT = 64;        // tile edge (elements)
constexpr int TTHREADS = 256;

template <typename T>
struct Vec;  // 16 bytes of T
template <>
struct Vec<uint32_t> {
  using type = uint4;
  static constexpr int n = 4;
};
template <>
struct Vec<uint16_t> {
  using type = uint4;
  static constexpr int n = 8;
};

// Row pitch of the shared tile, in elements: one extra 4-byte word per row.
template <typename T>
constexpr int tile_pitch() {
  return TT + 4 / static_cast<int>(sizeof(T));
}

template <typename T, bool VEC>
__global__ void __launch_bounds__(TTHREADS) transpose_kernel(const T* __restrict__ in, int64_t ld_in,
                                                            T* __restrict__ out, int64_t ld_out, int rows, int cols) {
  constexpr int P = tile_pitch<T>();
  constexpr int VN = VEC ? Vec<T>::n : 1;  // elements per access
  constexpr int VPR = TT / VN;              // accesses per tile row
  constexpr int PER = TT * VPR / TTHREADS;  // accesses per thread
  __shared__ __align__(16) T tile[TT * P];

  const int r0 = blockIdx.y * TT;  // first row of in (first column of out)
  const int c0 = blockIdx.x * TT;  // first column of in (first row of out)
  const int tid = threadIdx.x;

  // read in[r0.., c0..] along its rows
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int idx = tid + k * TTHREADS;
    const int r = idx / VPR, c = (idx % VPR) * VN;
    const int gr = r0 + r, gc = c0 + c;
    T v[VN];
    if (VEC && gr < rows && gc + VN <= cols) {
      const typename Vec<T>::type q =
          *reinterpret_cast<const typename Vec<T>::type*>(in + static_cast<int64_t>(gr) * ld_in + gc);
      const T* e = reinterpret_cast<const T*>(&q);
#pragma unroll
      for (int i = 0; i < VN; ++i) v[i] = e[i];
    } else {
#pragma unroll
      for (int i = 0; i < VN; ++i)
        v[i] = (gr < rows && gc + i < cols) ? in[static_cast<int64_t>(gr) * ld_in + gc + i] : T(0);
    }
#pragma unroll
    for (int i = 0; i < VN; ++i) tile[r * P + c + i] = v[i];
  }
  __syncthreads();

  // write out[c0.., r0..] along its rows: out row j is tile column j
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int idx = tid + k * TTHREADS;
    const int j = idx / VPR, i0 = (idx % VPR) * VN;
    const int gj = c0 + j, gi = r0 + i0;
    if (gj >= cols) continue;
    T v[VN];
#pragma unroll
    for (int i = 0; i < VN; ++i) v[i] = tile[(i0 + i) * P + j];
    T* dst = out + static_cast<int64_t>(gj) * ld_out + gi;
    if (VEC && gi + VN <= rows) {
      typename Vec<T>::type q;
      T* e = reinterpret_cast<T*>(&q);
#pragma unroll
      for (int i = 0; i < VN; ++i) e[i] = v[i];
      *reinterpret_cast<typename Vec<T>::type*>(dst) = q;
    } else {
#pragma unroll
      for (int i = 0; i < VN; ++i)
        if (gi + i < rows) dst[i] = v[i];
    }
  }
}

template <typename T>
cudaError_t launch_t(const void* in, int64_t ld_in, void* out, int64_t ld_out, int rows, int cols, bool vec,
                     cudaStream_t stream) {
  const dim3 grid((cols + TT - 1) / TT, (rows + TT - 1) / TT);
  if (vec)
    transpose_kernel<T, true><<<grid, TTHREADS, 0, stream>>>(static_cast<const T*>(in), ld_in, static_cast<T*>(out),
                                                             ld_out, rows, cols);
  else
    transpose_kernel<T, false><<<grid, TTHREADS, 0, stream>>>(static_cast<const T*>(in), ld_in, static_cast<T*>(out),
                                                              ld_out, rows, cols);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_transpose(const void* in, int64_t ld_in, void* out, int64_t ld_out, int rows, int cols,
                             int elem_bytes, bool vec, cudaStream_t stream) {
  if (elem_bytes == 4) return launch_t<uint32_t>(in, ld_in, out, ld_out, rows, cols, vec, stream);
  if (elem_bytes == 2) return launch_t<uint16_t>(in, ld_in, out, ld_out, rows, cols, vec, stream);
  return cudaErrorInvalidValue;
}

}  // namespace tgemm
