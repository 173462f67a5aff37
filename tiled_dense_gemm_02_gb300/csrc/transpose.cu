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
// HBM traffic, so the kernel is bound by HBM bandwidth, and several tiles per
// SM keep enough bytes in flight.  16-bit elements take their own kernel that
// moves them through shared memory as 32-bit pairs (below).
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

// 16-bit elements: the tile is 128 rows x 64 columns (16 KB, as the 32-bit
// tile) kept as 32-bit words (two elements of a row), so that shared memory is
// read and written a word at a time.  A word column of the tile holds two
// output rows; a thread reads one word from each of 8 consecutive tile rows
// and splits them into 8 elements of each of its two output rows (a 2 x 2
// transpose in registers with byte permutes).  Words are stored at column
// w ^ 4 in tile rows whose bit 5 is set: with a pitch of 33 words the 8
// threads that read one word column at rows 8 apart then fall in 8 different
// banks (without the swizzle, rows 32 apart share a bank).
constexpr int kRows16 = 128;          // tile rows (input rows, output columns)
constexpr int kPitch16 = TT / 2 + 1;  // words per tile row

__device__ __forceinline__ int swz16(int r, int w) { return w ^ ((r & 32) >> 3); }

template <bool VEC>
__global__ void __launch_bounds__(TTHREADS) transpose16_kernel(const uint16_t* __restrict__ in, int64_t ld_in,
                                                              uint16_t* __restrict__ out, int64_t ld_out, int rows,
                                                              int cols) {
  __shared__ uint32_t tile[kRows16 * kPitch16];
  const int r0 = blockIdx.y * kRows16;  // first row of in (first column of out)
  const int c0 = blockIdx.x * TT;       // first column of in (first row of out)
  const int tid = threadIdx.x;

  // read: 8 elements (4 words) of one tile row per thread and pass
#pragma unroll
  for (int k = 0; k < kRows16 * 8 / TTHREADS; ++k) {
    const int idx = tid + k * TTHREADS;
    const int r = idx >> 3, c = (idx & 7) * 8;
    const int gr = r0 + r, gc = c0 + c;
    uint32_t w[4];
    if (VEC && gr < rows && gc + 8 <= cols) {
      const uint4 q = *reinterpret_cast<const uint4*>(in + static_cast<int64_t>(gr) * ld_in + gc);
      w[0] = q.x;
      w[1] = q.y;
      w[2] = q.z;
      w[3] = q.w;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int64_t base = static_cast<int64_t>(gr) * ld_in + gc + 2 * i;
        const uint32_t lo = (gr < rows && gc + 2 * i < cols) ? in[base] : 0u;
        const uint32_t hi = (gr < rows && gc + 2 * i + 1 < cols) ? in[base + 1] : 0u;
        w[i] = lo | (hi << 16);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) tile[r * kPitch16 + swz16(r, c / 2 + i)] = w[i];
  }
  __syncthreads();

  // write: output rows 2 jp and 2 jp + 1, 8 elements each per pass
  const int jp = tid >> 3;
#pragma unroll
  for (int pass = 0; pass < kRows16 / 64; ++pass) {
    const int i0 = pass * 64 + (tid & 7) * 8;
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = tile[(i0 + i) * kPitch16 + swz16(i0 + i, jp)];
    uint32_t lo[4], hi[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      lo[m] = __byte_perm(w[2 * m], w[2 * m + 1], 0x5410);  // low halves: column 2 jp
      hi[m] = __byte_perm(w[2 * m], w[2 * m + 1], 0x7632);  // high halves: column 2 jp + 1
    }
    const int gi = r0 + i0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int gj = c0 + 2 * jp + h;
      if (gj >= cols) continue;
      const uint32_t* v = h ? hi : lo;
      uint16_t* dst = out + static_cast<int64_t>(gj) * ld_out + gi;
      if (VEC && gi + 8 <= rows) {
        *reinterpret_cast<uint4*>(dst) = make_uint4(v[0], v[1], v[2], v[3]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (gi + i < rows) dst[i] = static_cast<uint16_t>((i & 1) ? (v[i / 2] >> 16) : (v[i / 2] & 0xFFFFu));
      }
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
  if (elem_bytes == 2) {
    const dim3 grid((cols + TT - 1) / TT, (rows + kRows16 - 1) / kRows16);
    const uint16_t* src = static_cast<const uint16_t*>(in);
    uint16_t* dst = static_cast<uint16_t*>(out);
    if (vec)
      transpose16_kernel<true><<<grid, TTHREADS, 0, stream>>>(src, ld_in, dst, ld_out, rows, cols);
    else
      transpose16_kernel<false><<<grid, TTHREADS, 0, stream>>>(src, ld_in, dst, ld_out, rows, cols);
    return cudaGetLastError();
  }
  return cudaErrorInvalidValue;
}

}  // namespace tgemm
