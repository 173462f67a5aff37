// Internal interfaces between the host dispatcher (api.cu) and the kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace tgemm {

// Output formats of the tensor-core epilogue.
enum OutFmt : int { OUT_F32 = 0, OUT_F16 = 1, OUT_BF16 = 2 };

// Device-side status codes written by bounded waits (0 = none).  The low byte
// names the wait that gave up.
enum WaitSite : uint32_t {
  SITE_PRODUCER_EMPTY = 1,
  SITE_MMA_FULL = 2,
  SITE_MMA_ACC_EMPTY = 3,
  SITE_EPI_ACC_FULL = 4,
  SITE_COPY_EMPTY = 5,
  SITE_DRAIN = 6,
  SITE_TEARDOWN = 7,
  SITE_SK_FLAG = 8,
  SITE_EPI_PRIOR = 9,   // epilogue: the prior C block staged for beta != 0
};
constexpr uint32_t kTimeoutFlag = 0x7E000000u;

// Fused epilogue, applied in fp32 to each accumulator value v of C[row][col]:
//   z = alpha * v (+ beta * C_prior[row][col] when beta != 0) (+ bias[col]),
//   ReLU when act == 1.  on == 0: the plain product (v as it is).
struct Epilogue {
  int on;
  int act;              // 0 none, 1 ReLU
  float alpha, beta;
  const float* bias;    // N fp32 column biases, or null
};

#ifdef __CUDACC__
// The fused epilogue on one value: alpha v (+ beta prior) (+ bias[col]), then
// ReLU, which keeps a NaN.  `prior()` loads the prior C element; it is called
// only when beta != 0, so C is never read otherwise.
template <class Prior>
__device__ __forceinline__ float epi_apply(const Epilogue& e, float v, int col, Prior prior) {
  float z = e.alpha * v;
  if (e.beta != 0.0f) z = fmaf(e.beta, prior(), z);
  if (e.bias) z += e.bias[col];
  if (e.act == 1) z = z < 0.0f ? 0.0f : z;
  return z;
}
// The same with the prior C element and the bias already loaded (bias_v is 0
// when there is no bias vector; prior is used only when beta != 0).
__device__ __forceinline__ float epi_combine(const Epilogue& e, float v, float prior, float bias_v) {
  float z = e.alpha * v;
  if (e.beta != 0.0f) z = fmaf(e.beta, prior, z);
  z += bias_v;
  if (e.act == 1) z = z < 0.0f ? 0.0f : z;
  return z;
}
#endif

struct TcArgs {
  int M, N, K;
  int tiles_m, tiles_n, num_tiles, k_blocks;
  int group_m;
  const void* A;
  int64_t lda;
  const void* B;
  int64_t ldb;
  void* C;
  int64_t ldc;
  uint32_t idesc;       // tcgen05 instruction descriptor (kind::f16)
  int out_fmt;          // OutFmt
  int a_copy;           // granule (bytes) of A's per-thread copies; 0 = TMA
  int b_copy;           // granule (bytes) of B's per-thread copies; 0 = TMA
  int store_granule;    // granule (bytes) of per-thread C stores; 0 = TMA store
  int inject_fault;
  unsigned long long timeout_ns;
  unsigned int* status; // device status word
  // Stream-K tail (CTA-pair kernel): tiles [0, dp_tiles) are computed whole,
  // round-robin over the workers; the k-stages of the remaining tiles are
  // divided evenly over all workers.  sk_iters == 0 disables it.
  int dp_tiles;
  int sk_iters;         // (num_tiles - dp_tiles) * k_blocks
  float* sk_partials;   // per worker: 2 CTAs x 4 warps x (32 rows x BN) fp32
  unsigned int* sk_flags;  // per worker, CTA and epilogue warp
  unsigned int sk_epoch;   // value a flag holds once this call's partial is written
  Epilogue epi;
  // Strided batch (swapped-operand pair kernel): tiles [b * tiles_per,
  // (b + 1) * tiles_per) belong to matrix b, whose operands start stride_*
  // elements after matrix b - 1's (a stride of 0 repeats one matrix).  A plain
  // product is a batch of one.
  int tiles_per;
  int64_t stride_a, stride_b, stride_c;
  // 1: launched as a programmatic dependent of the kernel before it on the
  // stream (the repack of an operand): the producers wait for that kernel
  // (griddep_wait) before their first load, while set-up overlaps its end.
  int pdl;
};

// Launch attributes of a tensor-core launch: the 2-CTA cluster (pairs) and, when
// args.pdl, programmatic stream serialisation.  Returns the number used.
inline int tc_launch_attrs(cudaLaunchAttribute (&attr)[2], int cluster, const TcArgs& args) {
  int n = 0;
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (args.pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  return n;
}

// Workspace of the stream-K tail for `workers` CTA pairs and tile width bn.
constexpr int64_t sk_partial_floats(int bn) { return int64_t(2) * 4 * 32 * bn; }
// Workspace layout of a stream-K split: the flags (8 words per worker) always
// take the first kSkFlagBytes, whatever the worker count and tile width, and
// the partial sums follow.  So a flag word of one call can only ever land on a
// flag word of an earlier call (whose epoch differs), never on partial sums.
constexpr int64_t kSkFlagBytes = 4096;
constexpr int kSkMaxWorkers = static_cast<int>(kSkFlagBytes / (8 * 4));
inline int64_t sk_workspace_bytes(int workers, int bn) {
  return kSkFlagBytes + int64_t(workers) * sk_partial_floats(bn) * 4;
}

// Tile shapes of the tensor-core kernel: 128 x BN output tiles, K stages of
// 64.  BN is one of 64, 128, 192, 224, 256; B is staged in 64-column atoms of
// 8 KB (the last atom of BN = 224 is half used).
constexpr int kTileM = 128;
constexpr int kTileK = 64;
constexpr int kEpiWarps = 4;
constexpr int kCopyWarps = 4;
constexpr int kSmemLimit = 232448;                 // opt-in shared memory per CTA
constexpr int kEpiBytes = kEpiWarps * 2 * 4096;    // epilogue staging
constexpr int kBarrierBytes = 256;

constexpr bool tc_valid_bn(int bn) { return bn == 64 || bn == 128 || bn == 192 || bn == 224 || bn == 256; }
constexpr int tc_b_atoms(int bn) { return (bn + 63) / 64; }
constexpr int tc_stage_bytes(int bn) { return kTileM * kTileK * 2 + tc_b_atoms(bn) * 8192; }
constexpr int tc_stages(int bn) {
  return (kSmemLimit - 1024 - kEpiBytes - kBarrierBytes) / tc_stage_bytes(bn) > 8
             ? 8
             : (kSmemLimit - 1024 - kEpiBytes - kBarrierBytes) / tc_stage_bytes(bn);
}
constexpr int tc_smem_bytes(int bn) { return 1024 + tc_stages(bn) * tc_stage_bytes(bn) + kEpiBytes + kBarrierBytes; }
// Tensor-memory columns between the two accumulator buffers (a power of two).
constexpr int tc_acc_stride(int bn) { return bn <= 64 ? 64 : (bn <= 128 ? 128 : 256); }
constexpr int tc_threads(bool copy) { return 32 * (2 + kEpiWarps + (copy ? kCopyWarps : 0)); }

// CTA-pair kernel: 256 x BN tiles, each CTA stages 128 rows of A and BN/2
// columns of B.
constexpr bool tc2_valid_bn(int bn) { return bn == 128 || bn == 192 || bn == 224 || bn == 256; }
// A stage holds `ksub` 64-deep K sub-blocks (one commit per stage).
constexpr int tc2_stage_bytes(int bn, int ksub = 1) {
  return ksub * (kTileM * kTileK * 2 + tc_b_atoms(bn / 2) * 8192);
}
// `staged`: the epilogue stages C tiles in shared memory for bulk-tensor
// stores; without staging (per-thread stores) the ring gets that space.
constexpr int tc2_epi_bytes(bool staged) { return staged ? kEpiBytes : 0; }
constexpr int tc2_stages(int bn, bool staged, int ksub = 1) {
  return (kSmemLimit - 1024 - tc2_epi_bytes(staged) - kBarrierBytes) / tc2_stage_bytes(bn, ksub) > 8
             ? 8
             : (kSmemLimit - 1024 - tc2_epi_bytes(staged) - kBarrierBytes) / tc2_stage_bytes(bn, ksub);
}
constexpr int tc2_smem_bytes(int bn, bool staged, int ksub = 1) {
  return 1024 + tc2_stages(bn, staged, ksub) * tc2_stage_bytes(bn, ksub) + tc2_epi_bytes(staged) + kBarrierBytes;
}

// CTA-pair kernel with B staged by per-thread copies (tile 256 x bn, bn 128
// or 256): its ring depth and shared memory per CTA.
int copy_pair_stage_count(int bn);
int copy_pair_smem(int bn);

// Launchers (return the cudaError_t of the launch).
cudaError_t launch_tc(int bn, bool copy, const CUtensorMap& mapA, const CUtensorMap& mapB, const CUtensorMap& mapC,
                      const TcArgs& args, int ctas, cudaStream_t stream);
// `pairs` CTA pairs (2-CTA clusters).  mapB_tail: B with a box (bn/2) % 64
// columns wide, for the last, partial 64-column atom of a CTA's bn/2 columns
// (unused when bn/2 is a multiple of 64).
cudaError_t launch_tc_pair(int bn, bool staged, int ksub, const CUtensorMap& mapA, const CUtensorMap& mapB,
                           const CUtensorMap& mapB_tail, const CUtensorMap& mapC, const TcArgs& args, int pairs,
                           cudaStream_t stream);
// CTA pairs computing TM x 256 tiles of C as tiles of C^T = B^T A^T (the MMA's
// M along C's columns, its N = tm along C's rows).  The maps are 3-D (matrix
// index last, extent 1 for an operand whose batch stride is 0): mapA's box is
// tm/2 rows of A, mapB's 64 columns x 64 k, mapC's an unswizzled 32 x 32 block.
cudaError_t launch_tc_pair_copy(int bn, const CUtensorMap& mapA, const TcArgs& args, int pairs, cudaStream_t stream);
cudaError_t launch_tc_pair_swap(int tm, int ksub, const CUtensorMap& mapA, const CUtensorMap& mapB,
                                const CUtensorMap& mapC, const TcArgs& args, int pairs, cudaStream_t stream);
// Number of CTA pairs (2-CTA clusters) of the pair kernel that can be
// resident at once.
cudaError_t tc_pair_capacity(int* pairs);
cudaError_t launch_zero_fill(void* C, int64_t rows, int64_t cols, int64_t ldc, int elem_bytes, cudaStream_t stream);
// out[j][i] = in[i][j], in rows x cols; elem_bytes 2 or 4; vec: every row of
// in and out starts on a 16-byte boundary (16-byte accesses)
cudaError_t launch_transpose(const void* in, int64_t ld_in, void* out, int64_t ld_out, int rows, int cols,
                             int elem_bytes, bool vec, cudaStream_t stream);
// K = 0 with a fused epilogue (out_fmt: OutFmt)
cudaError_t launch_epilogue_fill(void* C, int64_t rows, int64_t cols, int64_t ldc, int out_fmt, const Epilogue& e,
                                 cudaStream_t stream);

}  // namespace tgemm
