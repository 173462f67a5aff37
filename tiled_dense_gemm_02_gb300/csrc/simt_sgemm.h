// fp32 SIMT kernel: launch arguments and tile shape (simt_sgemm.cu).
#pragma once
#include "tgemm_internal.h"

namespace tgemm {

struct SimtArgs {
  int M, N, K;
  const float* A;
  int64_t lda;
  const float* B;
  int64_t ldb;
  float* C;
  int64_t ldc;
  int vec;              // 1 when A/B/C rows allow 16-byte vector accesses
  int tiles_n;          // 128-column tiles per tile row (tiles are numbered row by row)
  int full_tiles;       // tiles [0, full_tiles) are computed whole by one CTA each
  int split_stage;      // k-stage dividing the two halves of each later tile
  Epilogue epi;
};

// Tile shape: 128 x 128 outputs per CTA, K stages 16 deep.
constexpr int kSimtBM = 128;
constexpr int kSimtBN = 128;
constexpr int kSimtBK = 16;

// Launches `units` CTAs: tiles [0, full_tiles) whole, then two per later tile.
cudaError_t launch_simt(const SimtArgs& args, int64_t units, cudaStream_t stream);

}  // namespace tgemm
