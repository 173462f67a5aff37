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
  int tiles_m, tiles_n;  // 128 x 128 tiles along M and N
  int group_m;          // raster group height in tile rows (simt_tile_coords)
  int full_tiles;       // tiles [0, full_tiles) are computed whole by one CTA each
  int split_stage;      // k-stage dividing the two halves of each later tile
  Epilogue epi;
};

// Tile shape: 128 x 128 outputs per CTA, K stages 16 deep.
constexpr int kSimtBM = 128;
constexpr int kSimtBN = 128;
constexpr int kSimtBK = 16;

// A split tile is computed as exactly two K halves, each added into C after
// the host zeroes it.  Two additions onto zero give the same float in either
// order (0 + x + y and 0 + y + x both round x + y once), so the result does
// not depend on which half lands first.  A third addend would make the sum
// depend on the order, so the split never has more than two ways.
constexpr int kSimtSplitWays = 2;
static_assert(kSimtSplitWays == 2, "the order-independence of the split holds for two halves only");

// Tile (row, column) of the t-th tile in launch order.  Tiles go in groups of
// `group_m` tile rows; within a group, down the rows of a column, then the next
// column.  A round of resident CTAs then covers about group_m rows by
// (round / group_m) columns, so its A rows and B columns stay in L2 and
// each is read from DRAM about once per group ("Tiling 策略与内存层次优化",
// 多级 Tiling 策略: the thread-block level tiles are scheduled so that the
// blocks resident together share operands).
__host__ __device__ inline void simt_tile_coords(int t, int tiles_m, int tiles_n, int group_m, int& row, int& col) {
  const int per_group = group_m * tiles_n;
  const int g = t / per_group;
  const int first = g * group_m;
  const int rows = tiles_m - first < group_m ? tiles_m - first : group_m;
  const int r = t - g * per_group;
  row = first + r % rows;
  col = r / rows;
}

// Launches `units` CTAs: tiles [0, full_tiles) whole, then two per later tile.
cudaError_t launch_simt(const SimtArgs& args, int64_t units, cudaStream_t stream);

// The small-product kernel (simt_small.cu): 32 x 32 tiles, 32-deep K stages
// through a 4-stage ring of asynchronous copies, one CTA per tile.  Uses
// M, N, K, the operands, vec and epi of `args`.
constexpr int kSimtSmallTile = 32;
constexpr int kSimtSmallK = 32;
constexpr int kSimtSmallStages = 4;
cudaError_t launch_simt_small(const SimtArgs& args, cudaStream_t stream);

}  // namespace tgemm
