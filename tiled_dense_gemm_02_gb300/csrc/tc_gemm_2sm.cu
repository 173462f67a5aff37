// Tensor-core GEMM on CTA pairs (clusters of two SMs): one 256 x BN output
// tile per pair, computed by tcgen05.mma.cta_group::2 with M = 256.
//
// This is the same tiling as tc_gemm.cu one level up: the block tile grows to
// 256 x BN so that each byte staged in shared memory feeds twice the MMA work
// of the 128 x BN tile ("Tiling 策略与内存层次优化", §约束一 and the tiled
// intensity 2*TM*TN/((TM+TN)*e); "矩阵乘法中的平铺": traffic 2mnk/b falls as
// the output block grows).  Each CTA of the pair stages its own 128 rows of A
// and half of the B columns, so the pair moves (256 + BN) x 64 elements per K
// stage for a 256 x BN x 64 product, against (128 + BN) x 64 for a 128 x BN x
// 64 product on one SM: 32 KB instead of 48 KB per SM per stage at BN = 256,
// which leaves room for six stages in flight.
//
// Roles (both CTAs unless noted):
//   warp 0      bulk-tensor producer: loads this CTA's A rows and B columns;
//               completion is signalled on the leader CTA's full barrier
//   warp 1      tensor-memory allocation (both CTAs together); MMA issue by
//               one thread of the leader CTA (cluster rank 0), whose commits
//               are multicast to both CTAs' empty / accumulator-full barriers
//   warps 2..5  epilogue of this CTA's 128 rows; they release the accumulator
//               buffer by arriving on the leader's accumulator-empty barrier
// Every wait is bounded (see tc_common.cuh); CTAs of a cluster only meet at
// the two cluster barriers (after set-up and before tensor memory is freed),
// which all always reach.
#include <atomic>

#include "tc_common.cuh"

namespace tgemm {
namespace {

template <int BN, bool kStaged, int KSUB>
__global__ void __launch_bounds__(32 * (2 + kEpiWarps), 1)
    tc_gemm_2sm_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                       const __grid_constant__ CUtensorMap mapB_tail,
                       const __grid_constant__ CUtensorMap mapC, const TcArgs args) {
  constexpr int BNH = BN / 2;  // B columns staged by each CTA
  constexpr int STAGES = tc2_stages(BN, kStaged, KSUB);
  constexpr int A_SUB = kTileM * kTileK * 2;           // one 64-deep K sub-block of A
  constexpr int B_SUB = tc_b_atoms(BNH) * 8192;        // one 64-deep K sub-block of B
  constexpr int A_BYTES = KSUB * A_SUB;
  constexpr int B_BYTES = KSUB * B_SUB;
  // A CTA's BN/2 columns of B are whole 64-column atoms plus, for BN = 192 and
  // 224, a last atom of which only B_TAIL columns belong to the tile: that one
  // comes through mapB_tail, whose box is B_TAIL columns wide, so no column of
  // the neighbouring tile is fetched (the atom's other columns are never read).
  constexpr int B_FULL = BNH / 64;
  constexpr int B_TAIL = BNH % 64;
  constexpr int B_LOAD = KSUB * BNH * kTileK * 2;  // bytes of B a CTA receives per stage
  constexpr int ACC = 256;
  constexpr uint32_t TMEM_COLS = 512;
  static_assert(tc2_valid_bn(BN), "pair tile width");
  static_assert(tc2_smem_bytes(BN, kStaged, KSUB) <= kSmemLimit, "shared memory per CTA");
  static_assert(STAGES >= 3, "ring depth");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + STAGES * A_BYTES;
  uint8_t* sC = sB + STAGES * B_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sC + tc2_epi_bytes(kStaged));
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint64_t* epi_bar = drain + 1;  // one per epilogue warp: bulk copies of partial sums
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(epi_bar + kEpiWarps);
  static_assert((2 * STAGES + 5 + kEpiWarps) * 8 + 8 <= kBarrierBytes, "barrier area");
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const uint32_t half = rank & 1u;         // which 128 rows of the pair's tile
  const bool leader = half == 0;           // issues the pair's MMAs
  const uint32_t leader_rank = 0;
  const int worker = blockIdx.x / 2;       // persistent worker: one pair
  const int workers = gridDim.x / 2;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(ptx::smem_u32(&full[s]), 1);   // leader only: its producer's expect_tx
      ptx::mbar_init(ptx::smem_u32(&empty[s]), 1);   // the pair's MMA commit, to both CTAs
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(ptx::smem_u32(&acc_full[b]), 1);              // the pair's MMA commit, to both CTAs
      ptx::mbar_init(ptx::smem_u32(&acc_empty[b]), 2 * kEpiWarps);  // leader only: both CTAs' epilogues
    }
    ptx::mbar_init(ptx::smem_u32(drain), 1);
    for (int w = 0; w < kEpiWarps; ++w) ptx::mbar_init(ptx::smem_u32(&epi_bar[w]), 1);
    *abort_flag = 0u;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&mapA);
    ptx::tma_prefetch_desc(&mapB);
    if (B_TAIL) ptx::tma_prefetch_desc(&mapB_tail);
    if (kStaged && args.store_granule == 0) ptx::tma_prefetch_desc(&mapC);
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  // both CTAs' barriers are initialised before any remote arrive
  ptx::tc_fence_before_sync();
  ptx::cluster_sync();
  ptx::tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  const Ctl ctl{abort_flag, args.timeout_ns, args.status};

  if (warp == 0) {
    // ------------------------------------------------ bulk-tensor producer
    if (lane == 0 && !args.inject_fault) {
      ptx::griddep_wait();  // operands written by the kernel before (repack) are visible
      const uint32_t tx_pair = 2u * (A_BYTES + B_LOAD);
      int stage = 0;
      uint32_t phase = 0, filled = 0, last_parity = 0;
      bool ok = true;
      Unit u;
      for (int ui = 0; ok && worker_unit(args, worker, workers, ui, u); ++ui) {
        int mb, nb;
        tile_coords(u.tile, args, mb, nb);
        const int a_row = mb * 2 * kTileM + static_cast<int>(half) * kTileM;
        for (int kb = u.lo; kb < u.hi; ++kb) {
          if (!wait_bounded(ptx::smem_u32(&empty[stage]), phase ^ 1u, ctl, SITE_PRODUCER_EMPTY)) {
            ok = false;
            break;
          }
          const uint32_t fb_local = ptx::smem_u32(&full[stage]);
          const uint32_t fb = ptx::mapa_shared(fb_local, leader_rank);
          if (leader) ptx::mbar_arrive_expect_tx(fb_local, tx_pair);
#pragma unroll
          for (int s = 0; s < KSUB; ++s) {
            const int k0 = (kb * KSUB + s) * kTileK;  // sub-blocks past K load zeros
            ptx::tma_load_2d_pair(ptx::smem_u32(sA + stage * A_BYTES + s * A_SUB), &mapA, k0, a_row, fb);
#pragma unroll
            for (int j = 0; j < tc_b_atoms(BNH); ++j) {
              const uint32_t dst = ptx::smem_u32(sB + stage * B_BYTES + s * B_SUB + j * 8192);
              const int col = nb * BN + static_cast<int>(half) * BNH + j * 64;
              const CUtensorMap* map = j < B_FULL ? &mapB : &mapB_tail;
              ptx::tma_load_2d_pair(dst, map, col, k0, fb);
            }
          }
          filled |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Loads still in flight must land before shared memory is released: the
      // leader waits for its full barriers (both CTAs' bytes), the peer for the
      // MMA's release of each stage it filled (consumption implies arrival).
      for (int s = 0; s < STAGES; ++s)
        if ((filled >> s) & 1u) {
          const uint32_t par = (last_parity >> s) & 1u;
          if (leader)
            wait_teardown(ptx::smem_u32(&full[s]), par, ctl, SITE_TEARDOWN);
          else
            wait_teardown(ptx::smem_u32(&empty[s]), par, ctl, SITE_TEARDOWN);
        }
    }
  } else if (warp == 1) {
    // ------------------------------------------ MMA issuer (leader CTA only)
    if (leader && lane == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      Unit u;
      for (int ui = 0; ok && worker_unit(args, worker, workers, ui, u); ++ui) {
        if (!wait_bounded(ptx::smem_u32(&acc_empty[acc]), acc_phase ^ 1u, ctl, SITE_MMA_ACC_EMPTY)) break;
        ptx::tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * ACC);
        for (int kb = u.lo; kb < u.hi; ++kb) {
          if (!wait_bounded(ptx::smem_u32(&full[stage]), phase, ctl, SITE_MMA_FULL)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after_sync();
          const uint32_t a0 = ptx::smem_u32(sA + stage * A_BYTES);
          const uint32_t b0 = ptx::smem_u32(sB + stage * B_BYTES);
#pragma unroll
          for (int s = 0; s < KSUB; ++s)
#pragma unroll
            for (int k = 0; k < kTileK / 16; ++k)
              ptx::tc_mma_f16_pair(d_tmem, sw128_desc(a0 + s * A_SUB + k * 32, 16, 1024),
                                   sw128_desc(b0 + s * B_SUB + k * 2048, 8192, 1024), args.idesc,
                                   (kb != u.lo || s != 0 || k != 0) ? 1u : 0u);
          ptx::tc_commit_pair_multicast(ptx::smem_u32(&empty[stage]), 0x3);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::tc_commit_pair_multicast(ptx::smem_u32(&acc_full[acc]), 0x3);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // all pair MMAs have finished before either CTA frees tensor memory
      ptx::tc_commit_pair(ptx::smem_u32(drain));
      wait_teardown(ptx::smem_u32(drain), 0, ctl, SITE_DRAIN);
    }
    __syncwarp();
  } else {
    // --------------------------------------------------------- epilogue
    const int q = warp & 3;
    uint8_t* stage_base = sC + (warp - 2) * 2 * 4096;
    int acc = 0, sbuf = 0;
    uint32_t acc_phase = 0;
    // this warp's partial-sum slot and flag (stream-K), per worker, CTA and warp
    const int64_t slot_floats = sk_partial_floats(BN);
    const int64_t warp_off = (static_cast<int64_t>(half) * 4 + q) * 32 * BN;
    const int flag_off = static_cast<int>(half) * 4 + q;
    uint32_t epi_phase = 0;
    Unit u;
    for (int ui = 0; worker_unit(args, worker, workers, ui, u); ++ui) {
      int mb, nb;
      tile_coords(u.tile, args, mb, nb);
      if (!warp_wait(ptx::smem_u32(&acc_full[acc]), acc_phase, ctl, SITE_EPI_ACC_FULL)) break;
      ptx::tc_fence_after_sync();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * ACC);
      const int row0 = mb * 2 * kTileM + static_cast<int>(half) * kTileM + q * 32;
      if (u.role == UNIT_PARTIAL) {
        epilogue_partial<BN>(tbase, lane, args.sk_partials + worker * slot_floats + warp_off);
        __threadfence();
        __syncwarp();
        if (lane == 0) st_release_gpu(args.sk_flags + worker * 8 + flag_off, args.sk_epoch);
      } else if (u.role == UNIT_FINISH) {
        // the last unit of this worker: the ring is idle, each warp borrows a quarter
        const int first = sk_first_contributor(args, worker, workers, u);
        if (!warp_wait_flags(args.sk_flags + first * 8 + flag_off, 8, worker - first, args.sk_epoch, ctl,
                             SITE_SK_FLAG))
          break;
        constexpr int RING_SHARE = (STAGES * (A_BYTES + B_BYTES) / kEpiWarps) / 4096 * 4096;
        static_assert(RING_SHARE / 4096 >= 2, "a 16-bit output chunk needs two 4 KB slots");
        if (!epilogue_finish<BN, kStaged>(tbase, row0, nb * BN, args, &mapC, stage_base, sbuf, lane,
                                          args.sk_partials + first * slot_floats + warp_off, slot_floats,
                                          worker - first, sA + (warp - 2) * RING_SHARE, RING_SHARE / 4096,
                                          ptx::smem_u32(&epi_bar[warp - 2]), epi_phase, ctl))
          break;
      } else if (row0 < args.M) {  // a warp whose 32 rows all lie below C stores nothing
        epilogue_tile<BN, kStaged>(tbase, row0, nb * BN, args, &mapC, stage_base, sbuf, lane);
      }
      ptx::tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa_shared(ptx::smem_u32(&acc_empty[acc]), leader_rank));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    // the stores must have read shared memory before the CTA exits (their
    // writes to C complete with the kernel)
    if (lane == 0) ptx::bulk_wait_group_read<0>();
    __syncwarp();
  }

  // ------------------------------------------------------------- teardown
  ptx::tc_fence_before_sync();
  ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after_sync();
    ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

template <int BN, bool kStaged, int KSUB>
cudaError_t launch_pair(const CUtensorMap& mA, const CUtensorMap& mB, const CUtensorMap& mBt, const CUtensorMap& mC,
                        const TcArgs& args, int pairs, cudaStream_t stream) {
  constexpr int smem = tc2_smem_bytes(BN, kStaged, KSUB);
  auto kernel = tc_gemm_2sm_kernel<BN, kStaged, KSUB>;
  static std::atomic<uint64_t> done_mask{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(done_mask.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    done_mask.fetch_or(bit, std::memory_order_acq_rel);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(32 * (2 + kEpiWarps), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  cfg.attrs = attr;
  cfg.numAttrs = static_cast<unsigned>(tc_launch_attrs(attr, 2, args));
  return cudaLaunchKernelEx(&cfg, kernel, mA, mB, mBt, mC, args);
}

}  // namespace

cudaError_t launch_tc_pair(int bn, bool staged, int ksub, const CUtensorMap& mA, const CUtensorMap& mB,
                           const CUtensorMap& mBt, const CUtensorMap& mC, const TcArgs& args, int pairs,
                           cudaStream_t stream) {
#define TGEMM_PAIR_LAUNCH(BNV, ST, KS) launch_pair<BNV, ST, KS>(mA, mB, mBt, mC, args, pairs, stream)
#define TGEMM_PAIR_BN(BNV)                                                                                   \
  case BNV:                                                                                                  \
    if (ksub == 2) return staged ? TGEMM_PAIR_LAUNCH(BNV, true, 2) : TGEMM_PAIR_LAUNCH(BNV, false, 2); \
    return staged ? TGEMM_PAIR_LAUNCH(BNV, true, 1) : TGEMM_PAIR_LAUNCH(BNV, false, 1);
  switch (bn) {
    TGEMM_PAIR_BN(128)
    TGEMM_PAIR_BN(192)
    TGEMM_PAIR_BN(224)
    TGEMM_PAIR_BN(256)
    default: return cudaErrorInvalidValue;
  }
#undef TGEMM_PAIR_BN
#undef TGEMM_PAIR_LAUNCH
}

// Resident pairs of the 256-wide instantiation, which stands for all widths
// (same threads, shared memory within a few KB of the limit).
cudaError_t tc_pair_capacity(int* pairs) {
  constexpr int smem = tc2_smem_bytes(256, true, 1);
  auto kernel = tc_gemm_2sm_kernel<256, true, 1>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(32 * (2 + kEpiWarps), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(pairs, kernel, &cfg);
}

}  // namespace tgemm
