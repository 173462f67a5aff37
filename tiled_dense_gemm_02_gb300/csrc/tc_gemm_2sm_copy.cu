// Tensor-core GEMM on CTA pairs whose B rows are not 16-byte aligned: one
// 256 x BN tile of C per pair (tcgen05.mma.cta_group::2, M = 256), A staged by
// bulk-tensor copies, B staged by per-thread async copies.
//
// Why a pair: per-thread copies are what bounds the one-SM copy kernel
// (tc_gemm.cu) when B's row pitch rules out bulk-tensor copies (a pitch of
// 3000 bytes, for example).  In a pair each CTA stages only its BN/2 columns
// of B and the MMA reads both halves, so every SM copies half the B bytes per
// FLOP of the one-SM 128 x BN tile ("Tiling 策略与内存层次优化", §约束一: a
// larger output block shares each staged operand).  A keeps its bulk-tensor
// loads, 128 rows per CTA as in tc_gemm_2sm.cu.
//
// Roles (both CTAs unless noted):
//   warp 0      bulk-tensor producer of this CTA's A rows, signalled on the
//               leader's full barrier (`.cta_group::2`)
//   warp 1      tensor-memory allocation (both CTAs); in the leader one thread
//               issues the pair's MMAs; in the other CTA one thread forwards
//               each stage's copy completion to the leader
//   warps 2..5  epilogue of this CTA's 128 rows (per-thread stores)
//   warps 6..9  per-thread copy producers of this CTA's BN/2 columns of B
// A stage is ready for the MMA once (1) both CTAs' A rows have landed (the
// leader's full barrier), (2) the leader's own copies have landed (its
// copy_done barrier, fed by asynchronous arrivals on copy completion) and (3)
// the peer's forwarder has seen its copy_done barrier complete and arrived on
// the leader's peer_ready barrier (one cluster-scope release per batch of
// landed stages; the MMA thread acquires at cluster scope).  The copies write
// through the generic proxy and the MMA reads through the async proxy, so the
// forwarder and the MMA thread each fence between the two.  The MMA's stage
// commit is multicast to both CTAs' empty barriers, which all producers of
// both CTAs wait on.
// Every wait is bounded (tc_common.cuh); the CTAs meet only at the two cluster
// barriers (after set-up and before tensor memory is freed).
//
// Stream-K split (with a caller workspace): every role walks the pair's list
// of work units (worker_unit, tc_common.cuh), k-stages [lo, hi) of one tile.
// When the tiles leave pairs idle, the k-stages of the remaining tiles are
// spread evenly over all pairs ("矩阵乘法中的平铺": splitting K into stages
// leaves the total unchanged, so the stages of one tile may run on several
// pairs).  A pair holding the start of a tile writes its fp32 partial sums to
// the workspace and releases a per-warp flag; the pair holding the tile's last
// k-stage waits for the flags, adds the partial sums in pair order (so the
// result does not depend on timing), applies the epilogue and stores C.
#include <atomic>

#include "tc_common.cuh"

namespace tgemm {
namespace {

constexpr int kCopyPairBarBytes = 512;

constexpr int copy_pair_stage_bytes(int bn) { return kTileM * kTileK * 2 + tc_b_atoms(bn / 2) * 8192; }
constexpr int copy_pair_stages(int bn) {
  return (kSmemLimit - 1024 - kCopyPairBarBytes) / copy_pair_stage_bytes(bn) > 8
             ? 8
             : (kSmemLimit - 1024 - kCopyPairBarBytes) / copy_pair_stage_bytes(bn);
}
constexpr int copy_pair_smem_bytes(int bn) {
  return 1024 + copy_pair_stages(bn) * copy_pair_stage_bytes(bn) + kCopyPairBarBytes;
}
constexpr int copy_pair_threads() { return 32 * (2 + kEpiWarps + kCopyWarps); }

// wait_bounded (tc_common.cuh) with acquire at cluster scope, for a phase that
// another CTA's release completes
__device__ __forceinline__ bool wait_bounded_cluster(uint32_t bar, uint32_t parity, const Ctl& c, uint32_t site) {
  if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
    if (*c.abort) return false;
    if (ptx::globaltimer_ns() - t0 > c.timeout_ns) {
      *c.abort = 1u;
      atomicCAS(c.status, 0u, kTimeoutFlag | site);
      return false;
    }
  }
}

template <int BN>
__global__ void __launch_bounds__(copy_pair_threads(), 1)
    tc_gemm_2sm_copy_kernel(const __grid_constant__ CUtensorMap mapA, const TcArgs args) {
  constexpr int BNH = BN / 2;  // B columns copied by each CTA
  constexpr int STAGES = copy_pair_stages(BN);
  constexpr int A_BYTES = kTileM * kTileK * 2;
  constexpr int B_BYTES = tc_b_atoms(BNH) * 8192;
  constexpr int ACC = 256;
  constexpr uint32_t TMEM_COLS = 512;
  static_assert(BN == 128 || BN == 256, "pair tile width");
  static_assert(copy_pair_smem_bytes(BN) <= kSmemLimit, "shared memory per CTA");
  static_assert(STAGES >= 3, "ring depth");
  static_assert((4 * STAGES + 5 + kEpiWarps) * 8 + 8 <= kCopyPairBarBytes, "barrier area");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + STAGES * A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * B_BYTES);  // leader: both CTAs' A rows
  uint64_t* copy_done = full + STAGES;       // this CTA's B copies (asynchronous arrivals)
  uint64_t* peer_ready = copy_done + STAGES;  // leader: the peer's B copies, forwarded
  uint64_t* empty = peer_ready + STAGES;      // multicast MMA commit
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint64_t* epi_bar = drain + 1;  // one per epilogue warp: bulk copies of partial sums
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(epi_bar + kEpiWarps);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(ptx::smem_u32(&full[s]), 1);                     // the leader's expect_tx
      ptx::mbar_init(ptx::smem_u32(&copy_done[s]), kCopyWarps * 32);  // one arrival per copy thread
      ptx::mbar_init(ptx::smem_u32(&peer_ready[s]), 1);               // the peer's forwarder
      ptx::mbar_init(ptx::smem_u32(&empty[s]), 1);                    // multicast MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(ptx::smem_u32(&acc_full[b]), 1);
      ptx::mbar_init(ptx::smem_u32(&acc_empty[b]), 2 * kEpiWarps);  // leader: both CTAs' epilogues
    }
    ptx::mbar_init(ptx::smem_u32(drain), 1);
    for (int w = 0; w < kEpiWarps; ++w) ptx::mbar_init(ptx::smem_u32(&epi_bar[w]), 1);
    *abort_flag = 0u;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) ptx::tma_prefetch_desc(&mapA);
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  // barriers of both CTAs are initialised before any remote arrive
  ptx::tc_fence_before_sync();
  ptx::cluster_sync();
  ptx::tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  const Ctl ctl{abort_flag, args.timeout_ns, args.status};

  if (warp == 0) {
    // ------------------------------------------------ bulk-tensor producer (A)
    if (lane == 0 && !args.inject_fault) {
      ptx::griddep_wait();  // operands written by the kernel before (repack) are visible
      const uint32_t tx_pair = 2u * A_BYTES;
      int stage = 0;
      uint32_t phase = 0, filled = 0, last_parity = 0;
      bool ok = true;
      Unit u;
      for (int ui = 0; ok && worker_unit(args, pair, npairs, ui, u); ++ui) {
        int mb, nb;
        tile_coords(u.tile, args, mb, nb);
        const int a_row = mb * 2 * kTileM + static_cast<int>(rank) * kTileM;
        for (int kb = u.lo; kb < u.hi; ++kb) {
          if (!wait_bounded(ptx::smem_u32(&empty[stage]), phase ^ 1u, ctl, SITE_PRODUCER_EMPTY)) {
            ok = false;
            break;
          }
          const uint32_t fb_local = ptx::smem_u32(&full[stage]);
          if (leader) ptx::mbar_arrive_expect_tx(fb_local, tx_pair);
          ptx::tma_load_2d_pair(ptx::smem_u32(sA + stage * A_BYTES), &mapA, kb * kTileK, a_row,
                                ptx::mapa_shared(fb_local, 0));
          filled |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // loads in flight land before shared memory is released: the leader
      // waits for its full barriers, the peer for the MMA's release of each
      // stage it filled (consumption implies arrival)
      for (int s = 0; s < STAGES; ++s)
        if ((filled >> s) & 1u) {
          const uint32_t par = (last_parity >> s) & 1u;
          wait_teardown(ptx::smem_u32(leader ? &full[s] : &empty[s]), par, ctl, SITE_TEARDOWN);
        }
    }
  } else if (warp == 1) {
    if (leader && lane == 0) {
      // ------------------------------------------------------- MMA issuer
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      Unit u;
      for (int ui = 0; ok && worker_unit(args, pair, npairs, ui, u); ++ui) {
        if (!wait_bounded(ptx::smem_u32(&acc_empty[acc]), acc_phase ^ 1u, ctl, SITE_MMA_ACC_EMPTY)) break;
        ptx::tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * ACC);
        for (int kb = u.lo; kb < u.hi; ++kb) {
          if (!wait_bounded(ptx::smem_u32(&full[stage]), phase, ctl, SITE_MMA_FULL) ||
              !wait_bounded(ptx::smem_u32(&copy_done[stage]), phase, ctl, SITE_MMA_FULL) ||
              !wait_bounded_cluster(ptx::smem_u32(&peer_ready[stage]), phase, ctl, SITE_MMA_FULL)) {
            ok = false;
            break;
          }
          // both CTAs' copies wrote through the generic proxy; the MMA reads through the async one
          ptx::fence_proxy_async_smem();
          ptx::tc_fence_after_sync();
          const uint32_t a0 = ptx::smem_u32(sA + stage * A_BYTES);
          const uint32_t b0 = ptx::smem_u32(sB + stage * B_BYTES);
#pragma unroll
          for (int k = 0; k < kTileK / 16; ++k)
            // A: K-major, 16 elements = 32 bytes along each swizzled row;
            // B: N-major, 16 k-rows = two 1 KB groups, atoms 8 KB apart
            ptx::tc_mma_f16_pair(d_tmem, sw128_desc(a0 + k * 32, 16, 1024), sw128_desc(b0 + k * 2048, 8192, 1024),
                                 args.idesc, (kb != u.lo || k != 0) ? 1u : 0u);
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
    } else if (!leader && lane == 0) {
      // ---------------------------------------------------------- forwarder
      // A release at cluster scope measured about 1700 cycles here with copies
      // in flight in this SM (a release per stage made the ragged bf16
      // 1000 x 1500 x 4096 product 74 us instead of 44), so one release covers
      // every stage that has landed by then: wait for the next stage, gather
      // the stages after it that are already complete, fence once, then
      // arrive on the leader's barriers of all of them.  A stage's next fill needs the
      // MMA's release of it, which needs this forward, so no stage can land
      // twice before it is forwarded.
      int total = 0;  // k-stages this pair stages, over all its units
      {
        Unit u;
        for (int ui = 0; worker_unit(args, pair, npairs, ui, u); ++ui) total += u.hi - u.lo;
      }
      const uint32_t ready0 = ptx::mapa_shared(ptx::smem_u32(&peer_ready[0]), 0);
      int stage = 0;
      uint32_t phase = 0;
      for (int done = 0; done < total;) {
        if (!wait_bounded(ptx::smem_u32(&copy_done[stage]), phase, ctl, SITE_MMA_FULL)) break;
        int n = 1, st = stage + 1 == STAGES ? 0 : stage + 1;
        uint32_t ph = stage + 1 == STAGES ? phase ^ 1u : phase;
        while (done + n < total && n < STAGES && ptx::mbar_test_wait(ptx::smem_u32(&copy_done[st]), ph)) {
          ++n;
          if (++st == STAGES) {
            st = 0;
            ph ^= 1u;
          }
        }
        // the copies wrote through the generic proxy; the MMA reads through the async one
        ptx::fence_proxy_async_smem();
        ptx::fence_acq_rel_cluster();
        for (int i = 0; i < n; ++i) {
          ptx::mbar_arrive_cluster_relaxed(ready0 + static_cast<uint32_t>(stage) * 8u);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        done += n;
      }
    }
    __syncwarp();
  } else if (warp < 2 + kEpiWarps) {
    // --------------------------------------------------------- epilogue
    const int q = warp & 3;
    int acc = 0, sbuf = 0;
    uint32_t acc_phase = 0;
    // this warp's partial-sum slot and flag (stream-K), per pair, CTA and warp
    const int64_t slot_floats = sk_partial_floats(BN);
    const int64_t warp_off = (static_cast<int64_t>(rank) * 4 + q) * 32 * BN;
    const int flag_off = static_cast<int>(rank) * 4 + q;
    uint32_t epi_phase = 0;
    Unit u;
    for (int ui = 0; worker_unit(args, pair, npairs, ui, u); ++ui) {
      int mb, nb;
      tile_coords(u.tile, args, mb, nb);
      if (!warp_wait(ptx::smem_u32(&acc_full[acc]), acc_phase, ctl, SITE_EPI_ACC_FULL)) break;
      ptx::tc_fence_after_sync();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * ACC);
      const int row0 = mb * 2 * kTileM + static_cast<int>(rank) * kTileM + q * 32;
      if (u.role == UNIT_PARTIAL) {
        epilogue_partial<BN>(tbase, lane, args.sk_partials + pair * slot_floats + warp_off);
        __threadfence();
        __syncwarp();
        if (lane == 0) st_release_gpu(args.sk_flags + pair * 8 + flag_off, args.sk_epoch);
      } else if (u.role == UNIT_FINISH) {
        // the last unit of this pair: the ring is idle, each warp borrows a share of it
        const int first = sk_first_contributor(args, pair, npairs, u);
        if (!warp_wait_flags(args.sk_flags + first * 8 + flag_off, 8, pair - first, args.sk_epoch, ctl,
                             SITE_SK_FLAG))
          break;
        constexpr int RING_SHARE = (STAGES * (A_BYTES + B_BYTES) / kEpiWarps) / 4096 * 4096;
        static_assert(RING_SHARE / 4096 >= 2, "a 16-bit output chunk needs two 4 KB slots");
        if (!epilogue_finish<BN, false>(tbase, row0, nb * BN, args, nullptr, nullptr, sbuf, lane,
                                        args.sk_partials + first * slot_floats + warp_off, slot_floats, pair - first,
                                        sA + (warp - 2) * RING_SHARE, RING_SHARE / 4096,
                                        ptx::smem_u32(&epi_bar[warp - 2]), epi_phase, ctl))
          break;
      } else if (row0 < args.M) {
        epilogue_tile<BN, false>(tbase, row0, nb * BN, args, nullptr, nullptr, sbuf, lane);
      }
      ptx::tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa_shared(ptx::smem_u32(&acc_empty[acc]), 0));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  } else {
    // -------------------------------------------------- copy producers (B)
    const int ct = threadIdx.x - (2 + kEpiWarps) * 32;
    const CopyOps ops{static_cast<const uint16_t*>(args.A), static_cast<const uint16_t*>(args.B), args.lda, args.ldb,
                      args.M, args.N, args.K, 0, args.b_copy};
    const uint32_t sB_u = ptx::smem_u32(sB);
    if (!args.inject_fault) {
      ptx::griddep_wait();
      const bool sync_arrive = ops.b_copy == 2;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      Unit u;
      for (int ui = 0; ok && worker_unit(args, pair, npairs, ui, u); ++ui) {
        int mb, nb;
        tile_coords(u.tile, args, mb, nb);
        const int n0 = nb * BN + static_cast<int>(rank) * BNH;
        for (int kb = u.lo; kb < u.hi; ++kb) {
          if (!warp_wait(ptx::smem_u32(&empty[stage]), phase ^ 1u, ctl, SITE_COPY_EMPTY)) {
            ok = false;
            break;
          }
          copy_b_dispatch<BNH>(sB_u + stage * B_BYTES, ops, kb * kTileK, n0, ct);
          const uint32_t cb = ptx::smem_u32(&copy_done[stage]);
          if (sync_arrive) {
            // 2-byte granules are plain stores: they are done, arrive now
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(cb);
          } else {
            // the arrival fires by itself once this thread's copies land
            ptx::cp_async_mbar_arrive_noinc(cb);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // no copy may still be writing shared memory when the CTA exits
      ptx::cp_async_commit();
      ptx::cp_async_wait<0>();
    }
  }

  // ------------------------------------------------------------- teardown
  ptx::tc_fence_before_sync();
  ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after_sync();
    ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

template <int BN>
cudaError_t launch_copy_pair(const CUtensorMap& mA, const TcArgs& args, int pairs, cudaStream_t stream) {
  constexpr int smem = copy_pair_smem_bytes(BN);
  auto kernel = tc_gemm_2sm_copy_kernel<BN>;
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
  cfg.blockDim = dim3(copy_pair_threads(), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  cfg.attrs = attr;
  cfg.numAttrs = static_cast<unsigned>(tc_launch_attrs(attr, 2, args));
  return cudaLaunchKernelEx(&cfg, kernel, mA, args);
}

}  // namespace

int copy_pair_stage_count(int bn) { return bn == 128 ? copy_pair_stages(128) : copy_pair_stages(256); }
int copy_pair_smem(int bn) { return bn == 128 ? copy_pair_smem_bytes(128) : copy_pair_smem_bytes(256); }

cudaError_t launch_tc_pair_copy(int bn, const CUtensorMap& mA, const TcArgs& args, int pairs, cudaStream_t stream) {
  if (bn == 128) return launch_copy_pair<128>(mA, args, pairs, stream);
  if (bn == 256) return launch_copy_pair<256>(mA, args, pairs, stream);
  return cudaErrorInvalidValue;
}

}  // namespace tgemm
