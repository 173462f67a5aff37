// Tensor-core GEMM on CTA pairs with the operand roles of the MMA exchanged:
// each pair computes a TM x 256 tile of C as the 256 x TM tile of
// C^T = B^T . A^T.
//
// Why: in the pair kernel (tc_gemm_2sm.cu) the MMA's N is C's tile width,
// and each CTA stages BN/2 columns of the N-major B in 64-column swizzle
// atoms; at BN = 192 or 224 a CTA's half ends in a partial atom, and those
// widths measured 10-16 % slower per FLOP than BN = 256 on GB300.  Here the
// MMA's M (256, split 128 + 128 over the pair) runs along C's columns, so
// each CTA stages exactly two whole atoms of B, and the MMA's N runs along
// C's rows: A is K-major, its rows come in 8-row groups, and any TM that is
// a multiple of 32 stages no waste.  The tile's height then follows the
// shape: 4096 x 4096 in 256 x 224 pair tiles is 16 x 19 = 304 tiles, exactly
// four rounds of 76 pairs (the wave arithmetic of "GPU Kernel 的 Tile、Grid、
// Wave 与 Launch Overhead", §Wave).
//
// The staging ring, barriers, roles and bounded waits are those of the pair
// kernel: warp 0 loads (bulk-tensor, `.cta_group::2`, signalled on the leader's
// full barrier), one thread of the leader issues tcgen05.mma.cta_group::2 with
// A = this stage's B columns (MN-major) and B = its A rows (K-major), warps
// 2..5 drain tensor memory.  The accumulator is transposed with respect to C:
// TMEM lane = C column, TMEM column = C row.  The epilogue therefore writes
// each 32 x 32 block of C through shared memory rows (one 4-byte store per
// lane and row, conflict-free) and a bulk-tensor store with an unswizzled
// 32 x 32 box, or stores per thread, where a warp's 32 lanes write 32
// consecutive columns of one row at a time.  Bulk stores mark C's lines first
// to evict in L2, which keeps more of A and B resident when the three share
// L2 (bf16 4096^3 -> fp32: DRAM traffic per launch 121.9 -> 111.6 MB).
#include <atomic>

#include "tc_common.cuh"

namespace tgemm {
namespace {

// One 32 x 32 block of C (rows m0.., columns n0..) from the lanes' values:
// lane l holds column n0 + l, v[i] is row m0 + i (the fused epilogue, when on,
// is applied in place first).  `throttle`: wait until this warp's previous
// bulk store has read its buffer before staging the block (one store in flight
// per warp) rather than the one before it (two in flight).
template <bool EPI>
__device__ __forceinline__ void store_block_t(uint32_t (&v)[32], int m0, int n0, int zc, int64_t c_off,
                                              bool tma_store, const TcArgs& args, const CUtensorMap* mapC,
                                              uint8_t* stage_base, int& sbuf, int lane, float bias_v,
                                              bool throttle) {
  const int out_fmt = args.out_fmt;
  if constexpr (EPI) {
    // lane = column (its bias is bias_v).  Each step is one uniform branch
    // over the 32 rows, so the per-element work is only the arithmetic (the
    // epilogue warps share issue slots with the producer and MMA threads).
    const float alpha = args.epi.alpha, beta = args.epi.beta;
    float z[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) z[i] = alpha * __uint_as_float(v[i]);
    if (beta != 0.0f) {
      // the 32 prior rows (each coalesced across the warp) are loaded before any is used
      const int n = n0 + lane;
      const bool col_in = n < args.N;
      float prior[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) prior[i] = (col_in && m0 + i < args.M) ? load_prior(args, m0 + i, n, c_off) : 0.0f;
#pragma unroll
      for (int i = 0; i < 32; ++i) z[i] = fmaf(beta, prior[i], z[i]);
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) z[i] += bias_v;
    if (args.epi.act == 1) {
#pragma unroll
      for (int i = 0; i < 32; ++i) z[i] = z[i] < 0.0f ? 0.0f : z[i];
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(z[i]);
  }
  if (tma_store) {
    uint8_t* buf = stage_base + sbuf * 4096;
    if (lane == 0) {
      if (throttle)
        ptx::bulk_wait_group_read<0>();
      else
        ptx::bulk_wait_group_read<1>();
    }
    __syncwarp();
    if (out_fmt == OUT_F32) {
#pragma unroll
      for (int i = 0; i < 32; ++i) *reinterpret_cast<uint32_t*>(buf + i * 128 + lane * 4) = v[i];
    } else {
      // rows of 64 bytes; lanes 2j and 2j+1 pack columns 2j, 2j+1 of rows i (even
      // lane) and i+1 (odd lane) into one word each
      const bool odd = lane & 1;
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        const float mine = __uint_as_float(odd ? v[i + 1] : v[i]);
        const float other = __shfl_xor_sync(0xffffffffu, __uint_as_float(odd ? v[i] : v[i + 1]), 1);
        const uint32_t word = odd ? pack_pair(other, mine, out_fmt) : pack_pair(mine, other, out_fmt);
        const int row = odd ? i + 1 : i;
        *reinterpret_cast<uint32_t*>(buf + row * 64 + (lane & ~1) * 2) = word;
      }
    }
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      ptx::tma_store_3d_hint(mapC, n0, m0, zc, ptx::smem_u32(buf), ptx::l2_evict_first_policy());
      ptx::bulk_commit_group();
    }
    sbuf ^= 1;
  } else {
    const int n = n0 + lane;
    if (n >= args.N) return;
    const int rows = min(32, args.M - m0);
    if (out_fmt == OUT_F32) {
      float* c = static_cast<float*>(args.C) + c_off + static_cast<int64_t>(m0) * args.ldc + n;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < rows) c[static_cast<int64_t>(i) * args.ldc] = __uint_as_float(v[i]);
    } else {
      uint16_t* c = static_cast<uint16_t*>(args.C) + c_off + static_cast<int64_t>(m0) * args.ldc + n;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < rows)
          c[static_cast<int64_t>(i) * args.ldc] =
              static_cast<uint16_t>(pack_pair(__uint_as_float(v[i]), 0.0f, out_fmt) & 0xFFFFu);
    }
  }
}

// EPI: the fused epilogue is compiled in (the plain product keeps its own
// instantiation and registers)
// The fused epilogue with beta != 0 and bulk-tensor stores: the 32 x 32 block's
// prior C already sits in `buf` (a bulk-tensor load of the same box, in the
// layout the store reads), so each lane reads its column of it, the results
// overwrite it in place, and the block goes out as in store_block_t.
__device__ __forceinline__ void store_block_staged_prior(const uint32_t (&v)[32], uint8_t* buf, int m0, int n0, int zc,
                                                         const TcArgs& args, const CUtensorMap* mapC, int lane,
                                                         float bias_v) {
  const int out_fmt = args.out_fmt;
  const float alpha = args.epi.alpha, beta = args.epi.beta;
  float z[32];
  if (out_fmt == OUT_F32) {
#pragma unroll
    for (int i = 0; i < 32; ++i) z[i] = *reinterpret_cast<const float*>(buf + i * 128 + lane * 4);
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const uint16_t h = *reinterpret_cast<const uint16_t*>(buf + i * 64 + lane * 2);
      z[i] = out_fmt == OUT_BF16 ? __uint_as_float(static_cast<uint32_t>(h) << 16) : __half2float(__ushort_as_half(h));
    }
  }
#pragma unroll
  for (int i = 0; i < 32; ++i) z[i] = fmaf(beta, z[i], alpha * __uint_as_float(v[i])) + bias_v;
  if (args.epi.act == 1) {
#pragma unroll
    for (int i = 0; i < 32; ++i) z[i] = z[i] < 0.0f ? 0.0f : z[i];
  }
  __syncwarp();  // every lane has read its prior column before any result overwrites the buffer
  if (out_fmt == OUT_F32) {
#pragma unroll
    for (int i = 0; i < 32; ++i) *reinterpret_cast<float*>(buf + i * 128 + lane * 4) = z[i];
  } else {
    const bool odd = lane & 1;
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      const float mine = odd ? z[i + 1] : z[i];
      const float other = __shfl_xor_sync(0xffffffffu, odd ? z[i] : z[i + 1], 1);
      const uint32_t word = odd ? pack_pair(other, mine, out_fmt) : pack_pair(mine, other, out_fmt);
      *reinterpret_cast<uint32_t*>(buf + (odd ? i + 1 : i) * 64 + (lane & ~1) * 2) = word;
    }
  }
  ptx::fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    ptx::tma_store_3d_hint(mapC, n0, m0, zc, ptx::smem_u32(buf), ptx::l2_evict_first_policy());
    ptx::bulk_commit_group();
  }
}

template <int TM, int KSUB, bool EPI>
__global__ void __launch_bounds__(32 * (2 + kEpiWarps), 1)
    tc_gemm_2sm_swap_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                            const __grid_constant__ CUtensorMap mapC, const TcArgs args) {
  constexpr int TN = 256;                // C columns per pair tile: the MMA's M
  constexpr int TMH = TM / 2;            // rows of A staged by each CTA
  constexpr int STAGES = tc2_stages(TM, true, KSUB);
  constexpr int A_SUB = 2 * 8192;        // 128 columns of B x 64 k: two atoms (the MMA's A)
  constexpr int B_SUB = tc_b_atoms(TMH) * 8192;  // room for TMH rows of A x 64 k (the MMA's B)
  constexpr int A_BYTES = KSUB * A_SUB;
  constexpr int B_BYTES = KSUB * B_SUB;
  constexpr int LOAD = KSUB * (A_SUB + TMH * kTileK * 2);  // bytes a CTA receives per stage
  constexpr int ACC = 256;
  constexpr uint32_t TMEM_COLS = 512;
  static_assert(TM % 32 == 0 && TM >= 128 && TM <= 256, "tile height");
  static_assert(TMH * kTileK * 2 <= B_SUB, "A rows fit their slot");
  static_assert(tc2_smem_bytes(TM, true, KSUB) <= kSmemLimit, "shared memory per CTA");
  static_assert(STAGES >= 3, "ring depth");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;  // the MMA's A operand: B columns
  uint8_t* sB = sA + STAGES * A_BYTES;  // the MMA's B operand: A rows
  uint8_t* sC = sB + STAGES * B_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sC + tc2_epi_bytes(true));
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint64_t* prior_bar = drain + 1;  // two per epilogue warp: prior C blocks staged for beta != 0
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(prior_bar + 2 * kEpiWarps);
  static_assert((2 * STAGES + 5 + 2 * kEpiWarps) * 8 + 8 <= kBarrierBytes, "barrier area");
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(ptx::smem_u32(&full[s]), 1);   // leader only: its producer's expect_tx
      ptx::mbar_init(ptx::smem_u32(&empty[s]), 1);  // multicast MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(ptx::smem_u32(&acc_full[b]), 1);              // multicast MMA commit
      ptx::mbar_init(ptx::smem_u32(&acc_empty[b]), 2 * kEpiWarps);  // leader only: both CTAs' epilogues
    }
    ptx::mbar_init(ptx::smem_u32(drain), 1);
    for (int i = 0; i < 2 * kEpiWarps; ++i) ptx::mbar_init(ptx::smem_u32(&prior_bar[i]), 1);
    *abort_flag = 0u;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&mapA);
    ptx::tma_prefetch_desc(&mapB);
    if (args.store_granule == 0) ptx::tma_prefetch_desc(&mapC);
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before_sync();
  ptx::cluster_sync();
  ptx::tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  const Ctl ctl{abort_flag, args.timeout_ns, args.status};

  if (warp == 0) {
    // ------------------------------------------------ bulk-tensor producer
    if (lane == 0 && !args.inject_fault) {
      ptx::griddep_wait();  // operands written by the kernel before (repack) are visible
      const uint32_t tx_pair = 2u * LOAD;
      int stage = 0;
      uint32_t phase = 0, filled = 0, last_parity = 0;
      bool ok = true;
      for (int t = pair; ok && t < args.num_tiles; t += npairs) {
        const int b = t / args.tiles_per;  // matrix of the batch
        int mb, nb;
        tile_coords(t - b * args.tiles_per, args, mb, nb);
        const int za = args.stride_a ? b : 0, zb = args.stride_b ? b : 0;
        const int a_row = mb * TM + static_cast<int>(rank) * TMH;
        const int b_col = nb * TN + static_cast<int>(rank) * (TN / 2);
        for (int kb = 0; kb < args.k_blocks; ++kb) {
          if (!wait_bounded(ptx::smem_u32(&empty[stage]), phase ^ 1u, ctl, SITE_PRODUCER_EMPTY)) {
            ok = false;
            break;
          }
          const uint32_t fb_local = ptx::smem_u32(&full[stage]);
          const uint32_t fb = ptx::mapa_shared(fb_local, 0);
          if (leader) ptx::mbar_arrive_expect_tx(fb_local, tx_pair);
#pragma unroll
          for (int s = 0; s < KSUB; ++s) {
            const int k0 = (kb * KSUB + s) * kTileK;  // sub-blocks past K load zeros
#pragma unroll
            for (int j = 0; j < 2; ++j)
              ptx::tma_load_3d_pair(ptx::smem_u32(sA + stage * A_BYTES + s * A_SUB + j * 8192), &mapB,
                                    b_col + j * 64, k0, zb, fb);
            ptx::tma_load_3d_pair(ptx::smem_u32(sB + stage * B_BYTES + s * B_SUB), &mapA, k0, a_row, za, fb);
          }
          filled |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // loads in flight land before shared memory is released (see tc_gemm_2sm.cu)
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
      for (int t = pair; ok && t < args.num_tiles; t += npairs) {
        if (!wait_bounded(ptx::smem_u32(&acc_empty[acc]), acc_phase ^ 1u, ctl, SITE_MMA_ACC_EMPTY)) break;
        ptx::tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * ACC);
        for (int kb = 0; kb < args.k_blocks; ++kb) {
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
              // A: B columns, N-major (atoms 8 KB apart, 8 k-rows per 1 KB);
              // B: A rows, K-major (8-row groups 1 KB apart, 16 k = 32 bytes)
              ptx::tc_mma_f16_pair(d_tmem, sw128_desc(a0 + s * A_SUB + k * 2048, 8192, 1024),
                                   sw128_desc(b0 + s * B_SUB + k * 32, 16, 1024), args.idesc,
                                   (kb != 0 || s != 0 || k != 0) ? 1u : 0u);
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
    const bool tma_store = args.store_granule == 0;
    int acc = 0, sbuf = 0;
    uint32_t acc_phase = 0;
    // beta != 0 with bulk-tensor stores: the prior C blocks come through this
    // warp's two staging buffers by bulk-tensor loads, one block ahead
    const bool staged_prior = EPI && tma_store && args.epi.beta != 0.0f;
    const uint32_t pbar0 = ptx::smem_u32(&prior_bar[2 * (warp - 2)]), pbar1 = pbar0 + 8;
    const uint32_t blk_bytes = args.out_fmt == OUT_F32 ? 4096u : 2048u;
    uint32_t pphase = 0u;   // bit i: phase of buffer i's barrier
    uint32_t pending = 0u;  // bit i: a load into buffer i is in flight
    for (int t = pair; t < args.num_tiles; t += npairs) {
      const int b = t / args.tiles_per;  // matrix of the batch
      const int64_t c_off = b * args.stride_c;
      int mb, nb;
      tile_coords(t - b * args.tiles_per, args, mb, nb);
      // this warp's TMEM lanes are 32 columns of C
      const int n0 = nb * TN + static_cast<int>(rank) * (TN / 2) + q * 32;
      float bias_v = 0.0f;
      if constexpr (EPI) {
        // while the tile's MMAs run: the prior C this warp will read goes to
        // L2, and the lane's column bias into a register
        if (args.epi.beta != 0.0f && tma_store && lane == 0 && n0 < args.N)
          for (int c = 0; c < TM / 32 && mb * TM + c * 32 < args.M; ++c)
            ptx::tma_prefetch_l2_3d(&mapC, n0, mb * TM + c * 32, b);
        if (args.epi.bias && n0 + lane < args.N) bias_v = args.epi.bias[n0 + lane];
      }
      const int nblk = min(TM / 32, (args.M - mb * TM + 31) / 32);  // blocks of rows inside C
      // The stores of C pass through the SM's bulk-copy path, which the next
      // tile's operand loads need at about the rate it can deliver.  While a
      // later tile of this pair is being loaded, fp32 blocks go out one store
      // per warp at a time (bf16 4096^3 -> fp32: 86.1 -> 84.5 us); the pair's
      // last tile, with nothing left to load, keeps two in flight.
      const bool throttle = args.out_fmt == OUT_F32 && t + npairs < args.num_tiles;
      if (staged_prior && n0 < args.N) {
        // the first block's prior C, loaded while the tile's MMAs run (after
        // the previous tile's stores have read the buffers)
        sbuf = 0;
        if (lane == 0) {
          ptx::bulk_wait_group_read<0>();
          ptx::mbar_arrive_expect_tx(pbar0, blk_bytes);
          ptx::tma_load_3d(ptx::smem_u32(stage_base), &mapC, n0, mb * TM, b, pbar0);
        }
        pending |= 1u;
      }
      if (!warp_wait(ptx::smem_u32(&acc_full[acc]), acc_phase, ctl, SITE_EPI_ACC_FULL)) break;
      ptx::tc_fence_after_sync();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * ACC);
      if (n0 < args.N) {
        bool ok = true;
#pragma unroll 1
        for (int c = 0; c < nblk; ++c) {
          const int m0 = mb * TM + c * 32;
          uint32_t v[32];
          if (staged_prior) {
            const int cur = c & 1, nxt = cur ^ 1;
            const uint32_t bar_cur = cur ? pbar1 : pbar0, bar_nxt = cur ? pbar0 : pbar1;
            if (c + 1 < nblk) {
              // block c+1's prior into the other buffer, once the store of
              // block c-1 (its last user) has read it
              if (lane == 0) {
                ptx::bulk_wait_group_read<0>();
                ptx::mbar_arrive_expect_tx(bar_nxt, blk_bytes);
                ptx::tma_load_3d(ptx::smem_u32(stage_base + nxt * 4096), &mapC, n0, m0 + 32, b, bar_nxt);
              }
              pending |= 1u << nxt;
            }
            if (!warp_wait(bar_cur, (pphase >> cur) & 1u, ctl, SITE_EPI_PRIOR)) {
              ok = false;
              break;
            }
            pphase ^= 1u << cur;
            pending &= ~(1u << cur);
            ptx::tmem_ld_32x32b_x32(tbase + c * 32, v);
            ptx::tmem_wait_ld();
            store_block_staged_prior(v, stage_base + cur * 4096, m0, n0, b, args, &mapC, lane, bias_v);
          } else {
            ptx::tmem_ld_32x32b_x32(tbase + c * 32, v);
            ptx::tmem_wait_ld();
            store_block_t<EPI>(v, m0, n0, b, c_off, tma_store, args, &mapC, stage_base, sbuf, lane, bias_v,
                               throttle);
          }
        }
        if (!ok) break;
      }
      ptx::tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa_shared(ptx::smem_u32(&acc_empty[acc]), 0));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    // a prior-C load still in flight (a wait gave up) lands before shared memory is released
    for (int i = 0; i < 2; ++i)
      if (((pending >> i) & 1u) && lane == 0) wait_teardown(i ? pbar1 : pbar0, (pphase >> i) & 1u, ctl, SITE_TEARDOWN);
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

template <int TM, int KSUB, bool EPI>
cudaError_t launch_swap(const CUtensorMap& mA, const CUtensorMap& mB, const CUtensorMap& mC, const TcArgs& args,
                        int pairs, cudaStream_t stream) {
  constexpr int smem = tc2_smem_bytes(TM, true, KSUB);
  auto kernel = tc_gemm_2sm_swap_kernel<TM, KSUB, EPI>;
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
  return cudaLaunchKernelEx(&cfg, kernel, mA, mB, mC, args);
}

}  // namespace

cudaError_t launch_tc_pair_swap(int tm, int ksub, const CUtensorMap& mA, const CUtensorMap& mB,
                                const CUtensorMap& mC, const TcArgs& args, int pairs, cudaStream_t stream) {
  const bool epi = args.epi.on != 0;
#define TGEMM_SWAP_TM(TMV)                                                                            \
  case TMV:                                                                                           \
    if (epi)                                                                                          \
      return ksub == 2 ? launch_swap<TMV, 2, true>(mA, mB, mC, args, pairs, stream)                   \
                       : launch_swap<TMV, 1, true>(mA, mB, mC, args, pairs, stream);                  \
    return ksub == 2 ? launch_swap<TMV, 2, false>(mA, mB, mC, args, pairs, stream)                    \
                     : launch_swap<TMV, 1, false>(mA, mB, mC, args, pairs, stream);
  switch (tm) {
    TGEMM_SWAP_TM(128)
    TGEMM_SWAP_TM(192)
    TGEMM_SWAP_TM(224)
    TGEMM_SWAP_TM(256)
    default: return cudaErrorInvalidValue;
  }
#undef TGEMM_SWAP_TM
}

}  // namespace tgemm
