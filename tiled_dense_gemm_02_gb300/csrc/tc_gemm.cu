// Tensor-core tiled GEMM for sm_103a: C[M,N] = A[M,K] . B[K,N], fp16/bf16 in,
// fp32 accumulate in tensor memory, fp32/fp16/bf16 out.
//
// Three levels of tiling ("Tiling 策略与内存层次优化", section 多级 Tiling 策略),
// mapped onto Blackwell:
//   * output tiles of 128 x BN (BN = 64/128/256) owned by one CTA at a time; a
//     persistent grid of at most one CTA per SM walks the tile list in a
//     grouped (swizzled) order, so consecutive tiles of a CTA wave share B
//     panels in L2 ("GPU Kernel 的 Tile、Grid、Wave 与 Launch Overhead": fewer,
//     larger workers instead of many waves);
//   * K is split into 64-element stages ("矩阵乘法中的平铺", the l-length
//     K-splitting paragraph); each stage's A and B tiles go through a
//     multi-stage shared-memory ring ("Double Buffering / Multi-Stage
//     Pipelining") with the 128-byte XOR swizzle ("Bank Conflict 与 Swizzling"),
//     filled by bulk-tensor copies (TMA) or, for rows that are not 16-byte
//     aligned, by per-thread async copies writing the same swizzled layout;
//   * the register/MMA level becomes tcgen05.mma issued by one thread, 128 x BN
//     x 16 per instruction, accumulating fp32 in tensor memory (two accumulator
//     buffers, so the epilogue of one tile overlaps the MMAs of the next).
// The epilogue reads tensor memory into registers, converts, and writes C by
// bulk-tensor stores (out-of-range rows/columns clipped) or by masked
// per-thread stores ("CUDA tile", section 四.4: zero-fill loads, masked stores).
//
// Warp roles (one CTA per SM):
//   warp 0      bulk-tensor producer (one elected lane)
//   warp 1      tensor-memory allocator and MMA issuer (one elected lane)
//   warps 2..5  epilogue, one warp per 32-lane quarter of tensor memory
//   warps 6..9  per-thread-copy producers (only in the copy variant)
// Every mbarrier wait is bounded in time; a wait that gives up records a code
// in the device status word, raises a CTA-wide abort flag so the other roles
// leave their loops, and the CTA still drains its copies and frees its tensor
// memory before exiting.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>

#include "tc_common.cuh"

namespace tgemm {
namespace {


// -------------------------------------------------------------- the kernel
template <int BN, bool kCopy>
__global__ void __launch_bounds__(tc_threads(kCopy), 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                   const __grid_constant__ CUtensorMap mapC, const TcArgs args) {
  constexpr int STAGES = tc_stages(BN);
  constexpr int A_BYTES = kTileM * kTileK * 2;
  constexpr int B_BYTES = tc_b_atoms(BN) * 8192;
  constexpr int ACC = tc_acc_stride(BN);
  constexpr uint32_t TMEM_COLS = 2 * ACC;
  static_assert(tc_valid_bn(BN), "tile width");
  static_assert(STAGES >= 3, "ring depth");
  static_assert(tc_smem_bytes(BN) <= kSmemLimit, "shared memory per CTA");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + STAGES * A_BYTES;
  uint8_t* sC = sB + STAGES * B_BYTES;
  uint64_t* full_tma = reinterpret_cast<uint64_t*>(sC + kEpiWarps * 2 * 4096);
  uint64_t* full_copy = full_tma + STAGES;
  uint64_t* empty = full_copy + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const bool has_tma = args.a_copy == 0 || args.b_copy == 0;
  const bool has_copy = kCopy && (args.a_copy != 0 || args.b_copy != 0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(ptx::smem_u32(&full_tma[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&full_copy[s]), kCopyWarps * 32);
      ptx::mbar_init(ptx::smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(ptx::smem_u32(&acc_full[b]), 1);
      ptx::mbar_init(ptx::smem_u32(&acc_empty[b]), kEpiWarps);
    }
    ptx::mbar_init(ptx::smem_u32(drain), 1);
    *abort_flag = 0u;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    if (args.a_copy == 0) ptx::tma_prefetch_desc(&mapA);
    if (args.b_copy == 0) ptx::tma_prefetch_desc(&mapB);
    if (args.store_granule == 0) ptx::tma_prefetch_desc(&mapC);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  const Ctl ctl{abort_flag, args.timeout_ns, args.status};
  const int num_tiles = args.num_tiles;
  const int kbs = args.k_blocks;

  if (warp == 0) {
    // ------------------------------------------------ bulk-tensor producer
    if (lane == 0 && has_tma && !args.inject_fault) {
      ptx::griddep_wait();  // operands written by the kernel before (repack) are visible
      const bool a_tma = args.a_copy == 0, b_tma = args.b_copy == 0;
      const uint32_t tx = (a_tma ? A_BYTES : 0) + (b_tma ? B_BYTES : 0);
      int stage = 0;
      uint32_t phase = 0, filled = 0, last_parity = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
        int mb, nb;
        tile_coords(t, args, mb, nb);
        for (int kb = 0; kb < kbs; ++kb) {
          if (!wait_bounded(ptx::smem_u32(&empty[stage]), phase ^ 1u, ctl, SITE_PRODUCER_EMPTY)) {
            ok = false;
            break;
          }
          const uint32_t fb = ptx::smem_u32(&full_tma[stage]);
          ptx::mbar_arrive_expect_tx(fb, tx);
          if (a_tma) ptx::tma_load_2d(ptx::smem_u32(sA + stage * A_BYTES), &mapA, kb * kTileK, mb * kTileM, fb);
          if (b_tma) {
#pragma unroll
            for (int j = 0; j < tc_b_atoms(BN); ++j)
              ptx::tma_load_2d(ptx::smem_u32(sB + stage * B_BYTES + j * 8192), &mapB, nb * BN + j * 64, kb * kTileK,
                               fb);
          }
          filled |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Every load this thread issued must land before shared memory is released.
      for (int s = 0; s < STAGES; ++s)
        if ((filled >> s) & 1u) {
          const Ctl own{abort_flag, ctl.timeout_ns, ctl.status};
          // a fill that completed long ago returns at once; after an abort the
          // wait still runs (bounded) because the copies are real
          uint32_t par = (last_parity >> s) & 1u;
          if (!ptx::mbar_try_wait(ptx::smem_u32(&full_tma[s]), par)) {
            const uint64_t t0 = ptx::globaltimer_ns();
            while (!ptx::mbar_try_wait(ptx::smem_u32(&full_tma[s]), par)) {
              if (ptx::globaltimer_ns() - t0 > own.timeout_ns) {
                atomicCAS(own.status, 0u, kTimeoutFlag | SITE_TEARDOWN);
                break;
              }
            }
          }
        }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
        if (!wait_bounded(ptx::smem_u32(&acc_empty[acc]), acc_phase ^ 1u, ctl, SITE_MMA_ACC_EMPTY)) break;
        ptx::tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * ACC);
        for (int kb = 0; kb < kbs; ++kb) {
          if (has_tma && !wait_bounded(ptx::smem_u32(&full_tma[stage]), phase, ctl, SITE_MMA_FULL)) {
            ok = false;
            break;
          }
          if (has_copy) {
            if (!wait_bounded(ptx::smem_u32(&full_copy[stage]), phase, ctl, SITE_MMA_FULL)) {
              ok = false;
              break;
            }
            // the copies wrote through the generic proxy; the MMA reads through the async one
            ptx::fence_proxy_async_smem();
          }
          ptx::tc_fence_after_sync();
          const uint32_t a0 = ptx::smem_u32(sA + stage * A_BYTES);
          const uint32_t b0 = ptx::smem_u32(sB + stage * B_BYTES);
#pragma unroll
          for (int k = 0; k < kTileK / 16; ++k) {
            // A: K-major, 16 elements = 32 bytes further along each swizzled row.
            // B: N-major, 16 k-rows = 2 groups of 8 rows (1024 B each) further on;
            //    64-column atoms are 8 KB apart.
            ptx::tc_mma_f16(d_tmem, sw128_desc(a0 + k * 32, 16, 1024), sw128_desc(b0 + k * 2048, 8192, 1024),
                            args.idesc, (kb | k) != 0 ? 1u : 0u);
          }
          ptx::tc_commit(ptx::smem_u32(&empty[stage]));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::tc_commit(ptx::smem_u32(&acc_full[acc]));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // All MMAs this thread issued have finished before tensor memory is freed.
      ptx::tc_commit(ptx::smem_u32(drain));
      const Ctl own{abort_flag, ctl.timeout_ns, ctl.status};
      if (!ptx::mbar_try_wait(ptx::smem_u32(drain), 0)) {
        const uint64_t t0 = ptx::globaltimer_ns();
        while (!ptx::mbar_try_wait(ptx::smem_u32(drain), 0)) {
          if (ptx::globaltimer_ns() - t0 > own.timeout_ns) {
            atomicCAS(own.status, 0u, kTimeoutFlag | SITE_DRAIN);
            break;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp < 2 + kEpiWarps) {
    // --------------------------------------------------------- epilogue
    const int q = warp & 3;  // tensor-memory lane quarter this warp may read
    uint8_t* stage_base = sC + (warp - 2) * 2 * 4096;
    int acc = 0, sbuf = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
      int mb, nb;
      tile_coords(t, args, mb, nb);
      if (!warp_wait(ptx::smem_u32(&acc_full[acc]), acc_phase, ctl, SITE_EPI_ACC_FULL)) break;
      ptx::tc_fence_after_sync();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * ACC);
      epilogue_tile<BN>(tbase, mb * kTileM + q * 32, nb * BN, args, &mapC, stage_base, sbuf, lane);
      // this warp's reads of the accumulator buffer are complete
      ptx::tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&acc_empty[acc]));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    // the stores must have read shared memory before the CTA exits (their
    // writes to C complete with the kernel)
    if (lane == 0) ptx::bulk_wait_group_read<0>();
    __syncwarp();
  } else if constexpr (kCopy) {
    // -------------------------------------------------- copy producers
    const int ct = threadIdx.x - (2 + kEpiWarps) * 32;
    const CopyOps ops{static_cast<const uint16_t*>(args.A), static_cast<const uint16_t*>(args.B), args.lda, args.ldb,
                      args.M, args.N, args.K, args.a_copy, args.b_copy};
    const uint32_t sA_u = ptx::smem_u32(sA), sB_u = ptx::smem_u32(sB);
    if (has_copy && !args.inject_fault) {
      ptx::griddep_wait();
      const bool sync_arrive = ops.a_copy == 2 || ops.b_copy == 2;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
        int mb, nb;
        tile_coords(t, args, mb, nb);
        for (int kb = 0; kb < kbs; ++kb) {
          if (!warp_wait(ptx::smem_u32(&empty[stage]), phase ^ 1u, ctl, SITE_COPY_EMPTY)) {
            ok = false;
            break;
          }
          if (ops.a_copy) copy_a_dispatch(sA_u + stage * A_BYTES, ops, mb * kTileM, kb * kTileK, ct);
          if (ops.b_copy) copy_b_dispatch<BN>(sB_u + stage * B_BYTES, ops, kb * kTileK, nb * BN, ct);
          const uint32_t fb = ptx::smem_u32(&full_copy[stage]);
          if (sync_arrive) {
            // 2-byte granules are plain stores: finish every copy, then arrive
            ptx::cp_async_commit();
            ptx::cp_async_wait<0>();
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(fb);
          } else {
            // the stage's arrival fires by itself once this thread's copies land
            ptx::cp_async_mbar_arrive_noinc(fb);
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
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after_sync();
    ptx::tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

__global__ void zero_fill_kernel(uint8_t* C, int64_t rows, int64_t row_bytes, int64_t ld_bytes) {
  const int64_t total = rows * row_bytes;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = i / row_bytes, b = i % row_bytes;
    C[r * ld_bytes + b] = 0;
  }
}

// K = 0 with a fused epilogue: C = act(alpha * 0 + beta * C + bias), element
// by element (the empty sum is 0).
__global__ void epilogue_fill_kernel(void* C, int64_t rows, int64_t cols, int64_t ldc, int out_fmt, Epilogue e) {
  const int64_t total = rows * cols;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = i / cols, c = i % cols;
    const int64_t idx = r * ldc + c;
    if (out_fmt == OUT_F32) {
      float* p = static_cast<float*>(C) + idx;
      *p = epi_apply(e, 0.0f, static_cast<int>(c), [&] { return *p; });
    } else if (out_fmt == OUT_BF16) {
      __nv_bfloat16* p = static_cast<__nv_bfloat16*>(C) + idx;
      *p = __float2bfloat16_rn(epi_apply(e, 0.0f, static_cast<int>(c), [&] { return __bfloat162float(*p); }));
    } else {
      __half* p = static_cast<__half*>(C) + idx;
      *p = __float2half_rn(epi_apply(e, 0.0f, static_cast<int>(c), [&] { return __half2float(*p); }));
    }
  }
}

template <int BN, bool kCopy>
cudaError_t launch_one(const CUtensorMap& mA, const CUtensorMap& mB, const CUtensorMap& mC, const TcArgs& args,
                       int ctas, cudaStream_t stream) {
  constexpr int smem = tc_smem_bytes(BN);
  auto kernel = tc_gemm_kernel<BN, kCopy>;
  // The attribute is per device; set it on every device the first time.
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
  cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
  cfg.blockDim = dim3(tc_threads(kCopy), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  cfg.attrs = attr;
  cfg.numAttrs = static_cast<unsigned>(tc_launch_attrs(attr, 1, args));
  return cudaLaunchKernelEx(&cfg, kernel, mA, mB, mC, args);
}

}  // namespace

cudaError_t launch_tc(int bn, bool copy, const CUtensorMap& mA, const CUtensorMap& mB, const CUtensorMap& mC,
                      const TcArgs& args, int ctas, cudaStream_t stream) {
#define TGEMM_LAUNCH_BN(BNV)                                                                       \
  case BNV:                                                                                        \
    return copy ? launch_one<BNV, true>(mA, mB, mC, args, ctas, stream)                            \
                : launch_one<BNV, false>(mA, mB, mC, args, ctas, stream);
  switch (bn) {
    TGEMM_LAUNCH_BN(64)
    TGEMM_LAUNCH_BN(128)
    TGEMM_LAUNCH_BN(192)
    TGEMM_LAUNCH_BN(224)
    TGEMM_LAUNCH_BN(256)
    default: return cudaErrorInvalidValue;
  }
#undef TGEMM_LAUNCH_BN
}

cudaError_t launch_epilogue_fill(void* C, int64_t rows, int64_t cols, int64_t ldc, int out_fmt, const Epilogue& e,
                                 cudaStream_t stream) {
  int blocks = static_cast<int>(std::min<int64_t>((rows * cols + 255) / 256, 4096));
  if (blocks < 1) blocks = 1;
  epilogue_fill_kernel<<<blocks, 256, 0, stream>>>(C, rows, cols, ldc, out_fmt, e);
  return cudaGetLastError();
}

cudaError_t launch_zero_fill(void* C, int64_t rows, int64_t cols, int64_t ldc, int elem_bytes, cudaStream_t stream) {
  const int64_t total = rows * cols * elem_bytes;
  int blocks = static_cast<int>(std::min<int64_t>((total + 255) / 256, 4096));
  if (blocks < 1) blocks = 1;
  zero_fill_kernel<<<blocks, 256, 0, stream>>>(static_cast<uint8_t*>(C), rows, cols * elem_bytes, ldc * elem_bytes);
  return cudaGetLastError();
}

}  // namespace tgemm
