// C ABI of the tiled GEMM library: argument validation, dispatch planning,
// bulk-tensor descriptor encoding and launch.  See include/tgemm.h for the
// contract of each entry point.
#include <cuda.h>
#include <cuda_runtime.h>

#include <unistd.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/tgemm.h"
#include "tgemm_internal.h"
#include "simt_sgemm.h"

namespace tgemm {

// Device-side status word: bounded in-kernel waits that give up write a code
// here; tgemm_device_status reads and clears it.
__device__ unsigned int g_device_status = 0;

namespace {

thread_local std::string t_last_error;
// Device the calling thread's current call runs on (set by device_info).
thread_local int t_device = 0;

struct DeviceInfo {
  bool ready = false;
  bool supported = false;
  int sm_count = 0;
  unsigned int* status = nullptr;
  int pair_capacity = 0;  // resident CTA pairs of the pair kernel (0 = not queried)
};

std::mutex g_mutex;
DeviceInfo g_devices[64];

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int cuda_fail(cudaError_t e, const char* what) {
  t_last_error = std::string(what) + ": " + cudaGetErrorString(e);
  return TGEMM_ERR_LAUNCH;
}

// Look up (once per device) SM count, compute capability and the status word.
int device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) {
    t_last_error = "device ordinal out of range";
    return TGEMM_ERR_LAUNCH;
  }
  t_device = dev;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceInfo& d = g_devices[dev];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    d.supported = (major == 10 && minor == 3);
    d.sm_count = sms;
    if (d.supported) {
      void* p = nullptr;
      if ((e = cudaGetSymbolAddress(&p, g_device_status)) != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress");
      d.status = static_cast<unsigned int*>(p);
    }
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
        t_last_error = "cuTensorMapEncodeTiled entry point not found";
        return TGEMM_ERR_LAUNCH;
      }
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    d.ready = true;
  }
  *out = &d;
  return d.supported ? TGEMM_OK : TGEMM_ERR_UNSUPPORTED_DEVICE;
}

// Streams that carry tgemm_gemm_host's copies: one for host-to-device and one
// for device-to-host per device, created on first use and kept for the life
// of the process (guarded by g_mutex).  Non-blocking, so they never
// synchronise implicitly with the legacy default stream; every ordering is an
// event.
struct CopyStreams {
  cudaStream_t in = nullptr, out = nullptr;
};
CopyStreams g_copy_streams[64];

int copy_streams(cudaStream_t* in, cudaStream_t* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) {
    t_last_error = "device ordinal out of range";
    return TGEMM_ERR_LAUNCH;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  CopyStreams& c = g_copy_streams[dev];
  for (cudaStream_t* sp : {&c.in, &c.out})
    if (!*sp && (e = cudaStreamCreateWithFlags(sp, cudaStreamNonBlocking)) != cudaSuccess) {
      *sp = nullptr;
      return cuda_fail(e, "cudaStreamCreateWithFlags");
    }
  *in = c.in;
  *out = c.out;
  return TGEMM_OK;
}

// A block of `rows` rows of `width` bytes between host and device memory: one
// linear copy when both sides are dense (the driver moves a pitched copy row
// by row, which costs it half its rate on rows of a few KB), else pitched.
cudaError_t copy_rows(void* dst, int64_t dpitch, const void* src, int64_t spitch, int64_t width, int64_t rows,
                      cudaMemcpyKind kind, cudaStream_t s) {
  if (dpitch == width && spitch == width) return cudaMemcpyAsync(dst, src, width * rows, kind, s);
  return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, rows, kind, s);
}

// Events of tgemm_gemm_host calls come from a per-device pool (guarded by
// g_mutex): a call takes the events it needs and hands them back when it
// returns, whether or not the work they mark has completed.  Recording an
// event again only changes what later waits and queries see; a wait already
// enqueued stays bound to the record it was enqueued against.  So calls
// create events only while the pool grows, and never destroy them.
struct EventPool {
  std::vector<cudaEvent_t> free;
};
EventPool g_event_pools[64];

struct CallEvents {
  int dev = 0;
  std::vector<cudaEvent_t> ev;
  ~CallEvents() {
    if (ev.empty()) return;
    std::lock_guard<std::mutex> lock(g_mutex);
    std::vector<cudaEvent_t>& f = g_event_pools[dev].free;
    f.insert(f.end(), ev.begin(), ev.end());
  }
  cudaError_t make(cudaEvent_t* out) {
    {
      std::lock_guard<std::mutex> lock(g_mutex);
      std::vector<cudaEvent_t>& f = g_event_pools[dev].free;
      if (!f.empty()) {
        *out = f.back();
        f.pop_back();
        ev.push_back(*out);
        return cudaSuccess;
      }
    }
    const cudaError_t e = cudaEventCreateWithFlags(out, cudaEventDisableTiming);
    if (e == cudaSuccess) ev.push_back(*out);
    return e;
  }
};

int in_bytes(int dtype) { return dtype == TGEMM_F32 ? 4 : 2; }
int out_bytes(int dtype) {
  return (dtype == TGEMM_F32 || dtype == TGEMM_BF16_F32OUT || dtype == TGEMM_F16_F32OUT) ? 4 : 2;
}

// Largest of 16/8/4/2 bytes dividing both the base address and the row pitch.
int granule(const void* p, int64_t ld, int es) {
  const uint64_t a = reinterpret_cast<uint64_t>(p);
  const uint64_t pitch = static_cast<uint64_t>(ld) * es;
  for (int g = 16; g >= 4; g /= 2)
    if (a % g == 0 && pitch % g == 0) return g;
  return 2;
}

bool ranges_overlap(uint64_t a0, uint64_t a1, uint64_t b0, uint64_t b1) { return a0 < b1 && b0 < a1; }

struct Plan {
  int kernel = TGEMM_KERNEL_AUTO;
  bool noop = false, zero = false;
  bool pair = false;
  bool swap = false;  // pair kernel with the MMA's operands exchanged (tile tm x 256)
  bool copy_pair = false;  // pair kernel with B staged by per-thread copies (A by bulk-tensor copies)
  int tm = 0;         // tile height of the swapped kernel
  int ksub = 1;  // 64-deep K sub-blocks per shared-memory stage (pair kernel)
  int bn = 256, stages = 4, tiles_m = 0, tiles_n = 0, ctas = 0, group_m = 1;
  int a_copy = 0, b_copy = 0, store = 0;
  int smem = 0;
  int k_blocks = 0;               // k-stages per tile
  int dp_tiles = 0, sk_iters = 0;  // stream-K split (sk_iters == 0: whole tiles only)
  int64_t workspace = 0;          // bytes of workspace the stream-K split uses
  int split_stage = 0;            // SIMT kernel: k-stage dividing the halves of its split tiles (0: none)
  bool simt_small = false;        // fp32: the small-product kernel (32 x 32 tiles)
  int64_t batch = 1;              // matrices computed by one launch (strided batch, swapped kernel)
  int packed = 0;                 // operands repacked into the workspace first: 1 = A, 2 = B
  int64_t lda_p = 0, ldb_p = 0;   // their pitches there (elements, multiples of 8)
  int64_t off_a = 0, off_b = 0;   // their byte offsets in the workspace
  int granule_a = 0, granule_b = 0;  // the source rows' alignment (bytes)
  bool batch_loop = false;        // a batch the kernels cannot index: one launch per matrix
  bool tuned = false;             // options from the tuned-shape table
};

// Relative throughput of one SM per output column for each tile width,
// measured on GB300 with bf16 4096^3 (per-wave time of one 128 x BN tile):
// operand traffic per FLOP grows as the tile narrows, and the 224-wide tile
// still moves four 64-column B atoms.
double width_rate(int bn) {
  switch (bn) {
    case 256: return 1.0;
    case 224: return 0.86;
    case 192: return 0.8;
    case 128: return 0.65;
    default: return 0.34;
  }
}

// Tile width minimising (waves x width / rate): the persistent grid runs
// ceil(tiles / SMs) rounds of BN-wide tiles.
int pick_tile_n(int64_t M, int64_t N, int sms, double* cost) {
  int best = 256;
  double best_t = 1e300;
  for (int bn : {256, 224, 192, 128, 64}) {
    const int64_t tiles = ((M + kTileM - 1) / kTileM) * ((N + bn - 1) / bn);
    const int64_t waves = (tiles + sms - 1) / sms;
    const double t = static_cast<double>(waves) * bn / width_rate(bn);
    if (t < best_t * 0.999) {
      best_t = t;
      best = bn;
    }
  }
  if (cost) *cost = best_t;
  return best;
}

// Per-SM throughput per output column of the pair kernel, in the units of
// width_rate (each SM of a pair computes 128 x BN per tile), measured on GB300
// with bf16 4096^3.
double pair_rate(int bn) {
  switch (bn) {
    case 256: return 1.13;
    case 224: return 0.99;
    case 192: return 0.88;
    default: return 0.64;
  }
}

// `stream_k`: the remainder of the last round is split along K over all pairs,
// costing its share of a round plus a fix-up of about a tenth of a round.
int pick_pair_tile_n(int64_t M, int64_t N, int pairs, bool stream_k, double* cost) {
  int best = 256;
  double best_t = 1e300;
  for (int bn : {256, 224, 192, 128}) {
    const int64_t tiles = ((M + 2 * kTileM - 1) / (2 * kTileM)) * ((N + bn - 1) / bn);
    double waves = static_cast<double>((tiles + pairs - 1) / pairs);
    const int64_t rem = tiles % pairs;
    if (stream_k && rem != 0 && rem * 10 <= 9 * pairs) waves = static_cast<double>(tiles / pairs) + 0.1 +
                                                                 static_cast<double>(rem) / pairs;
    const double t = waves * bn / pair_rate(bn);
    if (t < best_t * 0.999) {
      best_t = t;
      best = bn;
    }
  }
  if (cost) *cost = best_t;
  return best;
}

// Per-SM throughput per tile row of the swapped pair kernel (tile tm x 256),
// in the units of width_rate, measured on GB300 with bf16 8192^3 (1915, 1806,
// 1653 and 1397 TFLOP/s for tm = 256, 224, 192, 128).  It falls with tm
// because each SM stages and reads 128 columns of B per k-step whatever tm is.
double swap_rate(int tm) {
  switch (tm) {
    case 256: return 1.16;
    case 224: return 1.09;
    case 192: return 1.0;
    default: return 0.845;
  }
}

// Tile height of the swapped pair kernel minimising rounds x tm / rate: each
// round runs `pairs` tm x 256 tiles.
int pick_swap_tile_m(int64_t M, int64_t N, int pairs, double* cost, int64_t batch = 1) {
  int best = 256;
  double best_t = 1e300;
  for (int tm : {256, 224, 192, 128}) {
    const int64_t tiles = ((M + tm - 1) / tm) * ((N + 255) / 256) * batch;
    const double t = static_cast<double>((tiles + pairs - 1) / pairs) * tm / swap_rate(tm);
    if (t < best_t * 0.999) {
      best_t = t;
      best = tm;
    }
  }
  if (cost) *cost = best_t;
  return best;
}

// Launch options measured fastest per shape (tiled_dense_gemm_02_gb300/tune.py),
// used when a call leaves every tuned option at 0.
struct TunedShape {
  int64_t M, N, K;
  int dtype;
  int kernel, cta_group, tile_n, tile_m, swap_ab, tile_k, group_m;
};
const TunedShape kTuned[] = {
#include "tuned_shapes.inc"
    {0, 0, 0, -1, 0, 0, 0, 0, 0, 0, 0}  // end
};

}  // namespace

// Row repack of a 16-bit operand into a 16-byte-aligned pitch (repack.cu).
cudaError_t launch_repack(const void* src, int64_t ld_src, void* dst, int64_t ld_dst, int rows, int cols,
                          int src_granule, int sms, cudaStream_t stream);

namespace {

const TunedShape* tuned_entry(int64_t M, int64_t N, int64_t K, int dtype, const tgemm_options& o) {
  if (o.kernel || o.tile_n || o.group_m || o.max_ctas || o.cta_group || o.tile_k || o.stream_k || o.swap_ab ||
      o.tile_m)
    return nullptr;
  for (const TunedShape& t : kTuned)
    if (t.dtype == dtype && t.M == M && t.N == N && t.K == K) return &t;
  return nullptr;
}

int make_plan_core(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
                   const void* C, int64_t ldc, int dtype, const tgemm_options* o, int sms, int pair_cap,
                   int64_t workspace_bytes, Plan& p, int64_t batch);

// The plan of a call: the tuned options of its shape when there is an entry
// and they suit this call (pointers, alignment), else the heuristics.
int make_plan(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
              const void* C, int64_t ldc, int dtype, const tgemm_options* o, int sms, int pair_cap,
              int64_t workspace_bytes, Plan& p, int64_t batch = 1) {
  // every plan starts from the defaults: a Plan filled by an earlier call (the
  // device-free validation pass of run(), say) must not leak its choices
  p = Plan();
  tgemm_options opt;
  std::memset(&opt, 0, sizeof opt);
  if (o) opt = *o;
  if (batch == 1) {
    if (const TunedShape* t = tuned_entry(M, N, K, dtype, opt)) {
      tgemm_options tuned = opt;
      tuned.kernel = t->kernel;
      tuned.cta_group = t->cta_group;
      tuned.tile_n = t->tile_n;
      tuned.tile_m = t->tile_m;
      tuned.swap_ab = t->swap_ab;
      tuned.tile_k = t->tile_k;
      tuned.group_m = t->group_m;
      Plan q;
      if (make_plan_core(M, N, K, A, lda, B, ldb, C, ldc, dtype, &tuned, sms, pair_cap, workspace_bytes, q, batch) ==
          TGEMM_OK) {
        p = q;
        p.tuned = true;
        return TGEMM_OK;
      }
    }
  }
  return make_plan_core(M, N, K, A, lda, B, ldb, C, ldc, dtype, o, sms, pair_cap, workspace_bytes, p, batch);
}

int make_plan_core(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
                   const void* C, int64_t ldc, int dtype, const tgemm_options* o, int sms, int pair_cap,
                   int64_t workspace_bytes, Plan& p, int64_t batch) {
  if (dtype < TGEMM_F32 || dtype > TGEMM_F16_F32OUT) return TGEMM_ERR_UNSUPPORTED_DTYPE;
  if (M < 0 || N < 0 || K < 0) return TGEMM_ERR_INVALID_VALUE;
  if (M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31)) return TGEMM_ERR_TOO_LARGE;
  if (lda < std::max<int64_t>(1, K) || ldb < std::max<int64_t>(1, N) || ldc < std::max<int64_t>(1, N))
    return TGEMM_ERR_INVALID_VALUE;
  tgemm_options opt;
  std::memset(&opt, 0, sizeof opt);
  if (o) opt = *o;
  if (opt.kernel < TGEMM_KERNEL_AUTO || opt.kernel > TGEMM_KERNEL_SIMT) return TGEMM_ERR_INVALID_VALUE;
  if (opt.tile_n != 0 && !tc_valid_bn(opt.tile_n)) return TGEMM_ERR_INVALID_VALUE;
  if (opt.group_m < 0 || opt.max_ctas < 0 || opt.store_mode < 0 || opt.store_mode > 2 || opt.wait_timeout_us < 0 ||
      opt.cta_group < 0 || opt.cta_group > 2 || (opt.tile_k != 0 && opt.tile_k != 64 && opt.tile_k != 128) ||
      opt.stream_k < 0 || opt.stream_k > 2 || opt.reserved0 != 0 || opt.swap_ab < 0 || opt.swap_ab > 2 ||
      opt.repack < 0 || opt.repack > 2 || opt.reserved[0] != 0 ||
      (opt.swap_ab == 2 && (opt.stream_k == 2 || opt.cta_group == 1 || (opt.tile_n != 0 && opt.tile_n != 256))) ||
      (opt.tile_m != 0 && (opt.swap_ab != 2 || !tc2_valid_bn(opt.tile_m))))
    return TGEMM_ERR_INVALID_VALUE;
  if (M == 0 || N == 0) {
    p.noop = true;
    return TGEMM_OK;
  }
  const int ei = in_bytes(dtype), eo = out_bytes(dtype);
  if (!C) return TGEMM_ERR_INVALID_VALUE;
  if (K > 0 && (!A || !B)) return TGEMM_ERR_INVALID_VALUE;
  if (reinterpret_cast<uint64_t>(C) % eo) return TGEMM_ERR_MISALIGNED;
  if (K > 0 && (reinterpret_cast<uint64_t>(A) % ei || reinterpret_cast<uint64_t>(B) % ei)) return TGEMM_ERR_MISALIGNED;
  // byte extents of the three operands
  const uint64_t c0 = reinterpret_cast<uint64_t>(C), c1 = c0 + static_cast<uint64_t>((M - 1) * ldc + N) * eo;
  if (K > 0) {
    const uint64_t a0 = reinterpret_cast<uint64_t>(A), a1 = a0 + static_cast<uint64_t>((M - 1) * lda + K) * ei;
    const uint64_t b0 = reinterpret_cast<uint64_t>(B), b1 = b0 + static_cast<uint64_t>((K - 1) * ldb + N) * ei;
    if (ranges_overlap(c0, c1, a0, a1) || ranges_overlap(c0, c1, b0, b1)) return TGEMM_ERR_ALIAS;
  }
  if (K == 0) {
    p.zero = true;
    return TGEMM_OK;
  }
  if (opt.simt_split < 0 || opt.simt_split > 2 || (opt.simt_split != 0 && dtype != TGEMM_F32))
    return TGEMM_ERR_INVALID_VALUE;
  if (dtype == TGEMM_F32) {
    if (opt.kernel != TGEMM_KERNEL_AUTO && opt.kernel != TGEMM_KERNEL_SIMT) return TGEMM_ERR_INVALID_VALUE;
    p.kernel = TGEMM_KERNEL_SIMT;
    p.tiles_m = static_cast<int>((M + kSimtBM - 1) / kSimtBM);
    p.tiles_n = static_cast<int>((N + kSimtBN - 1) / kSimtBN);
    if (p.tiles_m > 65535) return TGEMM_ERR_TOO_LARGE;
    const int64_t tiles = static_cast<int64_t>(p.tiles_m) * p.tiles_n;
    if (tiles > INT32_MAX / 2) return TGEMM_ERR_TOO_LARGE;
    p.ctas = p.dp_tiles = static_cast<int>(tiles);
    p.k_blocks = static_cast<int>((K + kSimtBK - 1) / kSimtBK);
    {
      // Two 256-thread CTAs are resident per SM.  Tiles run in rounds of
      // 2 x SMs; a last round that fills at most half of the slots takes as
      // long as a full one, and split into K halves it takes half as long.
      const int64_t slots = 2 * static_cast<int64_t>(sms);
      const int64_t tail = tiles % slots;
      const bool fits = tail > 0 && 2 * tail <= slots && p.k_blocks >= 2;
      if (fits && (opt.simt_split == 2 || (opt.simt_split == 0 && p.k_blocks >= 16))) {
        p.dp_tiles = static_cast<int>(tiles - tail);
        p.ctas = static_cast<int>(tiles - tail + kSimtSplitWays * tail);
        p.split_stage = p.k_blocks / 2;
      }
    }
    // Raster group height: 16 tile rows keep a round of 2 x SMs resident
    // CTAs on about 16 rows of A and 19 columns of B at 152 SMs.
    p.group_m = std::max(1, std::min(opt.group_m ? opt.group_m : 16, p.tiles_m));
    p.bn = kSimtBN;
    p.stages = 2;
    p.smem = 0;
    const bool vec = reinterpret_cast<uint64_t>(A) % 16 == 0 && reinterpret_cast<uint64_t>(B) % 16 == 0 &&
                     reinterpret_cast<uint64_t>(C) % 16 == 0 && lda % 4 == 0 && ldb % 4 == 0 && ldc % 4 == 0;
    p.a_copy = p.b_copy = p.store = vec ? 16 : 4;
    // Small products: when the 128 x 128 tiles would occupy at most an
    // eighth of the SMs and K is short, 32 x 32 tiles with a deep copy ring
    // finish sooner (fixed costs dominate; more CTAs, fewer waits on DRAM).
    // Not with a forced split; the fused epilogue is supported.
    if (opt.simt_split != 2 && tiles * 8 <= sms && K <= 2048) {
      p.simt_small = true;
      p.split_stage = 0;
      p.tiles_m = static_cast<int>((M + kSimtSmallTile - 1) / kSimtSmallTile);
      p.tiles_n = static_cast<int>((N + kSimtSmallTile - 1) / kSimtSmallTile);
      if (p.tiles_m > 65535) return TGEMM_ERR_TOO_LARGE;
      p.ctas = p.dp_tiles = p.tiles_m * p.tiles_n;
      p.bn = kSimtSmallTile;
      p.stages = kSimtSmallStages;
      p.k_blocks = static_cast<int>((K + kSimtSmallK - 1) / kSimtSmallK);
      p.group_m = 1;
    }
    return TGEMM_OK;
  }
  if (opt.kernel == TGEMM_KERNEL_SIMT) return TGEMM_ERR_INVALID_VALUE;
  // bulk-tensor copies need 16-byte aligned bases and row pitches below 2^40
  const int ga = granule(A, lda, ei), gb = granule(B, ldb, ei), gc = granule(C, ldc, eo);
  const bool a_tma = ga == 16 && lda * ei < (int64_t(1) << 40);
  const bool b_tma = gb == 16 && ldb * ei < (int64_t(1) << 40);
  // A bulk-tensor store writes whole 16-byte units at the end of a row, so it
  // is used only when the row's byte extent is a multiple of 16 (otherwise it
  // would overwrite the ldc padding, or the bytes past the last row).
  const bool c_tma = gc == 16 && (N * eo) % 16 == 0 && ldc * eo < (int64_t(1) << 40);
  // Repack through the caller's workspace: an operand whose rows rule out
  // bulk-tensor copies is first copied into the workspace with a pitch of a
  // multiple of 8 elements (16 bytes), and the bulk-tensor kernels read that
  // copy.  Auto repacks an operand the product reads several times over (B
  // when M >= 512, A when N >= 512); 2 repacks any such operand, 1 never.
  // The workspace keeps its first kSkFlagBytes for stream-K flags, then the
  // partial sums (if any), then the copies.
  bool a_ok = a_tma, b_ok = b_tma;
  int64_t pack_a = 0, pack_b = 0;
  if (opt.repack != 1 && opt.kernel != TGEMM_KERNEL_TC_COPY && workspace_bytes > 0) {
    const int64_t lda_p = (K + 7) / 8 * 8, ldb_p = (N + 7) / 8 * 8;
    const bool want_a = !a_tma && (opt.repack == 2 || N >= 512) && lda_p * 2 < (int64_t(1) << 40);
    const bool want_b = !b_tma && (opt.repack == 2 || M >= 512) && ldb_p * 2 < (int64_t(1) << 40);
    const int64_t bytes_a = want_a ? (M * lda_p * 2 + 255) / 256 * 256 : 0;
    const int64_t bytes_b = want_b ? (K * ldb_p * 2 + 255) / 256 * 256 : 0;
    if ((want_a || want_b) && kSkFlagBytes + bytes_a + bytes_b <= workspace_bytes) {
      pack_a = bytes_a;
      pack_b = bytes_b;
      p.packed = (want_a ? 1 : 0) | (want_b ? 2 : 0);
      p.lda_p = lda_p;
      p.ldb_p = ldb_p;
      p.granule_a = ga;
      p.granule_b = gb;
      a_ok = a_ok || want_a;
      b_ok = b_ok || want_b;
      // what is left of the workspace for a stream-K split (its own flag
      // region is the one already reserved)
      workspace_bytes -= bytes_a + bytes_b;
    }
  }
  // byte offsets of the copies, after the stream-K region (or after the
  // reserved flag region when there is no split)
  auto place_copies = [&]() {
    if (!p.packed) return;
    const int64_t base = p.workspace > 0 ? p.workspace : kSkFlagBytes;
    p.off_a = base;
    p.off_b = base + pack_a;
    p.workspace = base + pack_a + pack_b;
  };
  if (opt.kernel == TGEMM_KERNEL_TC_TMA && (!a_ok || !b_ok)) return TGEMM_ERR_INVALID_VALUE;
  switch (opt.kernel) {
    case TGEMM_KERNEL_TC_TMA:
      p.kernel = TGEMM_KERNEL_TC_TMA;
      break;
    case TGEMM_KERNEL_TC_COPY:
      p.kernel = TGEMM_KERNEL_TC_COPY;
      p.a_copy = ga;
      p.b_copy = gb;
      break;
    default:
      p.kernel = (a_ok && b_ok) ? TGEMM_KERNEL_TC_TMA : TGEMM_KERNEL_TC_COPY;
      p.a_copy = a_ok ? 0 : ga;
      p.b_copy = b_ok ? 0 : gb;
  }
  if (opt.store_mode == 1 && !c_tma) return TGEMM_ERR_INVALID_VALUE;
  p.store = (c_tma && opt.store_mode != 2) ? 0 : gc;
  // a CTA cap limits every kind of worker
  if (opt.max_ctas) {
    sms = std::min(sms, opt.max_ctas);
    pair_cap = std::min(pair_cap, std::max(1, opt.max_ctas / 2));
  }
  // B rows that rule out bulk-tensor copies (A's do not): CTA pairs that copy
  // B per thread, each CTA its half of the tile's columns, move half the B
  // bytes per SM and FLOP of the one-SM copy kernel, which per-thread copies
  // bound.  Cost: rounds x the B columns one SM copies per tile.
  const bool copy_pair_ok = p.kernel == TGEMM_KERNEL_TC_COPY && a_ok && pair_cap > 0 &&
                            opt.cta_group != 1 && opt.swap_ab != 2 &&
                            opt.tile_k != 128 && opt.store_mode != 1 &&
                            (opt.tile_n == 0 || opt.tile_n == 128 || opt.tile_n == 256) &&
                            (opt.kernel == TGEMM_KERNEL_TC_COPY ? opt.cta_group == 2 : p.b_copy != 0);
  if (copy_pair_ok) {
    auto rounds = [&](int64_t tiles, int workers) { return static_cast<double>((tiles + workers - 1) / workers); };
    int bnc = 0;
    double cost_c = 1e300;
    for (int bn : {256, 128}) {
      if (opt.tile_n && bn != opt.tile_n) continue;
      const double c = rounds(((M + 2 * kTileM - 1) / (2 * kTileM)) * ((N + bn - 1) / bn), pair_cap) * bn / 2;
      if (c < cost_c * 0.999) {
        cost_c = c;
        bnc = bn;
      }
    }
    double cost_1 = 1e300;
    for (int bn : {256, 128, 64})
      cost_1 = std::min(cost_1, rounds(((M + kTileM - 1) / kTileM) * ((N + bn - 1) / bn), sms) * bn);
    if (opt.cta_group == 2 || cost_c < cost_1) {
      p.pair = true;
      p.copy_pair = true;
      p.bn = bnc;
      p.a_copy = 0;
      p.b_copy = gb;
      p.store = gc;  // the kernel stores C per thread
      p.ksub = 1;
      p.stages = copy_pair_stage_count(p.bn);
      p.tiles_m = static_cast<int>((M + 2 * kTileM - 1) / (2 * kTileM));
      p.tiles_n = static_cast<int>((N + p.bn - 1) / p.bn);
      const int64_t tiles = int64_t(p.tiles_m) * p.tiles_n;
      if (tiles >= (int64_t(1) << 31)) return TGEMM_ERR_TOO_LARGE;
      const int64_t in_bytes = (M * K + K * N) * 2;
      p.group_m = opt.group_m ? opt.group_m : (in_bytes <= (int64_t(64) << 20) ? 4 : 8);
      p.group_m = std::max(1, std::min(p.group_m, p.tiles_m));
      p.k_blocks = static_cast<int>((K + kTileK - 1) / kTileK);
      p.dp_tiles = static_cast<int>(tiles);
      p.ctas = static_cast<int>(2 * std::min<int64_t>(tiles, pair_cap));
      // Stream-K split of the tiles past the last full round of pairs, as in
      // the bulk-tensor pair kernel below (needs the caller's workspace).
      if (opt.stream_k == 2) {
        const int64_t cap = pair_cap;
        const int64_t rem = tiles % cap;
        const int64_t sk_iters = rem * p.k_blocks;
        const int64_t need = sk_workspace_bytes(static_cast<int>(cap), p.bn);
        if (rem != 0 && sk_iters >= cap && cap <= kSkMaxWorkers && workspace_bytes >= need &&
            sk_iters < (int64_t(1) << 31)) {
          p.dp_tiles = static_cast<int>(tiles - rem);
          p.sk_iters = static_cast<int>(sk_iters);
          p.workspace = need;
          p.ctas = static_cast<int>(2 * cap);
        }
      }
      p.smem = copy_pair_smem(p.bn);
      if (batch > 1) p.batch_loop = true;
      place_copies();
      return TGEMM_OK;
    }
  }
  // one SM per 128-row tile, or a CTA pair per 256-row tile (bulk-tensor
  // operands only)
  const bool pair_ok = p.kernel == TGEMM_KERNEL_TC_TMA && pair_cap > 0 &&
                       (opt.tile_n == 0 || tc2_valid_bn(opt.tile_n));
  if (opt.cta_group == 2 && !pair_ok) return TGEMM_ERR_INVALID_VALUE;
  double cost1 = 0, cost2 = 1e300, cost_s = 1e300;
  const int bn1 = opt.tile_n ? opt.tile_n : pick_tile_n(M, N, sms, &cost1);
  int bn2 = 0, tm_s = 0;
  if (pair_ok && opt.cta_group != 1) {
    // stream-K needs a workspace of at most sk_workspace_bytes(pairs, 256)
    const bool sk_possible = opt.stream_k == 2 && workspace_bytes >= sk_workspace_bytes(pair_cap, 256);
    bn2 = opt.tile_n ? opt.tile_n : pick_pair_tile_n(M, N, pair_cap, sk_possible, &cost2);
    // Pairs with the MMA's operands exchanged (tile tm x 256): no stream-K split.
    const bool swap_ok = opt.stream_k != 2 && opt.swap_ab != 1 &&
                         (opt.tile_n == 0 || opt.tile_n == 256);
    if (swap_ok) {
      tm_s = opt.tile_m ? opt.tile_m : pick_swap_tile_m(M, N, pair_cap, &cost_s);
      if (opt.tile_m) {
        const int64_t ts = ((M + tm_s - 1) / tm_s) * ((N + 255) / 256);
        cost_s = static_cast<double>((ts + pair_cap - 1) / pair_cap) * tm_s / swap_rate(tm_s);
      }
    }
    if (opt.tile_n) {
      const int64_t t1 = ((M + kTileM - 1) / kTileM) * ((N + bn1 - 1) / bn1);
      const int64_t t2 = ((M + 2 * kTileM - 1) / (2 * kTileM)) * ((N + bn2 - 1) / bn2);
      cost1 = static_cast<double>((t1 + sms - 1) / sms) * bn1 / width_rate(bn1);
      cost2 = static_cast<double>((t2 + pair_cap - 1) / pair_cap) * bn2 / pair_rate(bn2);
    }
  }
  p.pair = bn2 != 0 && (opt.cta_group == 2 || opt.swap_ab == 2 || (opt.cta_group == 0 && std::min(cost2, cost_s) < cost1));
  if (p.pair && tm_s != 0 && (opt.swap_ab == 2 || cost_s < cost2)) {
    p.swap = true;
    p.tm = tm_s;
    bn2 = 256;
  }
  if (opt.swap_ab == 2 && !p.swap) return TGEMM_ERR_INVALID_VALUE;
  // A strided batch runs in one launch of the swapped kernel, whose tile list
  // spans all matrices; when that kernel cannot serve it, each matrix is
  // launched on its own with the plan of a single product.
  if (batch > 1) {
    const bool in_kernel = pair_ok && opt.cta_group != 1 && opt.stream_k != 2 && opt.swap_ab != 1 &&
                           (opt.tile_n == 0 || opt.tile_n == 256);
    if (in_kernel) {
      p.pair = true;
      p.swap = true;
      p.tm = opt.tile_m ? opt.tile_m : pick_swap_tile_m(M, N, pair_cap, nullptr, batch);
      bn2 = 256;
      p.batch = batch;
    } else {
      p.batch_loop = true;
    }
  }
  if (opt.tile_k == 128 && !p.pair) return TGEMM_ERR_INVALID_VALUE;
  // 128-deep stages halve the MMA completion signals per FLOP (measured faster
  // for long K); short K keeps 64 so the last stage wastes little.
  p.ksub = p.pair && (opt.tile_k == 128 || (opt.tile_k == 0 && K >= 512)) ? 2 : 1;
  p.bn = p.pair ? bn2 : bn1;
  // the swapped kernel always keeps its staging buffers (sized by its height)
  p.stages = p.swap ? tc2_stages(p.tm, true, p.ksub)
                    : (p.pair ? tc2_stages(p.bn, p.store == 0, p.ksub) : tc_stages(p.bn));
  const int tm = p.swap ? p.tm : (p.pair ? 2 * kTileM : kTileM);
  p.tiles_m = static_cast<int>((M + tm - 1) / tm);
  p.tiles_n = static_cast<int>((N + p.bn - 1) / p.bn);
  const int64_t tiles = int64_t(p.tiles_m) * p.tiles_n * p.batch;
  if (tiles >= (int64_t(1) << 31)) return TGEMM_ERR_TOO_LARGE;
  const int sched_rows = p.tiles_m;
  // Raster group height.  8 keeps a round's A rows and B columns in L2 when
  // the operands do not fit there; when they do (A + B within half of L2),
  // 4 measured faster on GB300 (bf16 4096^3: +2.5 %; 8192^3 and
  // 4096 x 8192 x 4096 prefer 8 or more).
  const int64_t in_bytes = (M * K + K * N) * (dtype == TGEMM_F32 ? 4 : 2);
  p.group_m = opt.group_m ? opt.group_m : (in_bytes <= (int64_t(64) << 20) ? 4 : 8);
  p.group_m = std::max(1, std::min(p.group_m, sched_rows));
  p.k_blocks = static_cast<int>((K + kTileK * p.ksub - 1) / (kTileK * p.ksub));
  p.dp_tiles = static_cast<int>(int64_t(sched_rows) * p.tiles_n * p.batch);
  int64_t ctas;
  if (p.pair) {
    int64_t cap = pair_cap;
    int64_t pairs = std::min<int64_t>(tiles, cap);
    // Stream-K tail: when the last round of tiles would leave pairs idle, the
    // remaining tiles' k-stages are spread over every pair.  Needs the
    // caller's workspace; off when the round is (nearly) full or the split
    // would give a pair less than one k-stage on average.
    // Auto leaves it off: on the measured shapes (bf16 2048^3, 4096^3 on
    // GB300) the partial-sum traffic and the finishing epilogue cost more
    // than the idle part of the last round.
    if (opt.stream_k == 2) {
      const int64_t rem = tiles % cap;
      const int64_t sk_iters = rem * p.k_blocks;
      const bool worth = rem != 0 && sk_iters >= cap && cap <= kSkMaxWorkers;
      const int64_t need = sk_workspace_bytes(static_cast<int>(cap), p.bn);
      if (worth && workspace_bytes >= need && sk_iters < (int64_t(1) << 31)) {
        pairs = cap;
        p.dp_tiles = static_cast<int>(tiles - rem);
        p.sk_iters = static_cast<int>(sk_iters);
        p.workspace = need;
      }
    }
    ctas = 2 * pairs;
  } else {
    ctas = std::min<int64_t>(tiles, std::max(1, sms));
    if (opt.max_ctas) ctas = std::min<int64_t>(ctas, opt.max_ctas);
  }
  p.ctas = static_cast<int>(ctas);
  p.smem = p.swap ? tc2_smem_bytes(p.tm, true, p.ksub)
                  : (p.pair ? tc2_smem_bytes(p.bn, p.store == 0, p.ksub) : tc_smem_bytes(p.bn));
  place_copies();
  return TGEMM_OK;
}

CUtensorMapDataType tmap_type(int fmt_bytes, bool bf16) {
  if (fmt_bytes == 4) return CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  return bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

// Cache of encoded tensor maps.  A map is a pure function of its encode
// arguments (device, base address, element type, dimensions, strides, box,
// swizzle), so a cached map is reused exactly when all of them match: the
// same buffer called again with the same shape.  A buffer freed and
// reallocated at the same address with the same shape gets the same map it
// would be encoded to.  Least recently used entries are replaced; the cache is
// guarded by its own mutex.
struct MapKey {
  uint64_t base;
  uint64_t dims[3];
  uint64_t strides[2];
  uint32_t box[3];
  int32_t device, rank, type, swizzle;
};
struct MapSlot {
  MapKey key;
  CUtensorMap map;
  uint64_t stamp;  // 0: empty
};
constexpr int kMapSlots = 128;
std::mutex g_map_mutex;
MapSlot g_map_slots[kMapSlots];
uint64_t g_map_clock = 0;
std::atomic<uint64_t> g_map_hits{0}, g_map_encodes{0}, g_launch_calls{0};
// Host nanoseconds of tensor-core product calls: from entry to the launch
// call (validation, planning, tensor maps) and inside the launch call.
std::atomic<uint64_t> g_ns_prepare{0}, g_ns_launch{0};

uint64_t now_ns() {
  return static_cast<uint64_t>(
      std::chrono::duration_cast<std::chrono::nanoseconds>(std::chrono::steady_clock::now().time_since_epoch())
          .count());
}

int encode_cached(CUtensorMap* map, CUtensorMapDataType type, int rank, const void* base, const cuuint64_t* dims,
                  const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle swizzle) {
  MapKey key;
  std::memset(&key, 0, sizeof key);  // padding bytes take part in the comparison
  key.base = reinterpret_cast<uint64_t>(base);
  for (int i = 0; i < rank; ++i) {
    key.dims[i] = dims[i];
    key.box[i] = box[i];
  }
  for (int i = 0; i + 1 < rank; ++i) key.strides[i] = strides[i];
  key.device = t_device;
  key.rank = rank;
  key.type = static_cast<int32_t>(type);
  key.swizzle = static_cast<int32_t>(swizzle);
  std::lock_guard<std::mutex> lock(g_map_mutex);
  MapSlot* victim = &g_map_slots[0];
  for (MapSlot& slot : g_map_slots) {
    if (slot.stamp != 0 && slot.key.base == key.base && std::memcmp(&slot.key, &key, sizeof key) == 0) {
      slot.stamp = ++g_map_clock;
      *map = slot.map;
      g_map_hits.fetch_add(1, std::memory_order_relaxed);
      return TGEMM_OK;
    }
    if (slot.stamp < victim->stamp) victim = &slot;
  }
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, type, static_cast<cuuint32_t>(rank), const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    t_last_error = "cuTensorMapEncodeTiled (" + std::to_string(rank) + "-D) failed with CUresult " +
                   std::to_string(static_cast<int>(r));
    return TGEMM_ERR_LAUNCH;
  }
  g_map_encodes.fetch_add(1, std::memory_order_relaxed);
  victim->key = key;
  victim->map = *map;
  victim->stamp = ++g_map_clock;
  return TGEMM_OK;
}

// 2-D row-major tensor (cols x rows, pitch in bytes), box of box_cols x box_rows,
// 128-byte swizzle, zero fill outside the tensor.
int encode_2d(CUtensorMap* map, CUtensorMapDataType type, const void* base, int64_t cols, int64_t rows,
              int64_t pitch_bytes, uint32_t box_cols, uint32_t box_rows,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch_bytes)};
  const cuuint32_t box[2] = {box_cols, box_rows};
  return encode_cached(map, type, 2, base, dims, strides, box, swizzle);
}

// 3-D row-major tensor: `depth` matrices of cols x rows, `depth_bytes` apart
// (a depth of 1 for one matrix or for a batch stride of 0), box box_cols x
// box_rows x 1.
int encode_3d(CUtensorMap* map, CUtensorMapDataType type, const void* base, int64_t cols, int64_t rows,
              int64_t depth, int64_t pitch_bytes, int64_t depth_bytes, uint32_t box_cols, uint32_t box_rows,
              CUtensorMapSwizzle swizzle) {
  if (depth <= 1) depth_bytes = (rows * pitch_bytes + 15) / 16 * 16;  // unused, but must be valid
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(depth < 1 ? 1 : depth)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(pitch_bytes), static_cast<cuuint64_t>(depth_bytes)};
  const cuuint32_t box[3] = {box_cols, box_rows, 1};
  return encode_cached(map, type, 3, base, dims, strides, box, swizzle);
}

// Resident CTA pairs of the pair kernel on the current device, queried once.
// 0 when the query fails: pairs are then not used.
int pair_capacity(DeviceInfo* d) {
  std::lock_guard<std::mutex> lock(g_mutex);
  int& cap = d->pair_capacity;
  if (cap == 0) {
    int n = 0;
    if (tc_pair_capacity(&n) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = -1;
    }
    cap = n;
  }
  return cap > 0 ? cap : 0;
}

// Epoch of stream-K flags: a flag equal to the current call's epoch marks a
// partial sum written by this call.  Starts at a per-process pseudo-random
// value so that flags left in a reused workspace by another process are very
// unlikely to match; never 0 (the value of a zeroed workspace).
std::atomic<uint32_t> g_epoch{0};
uint32_t next_epoch() {
  uint32_t e = g_epoch.load();
  if (e == 0) {
    const uint64_t seed = static_cast<uint64_t>(std::chrono::steady_clock::now().time_since_epoch().count()) ^
                          (static_cast<uint64_t>(getpid()) << 32);
    uint32_t start = static_cast<uint32_t>(seed * 0x9E3779B97F4A7C15ull >> 32) | 1u;
    uint32_t expected = 0;
    g_epoch.compare_exchange_strong(expected, start);
  }
  uint32_t v;
  do {
    v = g_epoch.fetch_add(1) + 1;
  } while (v == 0);
  return v;
}

// The fused epilogue of a call, validated (no device access).  `on` stays 0
// for the plain product.
int make_epilogue(const tgemm_epilogue* in, int64_t M, int64_t N, const void* C, int64_t ldc, int dtype,
                  Epilogue& e) {
  e = Epilogue{0, 0, 1.0f, 0.0f, nullptr};
  if (!in) return TGEMM_OK;
  if (in->activation < TGEMM_ACT_NONE || in->activation > TGEMM_ACT_RELU) return TGEMM_ERR_INVALID_VALUE;
  for (int r : in->reserved)
    if (r != 0) return TGEMM_ERR_INVALID_VALUE;
  if (in->bias) {
    const uint64_t b0 = reinterpret_cast<uint64_t>(in->bias);
    if (b0 % 4) return TGEMM_ERR_INVALID_VALUE;
    if (M > 0 && N > 0) {
      const uint64_t c0 = reinterpret_cast<uint64_t>(C);
      const uint64_t c1 = c0 + static_cast<uint64_t>((M - 1) * ldc + N) * out_bytes(dtype);
      if (ranges_overlap(c0, c1, b0, b0 + static_cast<uint64_t>(N) * 4)) return TGEMM_ERR_ALIAS;
    }
  }
  e.alpha = in->alpha;
  e.beta = in->beta;
  e.bias = in->bias;
  e.act = in->activation;
  e.on = !(in->alpha == 1.0f && in->beta == 0.0f && !in->bias && in->activation == TGEMM_ACT_NONE);
  return TGEMM_OK;
}

// A strided batch: `count` products, operands of matrix b at element offsets
// b * stride_a, b * stride_b, b * stride_c.  Validated by batch_validate.
struct Batch {
  int64_t count = 1, stride_a = 0, stride_b = 0, stride_c = 0;
};

// Bulk-tensor copies need every matrix of a batch to start on a 16-byte
// boundary: the swapped kernel's 3-D maps can take the batch only then.
bool batch_tma_ok(const Batch& bt, int dtype) {
  const int ei = in_bytes(dtype);
  return (bt.stride_a * ei) % 16 == 0 && (bt.stride_b * ei) % 16 == 0;
}

int run(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
        int64_t ldc, int dtype, const tgemm_options* o, const tgemm_epilogue* epi_in, void* workspace,
        int64_t workspace_bytes, cudaStream_t stream, const Batch& bt = Batch()) {
  const uint64_t t_entry = now_ns();
  // validation that needs no device first, so bad arguments never touch CUDA
  Plan p;
  if (workspace_bytes < 0 || (workspace_bytes > 0 && (!workspace || reinterpret_cast<uint64_t>(workspace) % 256)))
    return TGEMM_ERR_INVALID_VALUE;
  const int64_t in_batch = (bt.count > 1 && batch_tma_ok(bt, dtype)) ? bt.count : 1;
  int st = make_plan(M, N, K, A, lda, B, ldb, C, ldc, dtype, o, 1, 1, workspace_bytes, p, in_batch);
  if (st != TGEMM_OK || p.noop) return st;
  Epilogue ep;
  st = make_epilogue(epi_in, M, N, C, ldc, dtype, ep);
  if (st != TGEMM_OK) return st;
  const int out_fmt = out_bytes(dtype) == 4 ? OUT_F32 : (dtype == TGEMM_BF16 ? OUT_BF16 : OUT_F16);
  DeviceInfo* dev = nullptr;
  st = device_info(&dev);
  if (st != TGEMM_OK) return st;
  st = make_plan(M, N, K, A, lda, B, ldb, C, ldc, dtype, o, dev->sm_count, pair_capacity(dev), workspace_bytes, p,
                 in_batch);
  if (st != TGEMM_OK) return st;
  if (bt.count > 1 && p.batch == 1) {
    // no kernel indexes this batch: one launch per matrix, each a single product
    const int ei = in_bytes(dtype), eo = out_bytes(dtype);
    for (int64_t b = 0; b < bt.count; ++b) {
      st = run(M, N, K, static_cast<const char*>(A) + b * bt.stride_a * ei, lda,
               static_cast<const char*>(B) + b * bt.stride_b * ei, ldb, static_cast<char*>(C) + b * bt.stride_c * eo,
               ldc, dtype, o, epi_in, workspace, workspace_bytes, stream);
      if (st != TGEMM_OK) return st;
    }
    return TGEMM_OK;
  }
  cudaError_t e;
  if (p.zero) {
    e = ep.on ? launch_epilogue_fill(C, M, N, ldc, out_fmt, ep, stream)
              : launch_zero_fill(C, M, N, ldc, out_bytes(dtype), stream);
    return e == cudaSuccess ? TGEMM_OK : cuda_fail(e, "zero-fill launch");
  }
  if (p.kernel == TGEMM_KERNEL_SIMT) {
    SimtArgs a;
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.A = static_cast<const float*>(A);
    a.lda = lda;
    a.B = static_cast<const float*>(B);
    a.ldb = ldb;
    a.C = static_cast<float*>(C);
    a.ldc = ldc;
    a.vec = p.a_copy == 16 ? 1 : 0;
    a.epi = ep;
    if (p.simt_small) {
      e = launch_simt_small(a, stream);
      return e == cudaSuccess ? TGEMM_OK : cuda_fail(e, "SIMT kernel launch");
    }
    a.tiles_m = p.tiles_m;
    a.tiles_n = p.tiles_n;
    a.group_m = p.group_m;
    a.full_tiles = p.dp_tiles;
    a.split_stage = p.split_stage;
    int64_t units = p.ctas;
    if (ep.on || p.split_stage == 0) {
      // an epilogue is applied once to the whole sum: every tile whole
      a.full_tiles = p.tiles_m * p.tiles_n;
      a.split_stage = 0;
      units = a.full_tiles;
    } else {
      // the halves add into zeros: clear the bounding box of the split tiles
      // (a whole tile inside it is stored over the zeros)
      int r_lo = p.tiles_m, r_hi = -1, c_lo = p.tiles_n, c_hi = -1;
      for (int t = p.dp_tiles; t < p.tiles_m * p.tiles_n; ++t) {
        int r, c;
        simt_tile_coords(t, p.tiles_m, p.tiles_n, p.group_m, r, c);
        r_lo = std::min(r_lo, r);
        r_hi = std::max(r_hi, r);
        c_lo = std::min(c_lo, c);
        c_hi = std::max(c_hi, c);
      }
      const int64_t r0 = int64_t(r_lo) * kSimtBM, r1 = std::min<int64_t>(M, int64_t(r_hi + 1) * kSimtBM);
      const int64_t c0 = int64_t(c_lo) * kSimtBN, c1 = std::min<int64_t>(N, int64_t(c_hi + 1) * kSimtBN);
      e = launch_zero_fill(static_cast<float*>(C) + r0 * ldc + c0, r1 - r0, c1 - c0, ldc, 4, stream);
      if (e != cudaSuccess) return cuda_fail(e, "zero-fill launch");
    }
    e = launch_simt(a, units, stream);
    return e == cudaSuccess ? TGEMM_OK : cuda_fail(e, "SIMT kernel launch");
  }
  const bool bf16 = (dtype == TGEMM_BF16 || dtype == TGEMM_BF16_F32OUT);
  const int eo = out_bytes(dtype);
  // operands repacked into the workspace: copy them, then read the copies
  if (p.packed & 1) {
    void* dst = static_cast<char*>(workspace) + p.off_a;
    e = launch_repack(A, lda, dst, p.lda_p, static_cast<int>(M), static_cast<int>(K), p.granule_a, dev->sm_count,
                      stream);
    if (e != cudaSuccess) return cuda_fail(e, "repack launch");
    A = dst;
    lda = p.lda_p;
  }
  if (p.packed & 2) {
    void* dst = static_cast<char*>(workspace) + p.off_b;
    e = launch_repack(B, ldb, dst, p.ldb_p, static_cast<int>(K), static_cast<int>(N), p.granule_b, dev->sm_count,
                      stream);
    if (e != cudaSuccess) return cuda_fail(e, "repack launch");
    B = dst;
    ldb = p.ldb_p;
  }
  CUtensorMap mA, mB, mBt, mC;
  std::memset(&mA, 0, sizeof mA);
  std::memset(&mB, 0, sizeof mB);
  std::memset(&mBt, 0, sizeof mBt);
  std::memset(&mC, 0, sizeof mC);
  // The swapped pair kernel: 3-D maps (the batch is the third dimension), tm/2
  // rows of A per CTA, C in unswizzled 32 x 32 blocks (bulk stores only when
  // every matrix of C starts on a 16-byte boundary).
  if (p.swap && p.batch > 1 && p.store == 0 && (bt.stride_c * eo) % 16 != 0) p.store = eo;
  if (p.swap) {
    const int64_t nb = p.batch;
    if ((st = encode_3d(&mA, tmap_type(2, bf16), A, K, M, bt.stride_a ? nb : 1, lda * 2, bt.stride_a * 2, kTileK,
                        static_cast<uint32_t>(p.tm / 2), CU_TENSOR_MAP_SWIZZLE_128B)) != TGEMM_OK)
      return st;
    if ((st = encode_3d(&mB, tmap_type(2, bf16), B, N, K, bt.stride_b ? nb : 1, ldb * 2, bt.stride_b * 2, 64, kTileK,
                        CU_TENSOR_MAP_SWIZZLE_128B)) != TGEMM_OK)
      return st;
    if (p.store == 0 && (st = encode_3d(&mC, tmap_type(eo, dtype == TGEMM_BF16), C, N, M, nb, ldc * eo,
                                        bt.stride_c * eo, 32, 32, CU_TENSOR_MAP_SWIZZLE_NONE)) != TGEMM_OK)
      return st;
  }
  if (!p.swap && p.a_copy == 0 &&
      (st = encode_2d(&mA, tmap_type(2, bf16), A, K, M, lda * 2, kTileK, kTileM)) != TGEMM_OK)
    return st;
  if (!p.swap && p.b_copy == 0 &&
      (st = encode_2d(&mB, tmap_type(2, bf16), B, N, K, ldb * 2, 64, kTileK)) != TGEMM_OK)
    return st;
  // the pair kernel's last, partial B atom (bn/2 = 96 or 112 columns per CTA)
  const uint32_t b_tail = (p.pair && !p.swap) ? static_cast<uint32_t>((p.bn / 2) % 64) : 0u;
  if (b_tail && (st = encode_2d(&mBt, tmap_type(2, bf16), B, N, K, ldb * 2, b_tail, kTileK)) != TGEMM_OK) return st;
  // C: 128-byte swizzled 32-row boxes; the swapped kernel writes unswizzled 32 x 32 blocks
  if (!p.swap && p.store == 0 &&
      (st = encode_2d(&mC, tmap_type(eo, dtype == TGEMM_BF16), C, N, M, ldc * eo, 128 / eo, 32)) != TGEMM_OK)
    return st;
  TcArgs a;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.tiles_m = p.tiles_m;
  a.tiles_n = p.tiles_n;
  a.tiles_per = a.tiles_m * p.tiles_n;
  a.num_tiles = static_cast<int>(a.tiles_per * p.batch);
  a.stride_a = p.batch > 1 ? bt.stride_a : 0;
  a.stride_b = p.batch > 1 ? bt.stride_b : 0;
  a.stride_c = p.batch > 1 ? bt.stride_c : 0;
  a.k_blocks = p.k_blocks;
  a.dp_tiles = p.dp_tiles;
  a.sk_iters = p.sk_iters;
  a.sk_partials = nullptr;
  a.sk_flags = nullptr;
  a.sk_epoch = 0;
  if (p.sk_iters) {
    a.sk_flags = static_cast<unsigned int*>(workspace);
    a.sk_partials = reinterpret_cast<float*>(static_cast<char*>(workspace) + kSkFlagBytes);
    a.sk_epoch = next_epoch();
  }
  a.group_m = p.group_m;
  a.A = A;
  a.lda = lda;
  a.B = B;
  a.ldb = ldb;
  a.C = C;
  a.ldc = ldc;
  const uint32_t ab = bf16 ? 1u : 0u;
  // kind::f16 instruction descriptor: D fp32 (bits 4-5 = 1), A/B format
  // (bits 7-9, 10-12), A K-major (bit 15 = 0), B N-major (bit 16 = 1),
  // N >> 3 (bits 17-22), M >> 4 (bits 24-28).
  // The swapped kernel's MMA takes B as its A operand (N-major, bit 15 = 1),
  // A as its B operand (K-major, bit 16 = 0), M = 256 and N = tm.
  const uint32_t mma_m = p.pair ? 2 * kTileM : kTileM;
  if (p.swap)
    a.idesc = (1u << 4) | (ab << 7) | (ab << 10) | (1u << 15) | (static_cast<uint32_t>(p.tm >> 3) << 17) |
              ((mma_m >> 4) << 24);
  else
    a.idesc = (1u << 4) | (ab << 7) | (ab << 10) | (1u << 16) | (static_cast<uint32_t>(p.bn >> 3) << 17) |
              ((mma_m >> 4) << 24);
  a.out_fmt = out_fmt;
  a.epi = ep;
  a.a_copy = p.a_copy;
  a.b_copy = p.b_copy;
  a.store_granule = p.store;
  a.inject_fault = (o && o->inject_fault) ? 1 : 0;
  const int to_us = (o && o->wait_timeout_us) ? o->wait_timeout_us : 2000000;
  a.timeout_ns = static_cast<unsigned long long>(to_us) * 1000ull;
  a.status = dev->status;
  a.pdl = p.packed ? 1 : 0;  // the product follows its operands' repack on the stream
  g_launch_calls.fetch_add(1, std::memory_order_relaxed);
  const uint64_t t_launch = now_ns();
  if (p.copy_pair)
    e = launch_tc_pair_copy(p.bn, mA, a, p.ctas / 2, stream);
  else if (p.swap)
    e = launch_tc_pair_swap(p.tm, p.ksub, mA, mB, mC, a, p.ctas / 2, stream);
  else if (p.pair)
    e = launch_tc_pair(p.bn, p.store == 0, p.ksub, mA, mB, mBt, mC, a, p.ctas / 2, stream);
  else
    e = launch_tc(p.bn, p.kernel == TGEMM_KERNEL_TC_COPY, mA, mB, mC, a, p.ctas, stream);
  const uint64_t t_done = now_ns();
  g_ns_prepare.fetch_add(t_launch - t_entry, std::memory_order_relaxed);
  g_ns_launch.fetch_add(t_done - t_launch, std::memory_order_relaxed);
  return e == cudaSuccess ? TGEMM_OK : cuda_fail(e, "tensor-core kernel launch");
}

}  // namespace
}  // namespace tgemm

extern "C" {

int tgemm_gemm(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
               int64_t ldc, int dtype, void* stream) {
  return tgemm::run(M, N, K, A, lda, B, ldb, C, ldc, dtype, nullptr, nullptr, nullptr, 0, static_cast<cudaStream_t>(stream));
}

int tgemm_gemm_ex(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
                  int64_t ldc, int dtype, const tgemm_options* opts, void* stream) {
  return tgemm::run(M, N, K, A, lda, B, ldb, C, ldc, dtype, opts, nullptr, nullptr, 0, static_cast<cudaStream_t>(stream));
}

int tgemm_gemm_ws(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
                  int64_t ldc, int dtype, const tgemm_options* opts, void* workspace, size_t workspace_bytes,
                  void* stream) {
  if (workspace_bytes > static_cast<size_t>(INT64_MAX)) return TGEMM_ERR_INVALID_VALUE;
  return tgemm::run(M, N, K, A, lda, B, ldb, C, ldc, dtype, opts, nullptr, workspace,
                    static_cast<int64_t>(workspace_bytes),
                    static_cast<cudaStream_t>(stream));
}

int tgemm_gemm_epilogue(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
                        void* C, int64_t ldc, int dtype, const tgemm_epilogue* epi, const tgemm_options* opts,
                        void* workspace, size_t workspace_bytes, void* stream) {
  if (workspace_bytes > static_cast<size_t>(INT64_MAX)) return TGEMM_ERR_INVALID_VALUE;
  return tgemm::run(M, N, K, A, lda, B, ldb, C, ldc, dtype, opts, epi, workspace,
                    static_cast<int64_t>(workspace_bytes), static_cast<cudaStream_t>(stream));
}

namespace tgemm {
namespace {
// Host checks of a strided batch: sizes, strides, disjoint C windows, and no
// overlap between the whole of C and the whole of A or B.
int batch_validate(int64_t batch, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, int64_t sa,
                   const void* B, int64_t ldb, int64_t sb, const void* C, int64_t ldc, int64_t sc, int dtype) {
  if (batch < 0 || sa < 0 || sb < 0 || sc < 0) return TGEMM_ERR_INVALID_VALUE;
  if (dtype < TGEMM_F32 || dtype > TGEMM_F16_F32OUT) return TGEMM_ERR_UNSUPPORTED_DTYPE;
  if (batch <= 1 || M <= 0 || N <= 0) return TGEMM_OK;  // the single-product checks cover the rest
  if (batch >= (int64_t(1) << 31) || sa >= (int64_t(1) << 40) || sb >= (int64_t(1) << 40) ||
      sc >= (int64_t(1) << 40))
    return TGEMM_ERR_TOO_LARGE;
  const int64_t c_span = (M - 1) * ldc + N;  // elements of one matrix's window of C
  if (sc < c_span) return TGEMM_ERR_ALIAS;    // the products would write the same elements
  if (K > 0 && A && B && C) {
    const int ei = in_bytes(dtype), eo = out_bytes(dtype);
    const uint64_t c0 = reinterpret_cast<uint64_t>(C), c1 = c0 + static_cast<uint64_t>((batch - 1) * sc + c_span) * eo;
    const uint64_t a0 = reinterpret_cast<uint64_t>(A);
    const uint64_t a1 = a0 + static_cast<uint64_t>((batch - 1) * sa + (M - 1) * lda + K) * ei;
    const uint64_t b0 = reinterpret_cast<uint64_t>(B);
    const uint64_t b1 = b0 + static_cast<uint64_t>((batch - 1) * sb + (K - 1) * ldb + N) * ei;
    if (ranges_overlap(c0, c1, a0, a1) || ranges_overlap(c0, c1, b0, b1)) return TGEMM_ERR_ALIAS;
  }
  return TGEMM_OK;
}
}  // namespace
}  // namespace tgemm

int tgemm_gemm_batched(int64_t batch, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, int64_t stride_a,
                       const void* B, int64_t ldb, int64_t stride_b, void* C, int64_t ldc, int64_t stride_c, int dtype,
                       const tgemm_epilogue* epi, const tgemm_options* opts, void* stream) {
  int st = tgemm::batch_validate(batch, M, N, K, A, lda, stride_a, B, ldb, stride_b, C, ldc, stride_c, dtype);
  if (st != TGEMM_OK || batch == 0) return st;
  tgemm::Batch bt;
  bt.count = batch;
  bt.stride_a = stride_a;
  bt.stride_b = stride_b;
  bt.stride_c = stride_c;
  return tgemm::run(M, N, K, A, lda, B, ldb, C, ldc, dtype, opts, epi, nullptr, 0, static_cast<cudaStream_t>(stream),
                    bt);
}

int tgemm_plan_batched(int64_t batch, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, int64_t stride_a,
                       const void* B, int64_t ldb, int64_t stride_b, const void* C, int64_t ldc, int64_t stride_c,
                       int dtype, const tgemm_options* opts, int sm_count, tgemm_plan_info* out, int* launches) {
  if (out) std::memset(out, 0, sizeof *out);
  if (launches) *launches = 0;
  int st = tgemm::batch_validate(batch, M, N, K, A, lda, stride_a, B, ldb, stride_b, C, ldc, stride_c, dtype);
  if (st != TGEMM_OK || batch == 0) return st;
  tgemm::Batch bt;
  bt.count = batch;
  bt.stride_a = stride_a;
  bt.stride_b = stride_b;
  const int64_t in_batch = (batch > 1 && tgemm::batch_tma_ok(bt, dtype)) ? batch : 1;
  const int sms = sm_count < 1 ? 1 : sm_count;
  tgemm::Plan p;
  st = tgemm::make_plan(M, N, K, A, lda, B, ldb, C, ldc, dtype, opts, sms, sms / 2, 0, p, in_batch);
  if (st != TGEMM_OK) return st;
  // an fp32 product split into K halves is a zero fill plus the product
  const int per_product = (p.kernel == TGEMM_KERNEL_SIMT && p.split_stage > 0) ? 2 : 1;
  if (launches)
    *launches = p.noop ? 0 : per_product * (batch > 1 && p.batch == 1 ? static_cast<int>(batch) : 1);
  if (out) {
    st = tgemm_plan(M, N, K, A, lda, B, ldb, C, ldc, dtype, opts, 0, sm_count, out);
    if (st == TGEMM_OK && p.batch > 1) {
      out->tile_m = p.tm;
      out->tile_n = p.bn;
      out->stages = p.stages;
      out->tiles_m = p.tiles_m;
      out->tiles_n = p.tiles_n;
      out->ctas = p.ctas;
      out->dp_tiles = p.dp_tiles;
      out->cta_group = 2;
      out->cluster_ctas = 2;
      out->swap_ab = 1;
      out->smem_bytes = p.smem;
      out->group_m = p.group_m;
      out->tile_k = tgemm::kTileK * p.ksub;
      // C windows that do not all start on a 16-byte boundary are stored per thread
      if (out->store_bytes == 0 && (stride_c * tgemm::out_bytes(dtype)) % 16 != 0)
        out->store_bytes = tgemm::out_bytes(dtype);
    }
  }
  return st;
}

int tgemm_transpose(int64_t rows, int64_t cols, const void* src, int64_t ld_src, void* dst, int64_t ld_dst,
                    int elem_bytes, void* stream) {
  if (rows < 0 || cols < 0) return TGEMM_ERR_INVALID_VALUE;
  if (elem_bytes != 2 && elem_bytes != 4) return TGEMM_ERR_UNSUPPORTED_DTYPE;
  if (rows >= (int64_t(1) << 31) || cols >= (int64_t(1) << 31) || (rows + 63) / 64 > 65535) return TGEMM_ERR_TOO_LARGE;
  if (ld_src < std::max<int64_t>(1, cols) || ld_dst < std::max<int64_t>(1, rows)) return TGEMM_ERR_INVALID_VALUE;
  if (rows == 0 || cols == 0) return TGEMM_OK;
  if (!src || !dst) return TGEMM_ERR_INVALID_VALUE;
  const uint64_t s0 = reinterpret_cast<uint64_t>(src), d0 = reinterpret_cast<uint64_t>(dst);
  if (s0 % elem_bytes || d0 % elem_bytes) return TGEMM_ERR_MISALIGNED;
  const uint64_t s1 = s0 + static_cast<uint64_t>((rows - 1) * ld_src + cols) * elem_bytes;
  const uint64_t d1 = d0 + static_cast<uint64_t>((cols - 1) * ld_dst + rows) * elem_bytes;
  if (tgemm::ranges_overlap(s0, s1, d0, d1)) return TGEMM_ERR_ALIAS;
  tgemm::DeviceInfo* dev = nullptr;
  int st = tgemm::device_info(&dev);
  if (st != TGEMM_OK) return st;
  const bool vec = s0 % 16 == 0 && d0 % 16 == 0 && (ld_src * elem_bytes) % 16 == 0 && (ld_dst * elem_bytes) % 16 == 0;
  const cudaError_t e = tgemm::launch_transpose(src, ld_src, dst, ld_dst, static_cast<int>(rows), static_cast<int>(cols),
                                                elem_bytes, vec, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TGEMM_OK : tgemm::cuda_fail(e, "transpose launch");
}

int tgemm_gemm_host(int64_t M, int64_t N, int64_t K, const void* A_host, int64_t lda, const void* B_host, int64_t ldb,
                    void* C_host, int64_t ldc, int dtype, void* dA, void* dB, void* dC, int panels, void* stream) {
  using tgemm::ranges_overlap;
  if (dtype < TGEMM_F32 || dtype > TGEMM_F16_F32OUT) return TGEMM_ERR_UNSUPPORTED_DTYPE;
  if (M < 0 || N < 0 || K < 0 || panels < 0) return TGEMM_ERR_INVALID_VALUE;
  if (M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31)) return TGEMM_ERR_TOO_LARGE;
  if (lda < std::max<int64_t>(1, K) || ldb < std::max<int64_t>(1, N) || ldc < std::max<int64_t>(1, N))
    return TGEMM_ERR_INVALID_VALUE;
  if (M == 0 || N == 0) return TGEMM_OK;
  const int ei = tgemm::in_bytes(dtype), eo = tgemm::out_bytes(dtype);
  if (!C_host || !dC || (K > 0 && (!A_host || !B_host || !dA || !dB))) return TGEMM_ERR_INVALID_VALUE;
  auto misaligned = [](const void* q, int e) { return reinterpret_cast<uint64_t>(q) % e != 0; };
  if (misaligned(C_host, eo) || misaligned(dC, eo)) return TGEMM_ERR_MISALIGNED;
  if (K > 0 && (misaligned(A_host, ei) || misaligned(B_host, ei) || misaligned(dA, ei) || misaligned(dB, ei)))
    return TGEMM_ERR_MISALIGNED;
  const uint64_t c0 = reinterpret_cast<uint64_t>(dC), c1 = c0 + static_cast<uint64_t>(M * N * eo);
  if (K > 0) {
    const uint64_t a0 = reinterpret_cast<uint64_t>(dA), a1 = a0 + static_cast<uint64_t>(M * K * ei);
    const uint64_t b0 = reinterpret_cast<uint64_t>(dB), b1 = b0 + static_cast<uint64_t>(K * N * ei);
    if (ranges_overlap(a0, a1, b0, b1) || ranges_overlap(c0, c1, a0, a1) || ranges_overlap(c0, c1, b0, b1))
      return TGEMM_ERR_ALIAS;
  }
  // Row panels, so that the copy of one panel of C back to the host overlaps
  // the copies in and the products of the next.  What can overlap is C's copy,
  // and it can start only once all of B, the first panel of A and that
  // panel's product are done.  Auto: one panel when C is below 6 MB (nothing
  // to overlap); above, graduated whole numbers of 128-row tiles, u, u, 2u,
  // then 4u, with u about M/16, so C's copy starts early and the later
  // products stay large (bf16 4096^3 -> fp32 on GB300: 772 us in one panel,
  // 625 us in six even panels, 605-610 us in 256, 256, 512, 1024, 1024, 1024
  // rows; the copy engines move about 200 GB/s each way, 335 GB/s both ways).
  // An explicit panel count gives even panels.
  const int64_t c_bytes = M * N * eo;
  std::vector<int64_t> panel_rows;
  if (panels) {
    const int64_t want = std::min<int64_t>(panels, M), per = (M + want - 1) / want;
    for (int64_t r0 = 0; r0 < M; r0 += per) panel_rows.push_back(std::min(per, M - r0));
  } else if (c_bytes < (int64_t(6) << 20)) {
    panel_rows.push_back(M);
  } else {
    const int64_t u = std::max<int64_t>(128, M / 16 / 128 * 128);
    int64_t r0 = 0;
    for (int i = 0; r0 < M; ++i) {
      const int64_t r = std::min(M - r0, i < 2 ? u : (i == 2 ? 2 * u : 4 * u));
      panel_rows.push_back(r);
      r0 += r;
    }
  }
  const int64_t npanels = static_cast<int64_t>(panel_rows.size());

  tgemm::DeviceInfo* dev = nullptr;
  int st = tgemm::device_info(&dev);
  if (st != TGEMM_OK) return st;
  cudaStream_t in = nullptr, out = nullptr;
  if ((st = tgemm::copy_streams(&in, &out)) != TGEMM_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Early first panel (fp32 output, several panels, K >= 256): the first
  // panel's product runs in two K halves, the first while the second half of
  // B is still being copied (B's rows are contiguous, so its first K1 rows
  // arrive first), the second added onto it (beta = 1) once B is complete.
  // The copy of C back, the longest leg, then starts sooner.  The partial sum
  // is rounded once to fp32, well inside the product's error bound; 16-bit
  // outputs keep the single pass.
  const bool split_first = K >= 256 && npanels > 1 && eo == 4 && dtype != TGEMM_F32;
  const int64_t k1 = split_first ? K / 2 / 64 * 64 : K;
  tgemm::CallEvents evs;
  cudaError_t e = cudaGetDevice(&evs.dev);
  if (e != cudaSuccess) return tgemm::cuda_fail(e, "cudaGetDevice");
  if (evs.dev < 0 || evs.dev >= 64) return tgemm::cuda_fail(cudaErrorInvalidDevice, "device ordinal");
  cudaEvent_t ev_start, ev_b, ev_b1, ev_done;
  std::vector<cudaEvent_t> ev_a(npanels), ev_c(npanels);
  if ((e = evs.make(&ev_start)) != cudaSuccess || (e = evs.make(&ev_b)) != cudaSuccess ||
      (e = evs.make(&ev_b1)) != cudaSuccess || (e = evs.make(&ev_done)) != cudaSuccess)
    return tgemm::cuda_fail(e, "cudaEventCreate");
  for (int64_t p = 0; p < npanels; ++p)
    if ((e = evs.make(&ev_a[p])) != cudaSuccess || (e = evs.make(&ev_c[p])) != cudaSuccess)
      return tgemm::cuda_fail(e, "cudaEventCreate");
  // both copy streams follow the work already on `stream` (it may still use
  // the device buffers or the host memory of C)
  if ((e = cudaEventRecord(ev_start, s)) != cudaSuccess || (e = cudaStreamWaitEvent(in, ev_start, 0)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(out, ev_start, 0)) != cudaSuccess)
    return tgemm::cuda_fail(e, "stream ordering");
  const char* ah = static_cast<const char*>(A_host);
  char* ch = static_cast<char*>(C_host);
  char* da = static_cast<char*>(dA);
  char* dc = static_cast<char*>(dC);
  if (K > 0) {
    const char* bh = static_cast<const char*>(B_host);
    char* db = static_cast<char*>(dB);
    if (split_first) {
      // the first panel of A, then B's first K1 rows, then the rest of B
      if ((e = tgemm::copy_rows(da, K * ei, ah, lda * ei, K * ei, panel_rows[0], cudaMemcpyHostToDevice, in)) !=
              cudaSuccess ||
          (e = cudaEventRecord(ev_a[0], in)) != cudaSuccess ||
          (e = tgemm::copy_rows(db, N * ei, bh, ldb * ei, N * ei, k1, cudaMemcpyHostToDevice, in)) != cudaSuccess ||
          (e = cudaEventRecord(ev_b1, in)) != cudaSuccess)
        return tgemm::cuda_fail(e, "copy of B");
    }
    if ((e = tgemm::copy_rows(db + k1 * N * ei * (split_first ? 1 : 0), N * ei,
                              bh + k1 * ldb * ei * (split_first ? 1 : 0), ldb * ei, N * ei, split_first ? K - k1 : K,
                              cudaMemcpyHostToDevice, in)) != cudaSuccess ||
        (e = cudaEventRecord(ev_b, in)) != cudaSuccess)
      return tgemm::cuda_fail(e, "copy of B");
    if (!split_first && (e = cudaStreamWaitEvent(s, ev_b, 0)) != cudaSuccess)
      return tgemm::cuda_fail(e, "stream ordering");
    for (int64_t p = split_first ? 1 : 0, r0 = split_first ? panel_rows[0] : 0; p < npanels;
         r0 += panel_rows[p], ++p) {
      const int64_t rows = panel_rows[p];
      if ((e = tgemm::copy_rows(da + r0 * K * ei, K * ei, ah + r0 * lda * ei, lda * ei, K * ei, rows,
                                cudaMemcpyHostToDevice, in)) != cudaSuccess ||
          (e = cudaEventRecord(ev_a[p], in)) != cudaSuccess)
        return tgemm::cuda_fail(e, "copy of A");
    }
  }
  for (int64_t p = 0, r0 = 0; p < npanels; r0 += panel_rows[p], ++p) {
    const int64_t rows = panel_rows[p];
    if (K > 0 && (e = cudaStreamWaitEvent(s, ev_a[p], 0)) != cudaSuccess) return tgemm::cuda_fail(e, "stream ordering");
    if (split_first && p == 0) {
      // K1 rows of B have arrived: the first half of the first panel's product
      if ((e = cudaStreamWaitEvent(s, ev_b1, 0)) != cudaSuccess) return tgemm::cuda_fail(e, "stream ordering");
      st = tgemm_gemm(rows, N, k1, da, K, dB, N, dc, N, dtype, stream);
      if (st != TGEMM_OK) return st;
      // all of B: the second half, added onto the first
      if ((e = cudaStreamWaitEvent(s, ev_b, 0)) != cudaSuccess) return tgemm::cuda_fail(e, "stream ordering");
      tgemm_epilogue acc_onto;
      std::memset(&acc_onto, 0, sizeof acc_onto);
      acc_onto.alpha = 1.0f;
      acc_onto.beta = 1.0f;
      st = tgemm_gemm_epilogue(rows, N, K - k1, da + k1 * ei, K, static_cast<char*>(dB) + k1 * N * ei, N, dc, N, dtype,
                               &acc_onto, nullptr, nullptr, 0, stream);
    } else {
      st = tgemm_gemm(rows, N, K, K > 0 ? da + r0 * K * ei : nullptr, K > 0 ? K : 1, dB, N, dc + r0 * N * eo, N,
                      dtype, stream);
    }
    if (st != TGEMM_OK) return st;
    if ((e = cudaEventRecord(ev_c[p], s)) != cudaSuccess || (e = cudaStreamWaitEvent(out, ev_c[p], 0)) != cudaSuccess ||
        (e = tgemm::copy_rows(ch + r0 * ldc * eo, ldc * eo, dc + r0 * N * eo, N * eo, N * eo, rows,
                              cudaMemcpyDeviceToHost, out)) != cudaSuccess)
      return tgemm::cuda_fail(e, "copy of C");
  }
  // later work on `stream` follows the last copy of C
  if ((e = cudaEventRecord(ev_done, out)) != cudaSuccess || (e = cudaStreamWaitEvent(s, ev_done, 0)) != cudaSuccess)
    return tgemm::cuda_fail(e, "stream ordering");
  return TGEMM_OK;
}

int tgemm_workspace_size(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
                         const void* C, int64_t ldc, int dtype, const tgemm_options* opts, size_t* bytes) {
  if (!bytes) return TGEMM_ERR_INVALID_VALUE;
  *bytes = 0;
  tgemm::Plan p;
  // validated as the call would be with an unbounded workspace (a forced
  // bulk-tensor option may be possible only with a repacked operand)
  int st = tgemm::make_plan(M, N, K, A, lda, B, ldb, C, ldc, dtype, opts, 1, 1, INT64_MAX, p);
  if (st != TGEMM_OK || p.noop || p.zero) return st;
  tgemm::DeviceInfo* dev = nullptr;
  st = tgemm::device_info(&dev);
  if (st != TGEMM_OK) return st;
  st = tgemm::make_plan(M, N, K, A, lda, B, ldb, C, ldc, dtype, opts, dev->sm_count, tgemm::pair_capacity(dev),
                        INT64_MAX, p);
  if (st == TGEMM_OK) *bytes = static_cast<size_t>(p.workspace);
  return st;
}

int tgemm_plan(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb, const void* C,
               int64_t ldc, int dtype, const tgemm_options* opts, size_t workspace_bytes, int sm_count,
               tgemm_plan_info* out) {
  tgemm::Plan p;
  const int sms = sm_count < 1 ? 1 : sm_count;
  const int64_t ws = workspace_bytes > static_cast<size_t>(INT64_MAX) ? INT64_MAX : static_cast<int64_t>(workspace_bytes);
  const int st = tgemm::make_plan(M, N, K, A, lda, B, ldb, C, ldc, dtype, opts, sms, sms / 2, ws, p);
  if (out) {
    std::memset(out, 0, sizeof *out);
    if (st == TGEMM_OK && !p.noop && !p.zero) {
      out->kernel = p.kernel;
      out->tile_m = p.kernel == TGEMM_KERNEL_SIMT ? (p.simt_small ? tgemm::kSimtSmallTile : tgemm::kSimtBM)
                                                  : (p.swap ? p.tm : (p.pair ? 2 : 1) * tgemm::kTileM);
      out->tile_n = p.bn;
      out->tile_k = p.kernel == TGEMM_KERNEL_SIMT ? (p.simt_small ? tgemm::kSimtSmallK : tgemm::kSimtBK)
                                                  : tgemm::kTileK * p.ksub;
      out->stages = p.stages;
      out->tiles_m = p.tiles_m;
      out->tiles_n = p.tiles_n;
      out->ctas = p.ctas;
      out->group_m = p.group_m;
      out->a_copy_bytes = p.a_copy;
      out->b_copy_bytes = p.b_copy;
      out->store_bytes = p.store;
      out->smem_bytes = p.smem;
      out->cta_group = p.pair ? 2 : 1;
      out->cluster_ctas = p.pair ? 2 : 1;
      out->swap_ab = p.swap ? 1 : 0;
      out->tuned = p.tuned ? 1 : 0;
      out->dp_tiles = p.dp_tiles;
      out->sk_iters = p.sk_iters;
      out->workspace_bytes = p.workspace;
      out->packed = p.packed;
    }
  }
  return st;
}

int tgemm_device_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return tgemm::cuda_fail(e, "cudaStreamSynchronize");
  tgemm::DeviceInfo* dev = nullptr;
  int st = tgemm::device_info(&dev);
  if (st != TGEMM_OK) return st;
  unsigned int word = 0;
  if ((e = cudaMemcpy(&word, dev->status, sizeof word, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return tgemm::cuda_fail(e, "reading the device status word");
  if (word == 0) return TGEMM_OK;
  const unsigned int zero = 0;
  if ((e = cudaMemcpy(dev->status, &zero, sizeof zero, cudaMemcpyHostToDevice)) != cudaSuccess)
    return tgemm::cuda_fail(e, "clearing the device status word");
  tgemm::t_last_error = "bounded wait gave up at site " + std::to_string(word & 0xFFu);
  return TGEMM_ERR_DEVICE_TIMEOUT;
}

const char* tgemm_status_string(int status) {
  switch (status) {
    case TGEMM_OK: return "success";
    case TGEMM_ERR_INVALID_VALUE: return "invalid value (size, leading dimension, pointer or option)";
    case TGEMM_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype";
    case TGEMM_ERR_MISALIGNED: return "pointer not aligned to its element size";
    case TGEMM_ERR_ALIAS: return "C overlaps A or B";
    case TGEMM_ERR_UNSUPPORTED_DEVICE: return "current device is not compute capability 10.3 (sm_103a)";
    case TGEMM_ERR_LAUNCH: return tgemm::t_last_error.empty() ? "CUDA error" : tgemm::t_last_error.c_str();
    case TGEMM_ERR_DEVICE_TIMEOUT: return "a kernel gave up a bounded wait";
    case TGEMM_ERR_TOO_LARGE: return "size too large";
    default: return "unknown status";
  }
}

int tgemm_version(void) { return TGEMM_VERSION; }

int tgemm_host_counters(tgemm_counters* out) {
  if (!out) return TGEMM_ERR_INVALID_VALUE;
  out->tc_launches = tgemm::g_launch_calls.load(std::memory_order_relaxed);
  out->map_hits = tgemm::g_map_hits.load(std::memory_order_relaxed);
  out->map_encodes = tgemm::g_map_encodes.load(std::memory_order_relaxed);
  out->ns_prepare = tgemm::g_ns_prepare.load(std::memory_order_relaxed);
  out->ns_launch = tgemm::g_ns_launch.load(std::memory_order_relaxed);
  return TGEMM_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free entry point.
//
// Some callers cannot allocate device memory when they multiply: a host
// application or plug-in host that hands out all device memory through its own
// pool at start-up, or a service whose memory budget is fixed after
// initialisation, cannot give this library a workspace and must not see it
// call cudaMalloc.  tgemm_gemm_noalloc serves them.  It runs the stream-K
// variant of the CTA-pair kernel, whose partial sums and flags live in the
// static device array below instead of a caller workspace.  The array belongs
// to the library image: every GPU that loads the library holds it until the
// process exits.
static constexpr size_t kNoAllocScratchBytes = TGEMM_NOALLOC_SCRATCH_BYTES;  // 4 KiB of flags + 20 MiB
static_assert(kNoAllocScratchBytes == size_t(tgemm::kSkFlagBytes) + (size_t(20) << 20), "scratch layout");
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[64] = {};

// Device address of the scratch array on the current device, looked up once
// per device with that device current (the host-side name of the array is not
// a device address).
int noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return tgemm::cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return TGEMM_ERR_LAUNCH;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) return tgemm::cuda_fail(e, "cudaGetSymbolAddress(scratch)");
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return TGEMM_OK;
}

}  // namespace

extern "C" int tgemm_gemm_noalloc(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                                  int64_t ldb, void* C, int64_t ldc, int dtype, const tgemm_options* opts,
                                  void* stream) {
  tgemm_options o;
  std::memset(&o, 0, sizeof o);
  if (opts) o = *opts;
  if (o.stream_k == 0) o.stream_k = 2;  // this entry point is the stream-K variant
  if (o.repack == 0) o.repack = 1;      // and does not repack operands unless asked
  // validation first (no CUDA call on bad arguments)
  tgemm::Plan p;
  int st = tgemm::make_plan(M, N, K, A, lda, B, ldb, C, ldc, dtype, &o, 1, 1, INT64_MAX, p);
  if (st != TGEMM_OK || p.noop) return st;
  tgemm::DeviceInfo* dev = nullptr;
  st = tgemm::device_info(&dev);
  if (st != TGEMM_OK) return st;
  // scratch the call would use with no limit; beyond the static array: rejected
  st = tgemm::make_plan(M, N, K, A, lda, B, ldb, C, ldc, dtype, &o, dev->sm_count, tgemm::pair_capacity(dev),
                        INT64_MAX, p);
  if (st != TGEMM_OK) return st;
  if (static_cast<size_t>(p.workspace) > kNoAllocScratchBytes) return TGEMM_ERR_TOO_LARGE;
  void* scratch = nullptr;
  st = noalloc_scratch(&scratch);
  if (st != TGEMM_OK) return st;
  return tgemm::run(M, N, K, A, lda, B, ldb, C, ldc, dtype, &o, nullptr, scratch,
                    static_cast<int64_t>(kNoAllocScratchBytes),
                    static_cast<cudaStream_t>(stream));
}
