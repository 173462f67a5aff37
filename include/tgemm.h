/*
 * tgemm -- tiled dense matrix multiply for NVIDIA GB300 (sm_103a).
 *
 * C ABI of the library (libtgemm.so).  Every entry point takes plain
 * integers and pointers; no CUDA or framework type appears in a signature.
 * A stream argument is a cudaStream_t passed as `void*` (NULL = the legacy
 * default stream).
 *
 * The operation is the dense product of the tiling pages:
 *     C[M,N] = A[M,K] . B[K,N],   C[i][j] = sum_{k<K} A[i][k] * B[k][j]
 * ("CUDA tile", section 2.1; "Tiling 策略与内存层次优化", section "Tiling 如何提升
 * 算术强度"), computed tile by tile with K split into stages
 * ("矩阵乘法中的平铺", the l-length K-splitting paragraph).  Splitting changes
 * only the order of the fp32 additions, never the set of terms.
 */
#ifndef TGEMM_H
#define TGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TGEMM_VERSION 10000 /* major * 10000 + minor * 100 + patch */

/* Entry points are the only symbols the library exports. */
#if defined(__GNUC__)
#define TGEMM_API __attribute__((visibility("default")))
#else
#define TGEMM_API
#endif

/* (input format, output format) pairs.  Every variant accumulates in fp32. */
enum tgemm_dtype {
  TGEMM_F32 = 0,         /* fp32 A, B -> fp32 C   (CUDA-core SIMT path)        */
  TGEMM_F16 = 1,         /* fp16 A, B -> fp16 C   (tensor-core path)           */
  TGEMM_BF16 = 2,        /* bf16 A, B -> bf16 C   (tensor-core path)           */
  TGEMM_BF16_F32OUT = 3, /* bf16 A, B -> fp32 C   (tensor-core path)           */
  TGEMM_F16_F32OUT = 4   /* fp16 A, B -> fp32 C   (tensor-core path)           */
};

/* Status codes.  0 is success; every other value is an error and nothing was
 * launched (except TGEMM_ERR_DEVICE_TIMEOUT, which reports a past launch). */
enum tgemm_status {
  TGEMM_OK = 0,
  TGEMM_ERR_INVALID_VALUE = 1,     /* negative size, leading dimension too small,
                                      null pointer with a non-empty extent,
                                      bad option value */
  TGEMM_ERR_UNSUPPORTED_DTYPE = 2, /* dtype not in enum tgemm_dtype */
  TGEMM_ERR_MISALIGNED = 3,        /* a pointer is not aligned to its element size */
  TGEMM_ERR_ALIAS = 4,             /* C's byte range overlaps A's or B's */
  TGEMM_ERR_UNSUPPORTED_DEVICE = 5,/* current device is not compute capability 10.3 */
  TGEMM_ERR_LAUNCH = 6,            /* a CUDA call failed while launching; see
                                      tgemm_status_string(TGEMM_ERR_LAUNCH) */
  TGEMM_ERR_DEVICE_TIMEOUT = 7,    /* a kernel gave up a bounded wait (reported
                                      by tgemm_device_status) */
  TGEMM_ERR_TOO_LARGE = 8          /* a size exceeds what the kernels index
                                      (M, N, K >= 2^31, or a bulk-copy bound) */
};

/*
 * C = A . B, row-major, asynchronous on `stream`.
 *
 *   A: M x K, element (i, k) at A[i*lda + k], lda >= max(1, K)
 *   B: K x N, element (k, j) at B[k*ldb + j], ldb >= max(1, N)
 *   C: M x N, element (i, j) at C[i*ldc + j], ldc >= max(1, N)
 * Leading dimensions are in elements of the operand's own format.  A, B and
 * C are device pointers owned by the caller; each must be aligned to its
 * element size.  C is overwritten (no alpha/beta); elements of C outside the
 * M x N window (the ldc - N padding of each row) are never written.
 *
 * M == 0 or N == 0: nothing is done.  K == 0: C is set to +0.
 * Any alignment and any leading dimension are accepted; 16-byte aligned rows
 * take the bulk-tensor (TMA) loads and stores, others take per-thread copies.
 *
 * The call validates its arguments on the host, picks a kernel and a tile
 * shape for the current device, and enqueues one kernel on `stream` (two for
 * an fp32 product whose last round of tiles is split into K halves: a fill
 * that zeroes the rows of C those halves add into, then the product; see
 * tgemm_options.simt_split); it returns before the product is computed.  It
 * allocates no device memory.
 * It keeps small, mutex-guarded host caches of device attributes and of
 * encoded tensor maps (see tgemm_host_counters).  It is safe to call from
 * several host threads.
 *
 * Errors: see enum tgemm_status.  Validation errors are returned before any
 * CUDA call.  A launch failure returns TGEMM_ERR_LAUNCH with the CUDA error
 * text available from tgemm_status_string.
 */
TGEMM_API int tgemm_gemm(int64_t M, int64_t N, int64_t K,
               const void* A, int64_t lda,
               const void* B, int64_t ldb,
               void* C, int64_t ldc,
               int dtype, void* stream);

/* Kernel selection for tgemm_gemm_ex.  AUTO picks as tgemm_gemm does. */
enum tgemm_kernel {
  TGEMM_KERNEL_AUTO = 0,
  TGEMM_KERNEL_TC_TMA = 1,     /* tensor cores; A and B by bulk-tensor copies */
  TGEMM_KERNEL_TC_COPY = 2,    /* tensor cores; A and/or B by per-thread async
                                  copies (any alignment); with cta_group = 2,
                                  A by bulk-tensor copies and B per thread */
  TGEMM_KERNEL_SIMT = 3        /* fp32 CUDA cores (TGEMM_F32 only) */
};

/* Options of tgemm_gemm_ex.  Zero-initialise and set what you need; a zero
 * field means "the default". */
typedef struct tgemm_options {
  int kernel;           /* enum tgemm_kernel */
  int tile_n;           /* tensor-core tile width: 0 (auto), 64, 128, 192,
                           224 or 256 */
  int group_m;          /* rasterisation group height in tiles (0 = auto) */
  int max_ctas;         /* cap on persistent CTAs (0 = one per SM) */
  int store_mode;       /* 0 auto, 1 bulk-tensor store, 2 per-thread stores */
  int wait_timeout_us;  /* bound of every in-kernel wait (0 = 2 s) */
  int inject_fault;     /* test hook: 1 = the producer never signals its first
                           stage, so the consumers' bounded waits run out and
                           the kernel exits with TGEMM_ERR_DEVICE_TIMEOUT
                           pending; no copy is ever issued */
  int cta_group;        /* tensor-core tiles per CTA (0 auto): 1 = 128 x N
                           tiles on one SM, 2 = 256 x N tiles on a pair of
                           SMs (a 2-CTA cluster): with bulk-tensor operands,
                           tile_n 128, 192, 224 or 256; with A by bulk-tensor
                           copies and B by per-thread copies (B's rows off the
                           16-byte grid, or kernel = TC_COPY), tile_n 128 or
                           256, 64-deep stages and per-thread stores of C */
  int tile_k;           /* K depth of one shared-memory stage (0 auto): 64, or
                           128 (two 64-deep sub-blocks per stage, one MMA
                           completion signal per stage; CTA-pair kernel only) */
  int stream_k;         /* split of the last round of tiles along K over all
                           CTA pairs (needs a workspace, tgemm_gemm_ws):
                           0 auto (currently off: on the measured shapes the
                           fix-up costs more than the idle tail), 1 off,
                           2 on whenever the tile count leaves a remainder */
  int reserved0;        /* must be 0 (TGEMM_ERR_INVALID_VALUE otherwise) */
  int swap_ab;          /* CTA pairs with the MMA's operands exchanged: 0 auto,
                           1 off, 2 on.  Each pair computes a tile_m x 256
                           tile of C as a tile of C^T = B^T A^T, so the tile
                           height can be any of 128, 192, 224, 256 with no
                           partly used shared-memory atoms.  Needs bulk-tensor
                           operands and no stream-K split */
  int tile_m;           /* tile height of swap_ab = 2 (0 auto): 128, 192, 224
                           or 256; other kernels take 0 */
  int simt_split;       /* fp32 SIMT kernel (TGEMM_F32 only; other dtypes
                           take 0).  When the last round of 128 x 128 tiles
                           fills at most half of the resident CTA slots (two
                           per SM), each of its tiles is computed as two K
                           halves by two CTAs, whose results are added into C
                           after the call zeroes those rows of C.  Two
                           additions onto zero commute, so the result does
                           not depend on which half lands first.  0 auto (on
                           when K >= 256), 1 off, 2 on whenever the round
                           fits and K spans two 16-deep stages.  A call with
                           an epilogue computes every tile whole */
  int repack;           /* tensor-core paths with a workspace (tgemm_gemm_ws,
                           tgemm_gemm_epilogue): an operand whose rows are not
                           16-byte aligned (base or pitch) is first copied into
                           the workspace with its pitch rounded up to a
                           multiple of 8 elements, and the bulk-tensor kernels
                           read that copy (one extra launch per copied
                           operand).  0 auto: copy B when M >= 512 and A when
                           N >= 512 (the product reads them several times),
                           whenever the workspace holds the copies; 1 never;
                           2 any such operand.  tgemm_workspace_size counts
                           the copies' bytes */
  int reserved[1];      /* must be 0 */
} tgemm_options;

/* tgemm_gemm with explicit options (opts may be NULL).  A forced kernel that
 * cannot serve the arguments (e.g. TC_TMA on rows that are not 16-byte
 * aligned) returns TGEMM_ERR_INVALID_VALUE. */
TGEMM_API int tgemm_gemm_ex(int64_t M, int64_t N, int64_t K,
                  const void* A, int64_t lda,
                  const void* B, int64_t ldb,
                  void* C, int64_t ldc,
                  int dtype, const tgemm_options* opts, void* stream);

/* The dispatch decision tgemm_gemm_ex would take, without launching and
 * without touching the GPU.  `sm_count` is the number of SMs to plan for.
 * Returns the same validation status as tgemm_gemm_ex. */
typedef struct tgemm_plan_info {
  int kernel;        /* enum tgemm_kernel actually chosen (never AUTO) */
  int tile_m, tile_n, tile_k;
  int stages;        /* shared-memory ring depth */
  int tiles_m, tiles_n;
  int ctas;          /* CTAs launched (persistent: min(tiles, SMs)) */
  int group_m;
  int a_copy_bytes;  /* granule of A's per-thread copies (0 = bulk-tensor) */
  int b_copy_bytes;  /* granule of B's per-thread copies (0 = bulk-tensor) */
  int store_bytes;   /* granule of C's per-thread stores (0 = bulk-tensor) */
  int smem_bytes;    /* dynamic shared memory per CTA */
  int cta_group;     /* 1: one SM per tile; 2: a CTA pair per 256-row tile
                        (tile_m is then 256 and ctas counts CTAs, two per pair) */
  int dp_tiles;      /* tiles computed whole (all of them without stream-K;
                        SIMT kernel: the rest are split in two K halves, and
                        ctas = dp_tiles + 2 x the split tiles) */
  int sk_iters;      /* k-stages of the remaining tiles split over the pairs */
  int workspace_bytes; /* workspace the call uses (0 without stream-K or
                          repacked operands) */
  int cluster_ctas;  /* CTAs per cluster: 1 (one-SM tiles) or 2 (a pair) */
  int swap_ab;       /* 1: pairs with the MMA's operands exchanged (tile_m x
                        256 tiles of C computed as tiles of C^T) */
  int tuned;         /* 1: options from the library's table of measured
                        shapes (the call left every tuned option at 0 and its
                        shape and dtype match an entry exactly) */
  int packed;        /* operands copied into the workspace before the
                        product (tgemm_options.repack): 1 = A, 2 = B, 3 = both */
} tgemm_plan_info;

TGEMM_API int tgemm_plan(int64_t M, int64_t N, int64_t K,
               const void* A, int64_t lda,
               const void* B, int64_t ldb,
               const void* C, int64_t ldc,
               int dtype, const tgemm_options* opts,
               size_t workspace_bytes, int sm_count,
               tgemm_plan_info* out);

/*
 * Stream-K workspace.  When the number of output tiles leaves the last round
 * of the persistent grid partly empty, tgemm_gemm_ws splits the k-stages of
 * the remaining tiles evenly over all CTA pairs.  The pairs holding the first
 * k-stages of a tile write fp32 partial sums to the workspace; the pair
 * holding its last k-stage adds them (in a fixed order, so results do not
 * depend on timing) and stores C.
 *
 * tgemm_workspace_size: bytes of workspace tgemm_gemm_ws would use for these
 * arguments on the current device, for the stream-K split and for operands it
 * repacks (tgemm_options.repack); 0 when it would use none.  Same validation
 * and status codes as tgemm_gemm_ex.
 *
 * Workspace layout: the first 4 KiB hold stream-K flags only, the partial sums
 * follow, then the repacked operands.
 *
 * tgemm_gemm_ws: tgemm_gemm_ex with a workspace.  `workspace` is device memory
 * owned by the caller, 256-byte aligned, zero-initialised before its first use
 * (later calls need no clearing, whatever their shapes: the flags always take
 * the first 4 KiB and the partial sums follow); `workspace_bytes` smaller than
 * tgemm_workspace_size (including 0 with a NULL workspace) makes the call run
 * without stream-K.  Two calls that may run at the same time on the GPU must
 * not share a workspace.  Its contents after a call are unspecified.
 * Finishing pairs wait (bounded, see wait_timeout_us) for the partial sums of
 * the others, so all CTA pairs of the call must be able to run at once: the
 * grid never exceeds the resident capacity of the device; a device shared
 * with kernels that keep SMs busy indefinitely can make the wait run out
 * (TGEMM_ERR_DEVICE_TIMEOUT, C unspecified).
 */
TGEMM_API int tgemm_workspace_size(int64_t M, int64_t N, int64_t K,
               const void* A, int64_t lda,
               const void* B, int64_t ldb,
               const void* C, int64_t ldc,
               int dtype, const tgemm_options* opts, size_t* bytes);

TGEMM_API int tgemm_gemm_ws(int64_t M, int64_t N, int64_t K,
               const void* A, int64_t lda,
               const void* B, int64_t ldb,
               void* C, int64_t ldc,
               int dtype, const tgemm_options* opts,
               void* workspace, size_t workspace_bytes, void* stream);

/*
 * Allocation-free variant (the tiling pages have no counterpart; this serves
 * callers of the library).
 *
 * Some callers cannot allocate device memory at the time they multiply: an
 * application or plug-in host that hands out all device memory from its own
 * pool, or a service whose memory budget is fixed after start-up, can neither
 * give this library a workspace nor let it call cudaMalloc.  For them,
 * tgemm_gemm_noalloc behaves as tgemm_gemm_ws with the stream-K split on
 * (opts->stream_k 0 is read as 2; 1 turns it off; opts->repack 0 is read as
 * 1, so operands are not copied unless asked), but takes its partial sums
 * and flags from a scratch array of TGEMM_NOALLOC_SCRATCH_BYTES built into the
 * library, in device memory that every GPU loading the library holds until
 * the process exits.  It allocates nothing and calls no allocating routine.
 *
 *  - The first call on a device looks up the device address of that array
 *    (with the device current); make that first call before any stream
 *    capture.
 *  - A call whose split would need more scratch than the array holds returns
 *    TGEMM_ERR_TOO_LARGE and launches nothing; tgemm_workspace_size (with
 *    stream_k = 2) gives the amount a call needs.
 *  - Every call shares the one array.  Calls that may run at the same time on
 *    the GPU (different streams, or several host threads) race on it and can
 *    produce wrong results; order them on one stream or use tgemm_gemm_ws.
 *  - Nothing in the array needs clearing between calls: the array starts
 *    zeroed, its first 4 KiB hold only flags, and a flag marks a partial sum
 *    with a value that differs from call to call, so whatever an earlier call
 *    left behind is never taken for this call's data.
 *  - The device address is looked up once per device and kept for the life of
 *    the process: after cudaDeviceReset (or any tear-down of the device's
 *    primary context) this entry point must not be called again.
 *  Other arguments, status codes and semantics: as tgemm_gemm_ex.
 */
#define TGEMM_NOALLOC_SCRATCH_BYTES ((size_t)20 * 1024 * 1024 + 4096)

TGEMM_API int tgemm_gemm_noalloc(int64_t M, int64_t N, int64_t K,
               const void* A, int64_t lda,
               const void* B, int64_t ldb,
               void* C, int64_t ldc,
               int dtype, const tgemm_options* opts, void* stream);

/*
 * Fused epilogue ("Tiling 策略与内存层次优化", section "Tiling 贯穿编译器栈",
 * Fusion stage: element-wise post-processing such as a bias add and ReLU is
 * applied to a GEMM tile's output in place, before it is written back).
 *
 *   C[i][j] = act(alpha * sum_k A[i][k] B[k][j] + beta * C_prior[i][j] + bias[j])
 *
 * computed in fp32 on the fp32 accumulator and rounded once (RNE) to the output
 * format.  act is the identity or ReLU (x < 0 ? 0 : x, which keeps a NaN).
 *  - alpha: scale of the product (1 for the plain product).
 *  - beta: scale of C's prior contents, read in C's own format.  With beta == 0
 *    C is not read at all, so it may hold anything, NaN included.
 *  - bias: NULL, or a device pointer to N fp32 values (4-byte aligned, owned by
 *    the caller, not written), one per column of C.
 *  - activation: TGEMM_ACT_NONE or TGEMM_ACT_RELU.
 * With K = 0 the product is the empty sum 0 and C = act(beta C_prior + bias).
 * Every kernel path applies it; `workspace`/`workspace_bytes` (NULL/0 allowed)
 * serve the stream-K split as in tgemm_gemm_ws.
 */
enum tgemm_activation { TGEMM_ACT_NONE = 0, TGEMM_ACT_RELU = 1 };

typedef struct tgemm_epilogue {
  float alpha;
  float beta;
  const float* bias;
  int activation;   /* enum tgemm_activation */
  int reserved[3];  /* zero */
} tgemm_epilogue;

/* tgemm_gemm_ws with a fused epilogue (epi may be NULL: the plain product).
 * Returns TGEMM_ERR_INVALID_VALUE for an unknown activation, nonzero reserved
 * fields or a misaligned bias pointer, and TGEMM_ERR_ALIAS if the bias lies
 * inside C.  Asynchronous on `stream`, like tgemm_gemm_ex. */
TGEMM_API int tgemm_gemm_epilogue(int64_t M, int64_t N, int64_t K,
               const void* A, int64_t lda,
               const void* B, int64_t ldb,
               void* C, int64_t ldc,
               int dtype, const tgemm_epilogue* epi,
               const tgemm_options* opts,
               void* workspace, size_t workspace_bytes, void* stream);

/*
 * Strided batch of independent products ("矩阵乘法中的平铺", closing advice:
 * where tensor cores are available, use a batched interface).
 *
 *   for b < batch:  C_b = act(alpha A_b . B_b + beta C_b + bias)
 *   A_b = A + b * stride_a, B_b = B + b * stride_b, C_b = C + b * stride_c
 *
 * Strides are in elements of each operand's format.  stride_a or stride_b may
 * be 0 (every product uses the same matrix); the C windows must not overlap
 * (stride_c >= (M - 1) * ldc + N, else TGEMM_ERR_ALIAS), and no C window may
 * overlap any A or B matrix.  epi (may be NULL) applies to every product, with
 * one bias vector for all.  When every A_b and B_b starts on a 16-byte boundary
 * and the operands suit bulk-tensor copies, the whole batch runs in one launch
 * of the swapped-operand pair kernel, whose tile list spans all matrices.
 * Otherwise each product is launched on its own.  batch == 0: nothing is done.
 * Other arguments and errors: as tgemm_gemm_ex.
 */
TGEMM_API int tgemm_gemm_batched(int64_t batch, int64_t M, int64_t N, int64_t K,
               const void* A, int64_t lda, int64_t stride_a,
               const void* B, int64_t ldb, int64_t stride_b,
               void* C, int64_t ldc, int64_t stride_c,
               int dtype, const tgemm_epilogue* epi,
               const tgemm_options* opts, void* stream);

/* The plan of tgemm_gemm_batched without touching the GPU (pair counts
 * modelled from sm_count as tgemm_plan does).  *launches: kernel launches the
 * call makes without an epilogue (1 for an in-kernel batch, batch for one
 * launch per product, twice that for fp32 products split into K halves, each
 * preceded by its zero fill; 0 when nothing is done).  out describes one
 * product's launch. */
TGEMM_API int tgemm_plan_batched(int64_t batch, int64_t M, int64_t N, int64_t K,
               const void* A, int64_t lda, int64_t stride_a,
               const void* B, int64_t ldb, int64_t stride_b,
               const void* C, int64_t ldc, int64_t stride_c,
               int dtype, const tgemm_options* opts, int sm_count,
               tgemm_plan_info* out, int* launches);

/*
 * Tiled transpose ("CUDA tile", section 三: a tile read along the rows of the
 * input and written along the rows of the output, so both sides coalesce):
 *
 *   dst[j * ld_dst + i] = src[i * ld_src + j]   for i < rows, j < cols
 *
 * src is rows x cols (ld_src >= max(1, cols)), dst is cols x rows
 * (ld_dst >= max(1, rows)); elements are moved as raw elem_bytes-byte units
 * (2 or 4: fp16/bf16 or fp32), so the result is bit-exact.  Elements of dst
 * past `rows` in each row are not written.  src and dst must not overlap
 * (TGEMM_ERR_ALIAS; no in-place transpose).  rows or cols == 0: nothing is
 * done.  Asynchronous on `stream`; allocates nothing.
 */
TGEMM_API int tgemm_transpose(int64_t rows, int64_t cols,
               const void* src, int64_t ld_src,
               void* dst, int64_t ld_dst,
               int elem_bytes, void* stream);

/*
 * The product with A, B and C in host memory (the pages have no counterpart:
 * this serves callers whose data lives on the host).  The library copies B
 * and row panels of A into caller-owned device buffers, multiplies each panel
 * as soon as its rows have arrived, and copies each panel of C back while the
 * next one is computed, so host-to-device copies, kernels and
 * device-to-host copies of different panels overlap.
 *
 *   C_host[i * ldc + j] = sum_k A_host[i * lda + k] * B_host[k * ldb + j]
 *
 * A_host, B_host, C_host: host memory, row-major with the given leading
 *   dimensions (elements, as in tgemm_gemm).  Page-locked memory
 *   (cudaHostAlloc / cudaHostRegister) lets the copies run asynchronously and
 *   overlap; pageable memory gives the same result, but each copy then blocks
 *   the calling thread.  Elements of C_host past N in each row are not written.
 * dA, dB, dC: device buffers owned by the caller, at least M*K, K*N and M*N
 *   elements, used densely (row pitches K, N and N).  Afterwards dC holds the
 *   product; dA and dB hold the copied operands.  They must not overlap.
 * panels: row panels of A and C (0 = chosen by the library: one when C is
 *   below 6 MB, else graduated whole numbers of 128-row tiles, small first so
 *   that C's copy back starts early; n > 0 = n even panels; 1 = no overlap).
 *   With fp32 output, several panels and K >= 256, the first panel's product
 *   runs in two K halves, the first while B's second half is being copied
 *   (the partial sum is rounded once to fp32 before the second half is added).
 * stream: everything the call does follows the work already enqueued on
 *   `stream`, and later work on `stream` follows all of it, including the
 *   copy of C to the host.  The call returns once the work is enqueued:
 *   synchronise `stream` before reading C_host.  The copies run on two
 *   streams per device that the library creates on first use and keeps;
 *   ordering with `stream` is by events, taken from a per-device pool that
 *   the library keeps (created as the pool grows, never destroyed).
 * Errors: as tgemm_gemm for the product (M, N, K, dtype, leading dimensions);
 *   TGEMM_ERR_INVALID_VALUE for a null buffer with a nonzero extent or
 *   panels < 0, TGEMM_ERR_MISALIGNED for a pointer not aligned to its element
 *   size, TGEMM_ERR_ALIAS for overlapping device buffers.  Argument errors are
 *   returned before any CUDA call.
 */
TGEMM_API int tgemm_gemm_host(int64_t M, int64_t N, int64_t K,
               const void* A_host, int64_t lda,
               const void* B_host, int64_t ldb,
               void* C_host, int64_t ldc,
               int dtype, void* dA, void* dB, void* dC,
               int panels, void* stream);

/* Waits for `stream`, then returns and clears the device-side status word
 * that bounded in-kernel waits set when they give up (TGEMM_OK or
 * TGEMM_ERR_DEVICE_TIMEOUT).  A CUDA error while synchronising returns
 * TGEMM_ERR_LAUNCH. */
TGEMM_API int tgemm_device_status(void* stream);

/* Static text for a status code; for TGEMM_ERR_LAUNCH the text of the last
 * CUDA error seen by the calling thread. */
TGEMM_API const char* tgemm_status_string(int status);

/* TGEMM_VERSION of the loaded library. */
TGEMM_API int tgemm_version(void);

/*
 * Host-side counters of the library, process-wide and cumulative ("GPU Kernel
 * 的 Tile、Grid、Wave 与 Launch Overhead", section Launch Overhead: at small
 * sizes the fixed cost of a launch dominates, so the host work per call is
 * kept small and observable).
 *
 * Every bulk-tensor (TMA) descriptor a call needs is looked up in a cache of
 * encoded tensor maps keyed on all of its encode arguments (device, base
 * address, element type, dimensions, strides, box, swizzle); only a miss calls
 * the driver's encoder.  Repeated calls on the same buffers and shapes then
 * encode nothing.
 *
 *   tc_launches: tensor-core kernel launches enqueued by product calls
 *   map_hits:    tensor maps taken from the cache
 *   map_encodes: tensor maps encoded (cache misses)
 *   ns_prepare:  host nanoseconds those calls spent before their launch
 *                (validation, planning, tensor maps)
 *   ns_launch:   host nanoseconds spent inside their CUDA launch calls
 * Returns TGEMM_ERR_INVALID_VALUE for a NULL `out`; needs no GPU.
 */
typedef struct tgemm_counters {
  uint64_t tc_launches;
  uint64_t map_hits;
  uint64_t map_encodes;
  uint64_t ns_prepare;
  uint64_t ns_launch;
} tgemm_counters;

TGEMM_API int tgemm_host_counters(tgemm_counters* out);

#ifdef __cplusplus
}
#endif

#endif /* TGEMM_H */
