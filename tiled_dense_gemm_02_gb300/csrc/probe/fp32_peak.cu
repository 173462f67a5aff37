// FP32 FMA throughput probe: the denominator of the SIMT kernel's roofline,
// measured instead of derived from an assumed lane count ("寄存器Tiling",
// section 5.4: the self-check compares the issue rate reached with the
// pipe's peak, so the peak has to be known).
//
// Every thread runs 8 independent FMA chains (x = x * m + c), so neither the
// FMA latency nor a dependence limits the issue rate; the loop body is
// unrolled 16 times to keep branch and counter instructions out of the way.
// The paired variant issues fma.rn.f32x2 (two FMAs per instruction on a float2),
// the instruction the SIMT GEMM kernel uses.  Each thread writes the sum of
// its chains, so nothing is optimised away.  The probe reads no memory and
// writes blocks x threads floats: out must hold that many.
//
// Built as its own library (libtgemm_probe.so); the GEMM library does not
// contain or call it.
#include <cuda_runtime.h>

namespace {

constexpr int kChains = 8;
constexpr int kUnroll = 16;

template <bool kPaired>
__global__ void __launch_bounds__(256) ffma_peak_kernel(float* out, int iters, float m, float c) {
  const int tid = blockIdx.x * blockDim.x + threadIdx.x;
  float sum = 0.0f;
  if constexpr (kPaired) {
    float2 x[kChains];
    const float2 m2 = make_float2(m, m), c2 = make_float2(c, c);
#pragma unroll
    for (int j = 0; j < kChains; ++j) x[j] = make_float2(1e-3f * threadIdx.x + j, 2e-3f * threadIdx.x - j);
    for (int i = 0; i < iters; ++i)
#pragma unroll
      for (int r = 0; r < kUnroll; ++r)
#pragma unroll
        for (int j = 0; j < kChains; ++j) x[j] = __ffma2_rn(x[j], m2, c2);
#pragma unroll
    for (int j = 0; j < kChains; ++j) sum += x[j].x + x[j].y;
  } else {
    float x[kChains];
#pragma unroll
    for (int j = 0; j < kChains; ++j) x[j] = 1e-3f * threadIdx.x + j;
    for (int i = 0; i < iters; ++i)
#pragma unroll
      for (int r = 0; r < kUnroll; ++r)
#pragma unroll
        for (int j = 0; j < kChains; ++j) x[j] = __fmaf_rn(x[j], m, c);
#pragma unroll
    for (int j = 0; j < kChains; ++j) sum += x[j];
  }
  out[tid] = sum;
}

}  // namespace

// FLOPs of one launch: blocks x threads x iters x 16 x 8 x 2, twice that when
// paired.  Returns the cudaError_t of the launch (0 = success).
extern "C" __attribute__((visibility("default"))) int tgemm_probe_ffma(int paired, int blocks, int threads,
                                                                       int iters, float* out, void* stream) {
  if (blocks < 1 || threads < 32 || threads > 256 || threads % 32 != 0 || iters < 1 || !out)
    return static_cast<int>(cudaErrorInvalidValue);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (paired)
    ffma_peak_kernel<true><<<blocks, threads, 0, s>>>(out, iters, 0.99990f, 1e-4f);
  else
    ffma_peak_kernel<false><<<blocks, threads, 0, s>>>(out, iters, 0.99990f, 1e-4f);
  return static_cast<int>(cudaGetLastError());
}

// FMA instructions of one thread per loop iteration, for the caller's FLOP count.
extern "C" __attribute__((visibility("default"))) int tgemm_probe_ffma_per_iter(void) { return kChains * kUnroll; }
