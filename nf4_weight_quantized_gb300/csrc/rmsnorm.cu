// rmsnorm.cu -- RMSNorm as its own small producer kernel ahead of a projection.
//
// y[r][k] = x[r][k] * rsqrt(mean_k(x[r][k]^2) + eps) * w[k]
// Source: "Decode V2 -- resident executor", section 3 (x * rsqrt(mean(x^2) +
// eps) * w, Qwen-style, no bias; RMS weights are bf16 [hidden]), section 6
// (RMS writes in place) and the status table with its notes (fusing RMS into
// the following GEMV was measured as a loss: every block of the projection
// repeats the same reduction, ~152k times on lm_head, so RMS stays a one-block
// kernel); "golang.design/x/accel/tensor", func RMSNorm (each row by its own
// root mean square; the mean square and the reciprocal square root in f32).
//
// One block per row.  Each thread sums the squares of its strided elements
// with fused multiply-adds, the block adds the per-thread sums in a fixed
// order (warp shuffles, then the warps' totals in warp order), and the row is
// scaled by 1 / sqrt(ms + eps) (IEEE square root and division) and by the
// bf16 gain widened exactly.  The result depends only on the row's data.
// Launched with programmatic dependent launch: the kernel lets the next one
// (typically the projection) launch at once, so the projection's blocks can
// prefetch their weights on the other SMs while this block normalizes; x is
// read only after the previous kernel on the stream has completed.  For rows
// of up to 8 x 1024 elements each thread keeps its elements and their gains
// in registers: the gains are loaded before the dependency wait (they never
// depend on the previous kernel) and x is read from memory once; longer rows
// take a loop that reads x twice.  Both forms sum in the same order.
#include <cuda_bf16.h>

#include "common.cuh"

namespace nf4k {

namespace {

constexpr int kMaxThreads = 1024;
constexpr int kRegElems = 8;  // elements per thread held in registers

// Block-wide sum of one value per thread: shuffles within each warp, then the
// warps' totals in warp order (every thread gets the same total).
__device__ __forceinline__ float block_sum(float v, float* warp_sums) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  if (lane == 0) warp_sums[warp] = v;
  __syncthreads();
  float total = 0.f;
  const int nw = (int)(blockDim.x >> 5);
  for (int i = 0; i < nw; ++i) total += warp_sums[i];
  return total;
}

// Rows of at most kRegElems * blockDim.x elements: element k = tid + i *
// blockDim.x of the row is held in registers (the same elements, in the same
// order, as the loop form below).
__global__ void __launch_bounds__(kMaxThreads) rmsnorm_reg_kernel(const float* __restrict__ x,
                                                                  const uint16_t* __restrict__ w, int K, float eps,
                                                                  void* y, int y_bf16) {
  __shared__ float warp_sums[32];
  pdl_launch_dependents();
  const int tid = threadIdx.x, bd = (int)blockDim.x;
  float g[kRegElems];
#pragma unroll
  for (int i = 0; i < kRegElems; ++i) {
    const int k = tid + i * bd;
    g[i] = k < K ? __uint_as_float((uint32_t)w[k] << 16) : 0.f;
  }
  pdl_wait();  // x is the previous kernel's output
  const int64_t base = (int64_t)blockIdx.x * K;
  const float* xr = x + base;
  float v[kRegElems];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < kRegElems; ++i) {
    const int k = tid + i * bd;
    v[i] = k < K ? xr[k] : 0.f;
  }
#pragma unroll
  for (int i = 0; i < kRegElems; ++i)
    if (tid + i * bd < K) ss = fmaf(v[i], v[i], ss);
  const float total = block_sum(ss, warp_sums);
  const float inv = 1.0f / sqrtf(total / (float)K + eps);
  // in place (y == x, fp32) is safe: every read of x finished before the barrier
  if (y_bf16) {
    uint16_t* yr = static_cast<uint16_t*>(y) + base;
#pragma unroll
    for (int i = 0; i < kRegElems; ++i) {
      const int k = tid + i * bd;
      if (k < K) yr[k] = __bfloat16_as_ushort(__float2bfloat16_rn((v[i] * inv) * g[i]));
    }
  } else {
    float* yr = static_cast<float*>(y) + base;
#pragma unroll
    for (int i = 0; i < kRegElems; ++i) {
      const int k = tid + i * bd;
      if (k < K) yr[k] = (v[i] * inv) * g[i];
    }
  }
}

__global__ void __launch_bounds__(kMaxThreads) rmsnorm_kernel(const float* __restrict__ x,
                                                              const uint16_t* __restrict__ w, int K, float eps,
                                                              void* y, int y_bf16) {
  __shared__ float warp_sums[32];
  pdl_launch_dependents();
  pdl_wait();  // x is the previous kernel's output
  const int tid = threadIdx.x;
  const int64_t base = (int64_t)blockIdx.x * K;
  const float* xr = x + base;
  float ss = 0.f;
  for (int k = tid; k < K; k += blockDim.x) {
    const float v = xr[k];
    ss = fmaf(v, v, ss);
  }
  const float total = block_sum(ss, warp_sums);  // every thread, same order
  const float inv = 1.0f / sqrtf(total / (float)K + eps);
  // in place (y == x, fp32) is safe: every read of the first pass finished
  // before the barrier, and each element is read and written by one thread
  if (y_bf16) {
    uint16_t* yr = static_cast<uint16_t*>(y) + base;
    for (int k = tid; k < K; k += blockDim.x) {
      const float g = __uint_as_float((uint32_t)w[k] << 16);
      yr[k] = __bfloat16_as_ushort(__float2bfloat16_rn((xr[k] * inv) * g));
    }
  } else {
    float* yr = static_cast<float*>(y) + base;
    for (int k = tid; k < K; k += blockDim.x) {
      const float g = __uint_as_float((uint32_t)w[k] << 16);
      yr[k] = (xr[k] * inv) * g;
    }
  }
}

}  // namespace

// Threads per block: about eight elements per thread, whole warps, 64..1024.
int rmsnorm_threads(int64_t K) {
  int64_t t = (K + 7) / 8;
  t = (t + 31) / 32 * 32;
  return (int)(t < 64 ? 64 : (t > kMaxThreads ? kMaxThreads : t));
}

cudaError_t launch_rmsnorm(const float* x, const uint16_t* w, int64_t rows, int64_t K, float eps, void* y,
                           bool y_bf16, cudaStream_t s) {
  const int threads = rmsnorm_threads(K);
  const bool reg = K <= (int64_t)kRegElems * threads;
  const void* fn = reg ? reinterpret_cast<const void*>(&rmsnorm_reg_kernel) : reinterpret_cast<const void*>(&rmsnorm_kernel);
  return checked_launch(fn, threads, 0, [&] {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)rows);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    if (reg)
      cudaLaunchKernelEx(&cfg, rmsnorm_reg_kernel, x, w, (int)K, eps, y, y_bf16 ? 1 : 0);
    else
      cudaLaunchKernelEx(&cfg, rmsnorm_kernel, x, w, (int)K, eps, y, y_bf16 ? 1 : 0);
  });
}

}  // namespace nf4k
