// common.cuh -- device helpers and launch descriptors shared by the libnf4 kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

namespace nf4k {

// The 16 NormalFloat levels, ascending, passed to every kernel by value and
// copied into shared memory once per block (never read from __constant__ in
// the hot loop: divergent nibble lookups serialize there -- "Decode V2 --
// resident executor", the ~50 GB/s constant-LUT wall in the status paragraph).
struct Codebook {
  float v[16];
};

// Streaming 16-byte load of data read exactly once: bypasses L1 allocation.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

__device__ __forceinline__ float ld_nc_f32(const float* p) {
  float r;
  asm("ld.global.nc.f32 %0, [%1];" : "=f"(r) : "l"(p));
  return r;
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// bf16 bit pair -> two fp32 (exact widening).
__device__ __forceinline__ float bf16lo_to_f32(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Named barrier over `count` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Epilogue kinds of the N=1 kernel.
enum Epi : int { EPI_PLAIN = 0, EPI_RESID = 1, EPI_SWIGLU = 2, EPI_ARGMAX = 3 };

// Arguments of one N=1 launch.
struct GemvArgs {
  const uint8_t* codes;   // [M][K/2]
  const float* scales;    // [M][K/64]
  const uint8_t* codes2;  // SwiGLU: up-projection codes
  const float* scales2;   // SwiGLU: up-projection scales
  const void* x;          // [K] fp32 or bf16
  const float* resid;     // [M] residual (may equal y)
  float* y;               // [M] fp32 out (plain / residual / logits)
  uint16_t* out_bf16;     // [M] SwiGLU out
  int64_t* index;         // argmax out
  unsigned long long* ws; // argmax workspace: [0] key, [1] block ticket
  int M;
  int K;
  int G;    // threads cooperating on one row (multiple of 32)
  int gpc;  // row groups per block
  Codebook cb;
};

// Kernel configuration for an N=1 launch (chosen on the host per shape).
struct GemvConfig {
  int nch;      // 16-byte chunks (32 weights) per thread per row
  int rb;       // rows per batch (registers in flight per thread: rb * nch * 16 B)
  bool big;     // register-capped instantiation for very long rows
  int G;        // threads per row group
  int gpc;      // groups per block
  int blocks;   // grid size
  int smem;     // dynamic shared memory bytes
};

// Host launchers (gemv.cu / quantize.cu).
cudaError_t launch_gemv(int epi, bool x_bf16, const GemvArgs& a, GemvConfig cfg, cudaStream_t s);
GemvConfig choose_gemv_config(int epi, int64_t M, int64_t K, int device);
cudaError_t launch_quantize(const float* W, int64_t M, int64_t K, uint8_t* codes, float* scales,
                            const Codebook& cb, cudaStream_t s, int device);

// Prefill chunk (chunk.cu).
cudaError_t launch_chunk(const uint8_t* codes, const float* scales, int M, int K, const uint16_t* X, int N,
                         float* Y, void* workspace, const Codebook& cb, cudaStream_t s, int device);
size_t chunk_workspace_bytes(int64_t M, int64_t K, int N);
std::string describe_chunk(int64_t M, int64_t K, int N, int device);

}  // namespace nf4k
