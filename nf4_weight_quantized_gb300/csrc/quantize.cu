// quantize.cu -- NF4 encoder on the device (not on the decode hot path).
//
// Per 64-weight block: scale = max |w| (exact in fp32); an all-zero block gets
// scale 0 and the zero level (code 7) everywhere; otherwise each weight takes
// the level nearest to w / scale, ties to the lower level.  The comparison is
// made exactly: with mid_i = (cb[i] + cb[i+1]) / 2 the tie point between
// levels i and i+1, w / s > mid_i  <=>  w > mid_i * s (s > 0), and in float64
// both mid_i (at most 26 significant bits) and mid_i * s (at most 50) are
// exact, so the code is the count of mid_i * s strictly below w.
// Source: "Decode V2 -- resident executor", section 2 (NF4 linears in
// 64-weight groups; encode_nf4 is the one codec).
#include "common.cuh"

namespace nf4k {

namespace {

// One warp per block of 64 weights: lane l handles w[2l] and w[2l+1] and
// writes code byte l (low nibble = even k).
__global__ void quantize_kernel(const float* __restrict__ W, int64_t nblocks, uint8_t* __restrict__ codes,
                                float* __restrict__ scales, const __grid_constant__ Codebook cb) {
  __shared__ double mids[15];
  if (threadIdx.x < 15) mids[threadIdx.x] = ((double)cb.v[threadIdx.x] + (double)cb.v[threadIdx.x + 1]) * 0.5;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t blk = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); blk < nblocks; blk += warps) {
    const float2 w = reinterpret_cast<const float2*>(W + blk * 64)[lane];
    float s = fmaxf(fabsf(w.x), fabsf(w.y));
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) s = fmaxf(s, __shfl_xor_sync(0xffffffffu, s, off));
    int lo = 7, hi = 7;
    if (s > 0.0f) {
      lo = 0;
      hi = 0;
      const double sd = (double)s;
#pragma unroll
      for (int i = 0; i < 15; ++i) {
        const double t = mids[i] * sd;
        lo += ((double)w.x > t) ? 1 : 0;
        hi += ((double)w.y > t) ? 1 : 0;
      }
    }
    codes[blk * 32 + lane] = (uint8_t)(lo | (hi << 4));
    if (lane == 0) scales[blk] = s;
  }
}

}  // namespace

cudaError_t launch_quantize(const float* W, int64_t M, int64_t K, uint8_t* codes, float* scales,
                            const Codebook& cb, cudaStream_t s, int device) {
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  const int64_t nblocks = M * (K / 64);
  const int threads = 256;
  int64_t want = (nblocks + 7) / 8;
  int64_t cap = (int64_t)(sms > 0 ? sms : 1) * 8;
  const int grid = (int)(want < cap ? want : cap);
  quantize_kernel<<<grid, threads, 0, s>>>(W, nblocks, codes, scales, cb);
  return cudaGetLastError();
}

}  // namespace nf4k
