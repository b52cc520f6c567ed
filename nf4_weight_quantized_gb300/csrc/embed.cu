// embed.cu -- NF4 embedding rows gathered and dequantized (nf4_dequant_rows).
//
// Source: "Decode V2 -- resident executor", section 10: the embedding table
// stays as NF4 rows and the rows a step needs are dequantized into the arena;
// no dense [vocab, hidden] table exists.  out[i][k] = level(code) * scale, one
// fp32 product (the same rounding as every other consumer of W_hat), stored as
// fp32 or rounded once to bf16.
//
// The work is a gather bound by memory traffic (0.5625 B read and 2 or 4 B
// written per weight): one thread per 32-weight chunk loads 16 code bytes and
// its block scale and writes 128 (fp32) or 64 (bf16) contiguous bytes, so a
// warp stores whole 128-byte lines.  The 16 levels sit in shared memory (one
// bank each).  An id outside the table writes a zero row and sets the
// library's device error word (kErrBadIndex), read by nf4_check_device_errors.
#include "common.cuh"

namespace nf4k {

namespace {

struct EmbedArgs {
  const uint8_t* codes;  // [V][K/2]
  const float* scales;   // [V][K/64]
  const int64_t* ids;    // [n]
  void* out;             // [n][K] fp32 or bf16
  int64_t V, K, n;
  int out_bf16;
  Codebook cb;
};

__global__ void __launch_bounds__(256) embed_rows_kernel(const __grid_constant__ EmbedArgs a) {
  __shared__ float lv[16];
  if (threadIdx.x < 16) lv[threadIdx.x] = a.cb.v[threadIdx.x];
  __syncthreads();
  const int64_t H = a.K >> 5;  // 32-weight chunks per row
  const int64_t total = a.n * H;
  for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < total; c += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = c / H, h = c - i * H;
    const int64_t id = __ldg(a.ids + i);
    const bool ok = id >= 0 && id < a.V;
    float w[32];
    if (ok) {
      const uint4 cw = ld_nc_v4(a.codes + id * (a.K >> 1) + h * 16);
      const float s = ld_nc_f32(a.scales + id * (a.K >> 6) + (h >> 1));
      const uint32_t q[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int b = 0; b < 8; ++b) w[8 * j + b] = lv[(q[j] >> (4 * b)) & 15u] * s;  // nibble b: k = 8j + b
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) w[e] = 0.f;
      if (h == 0) atomicOr(&g_nf4_device_error, kErrBadIndex);
    }
    if (a.out_bf16) {
      uint4* o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + i * a.K + h * 32);
#pragma unroll
      for (int v = 0; v < 4; ++v)
        o[v] = make_uint4(pack_bf16x2(w[8 * v + 0], w[8 * v + 1]), pack_bf16x2(w[8 * v + 2], w[8 * v + 3]),
                          pack_bf16x2(w[8 * v + 4], w[8 * v + 5]), pack_bf16x2(w[8 * v + 6], w[8 * v + 7]));
    } else {
      float4* o = reinterpret_cast<float4*>(static_cast<float*>(a.out) + i * a.K + h * 32);
#pragma unroll
      for (int v = 0; v < 8; ++v) o[v] = make_float4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
    }
  }
}

}  // namespace

cudaError_t launch_embed_rows(const uint8_t* codes, const float* scales, int64_t V, int64_t K, const int64_t* ids,
                              int64_t n, void* out, bool out_bf16, const Codebook& cb, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  EmbedArgs a{codes, scales, ids, out, V, K, n, out_bf16 ? 1 : 0, cb};
  const int64_t chunks = n * (K >> 5);
  int64_t blocks = (chunks + 255) / 256;
  const int64_t cap = 152 * 8;  // grid-stride beyond eight blocks per SM
  blocks = blocks < cap ? blocks : cap;
  return checked_launch(reinterpret_cast<const void*>(&embed_rows_kernel), 256, 0,
                        [&] { embed_rows_kernel<<<(unsigned)blocks, 256, 0, s>>>(a); });
}

}  // namespace nf4k
