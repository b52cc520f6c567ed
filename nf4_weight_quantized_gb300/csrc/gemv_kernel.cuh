// gemv_kernel.cuh -- the N=1 NF4 GEMV kernel family (plain / residual / SwiGLU / argmax).
//
// y[m] = sum_k cb[code(m,k)] * scale[m][k/64] * x[k], fp32 accumulation.
// Source: "Decode V2 -- resident executor", section 6 "Linear primitive" (the
// CUDA-core gemv backend: LUT x scale x x, split-K across threads, rows per
// block chosen per (M, K)) and section 3 (SiLU on the full gate sum).
//
// GB300 design (differs from the page's 4-warp / NR-rows block):
//  * x-stationary threads: a "row group" of G threads (a multiple of 32) walks
//    rows; thread t of the group always owns the same 16-byte code chunks
//    c = t + G*j (32 weights each) of every row, so its slice of x is widened
//    to fp32 into registers once per launch and reused for every row.
//  * weights stream with 128-bit non-allocating loads, one warp instruction
//    covering 512 contiguous bytes; a batch of RB rows is prefetched into
//    registers while the previous batch is computed.
//  * dequantization goes through a shared-memory pair table: for each code
//    byte (two weights) the float2 (cb[lo], cb[hi]) is replicated 32 times so
//    that lane l reads its own copy: one PRMT builds the address
//    (byte * 256 + lane * 8), one conflict-free LDS.64 yields two exact fp32
//    levels, two FFMAs consume them.  The block scale is applied once per chunk.
//  * row sums are reduced inside the warp by a transpose reduction (RB rows in
//    RB-1+5-log2(RB) shuffles instead of 5*RB) and across the warps of a group
//    through shared memory in a fixed order, so a row's result depends only on
//    its data, never on its position (identical rows give identical sums).
//  * argmax: one 64-bit key per block, (order-preserving value bits << 32) |
//    (~index), folded with atomicMax; the last block (ticket) decodes it and
//    re-zeroes the workspace.  No second launch, no waiting.
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"

namespace nf4k {

constexpr int LUT_BYTES = 256 * 256;  // 256 code bytes x 32 lane replicas x float2

template <int RB>
struct Log2 {
  static constexpr int value = RB <= 1 ? 0 : RB == 2 ? 1 : RB == 4 ? 2 : RB == 8 ? 3 : 4;
};

// Reduce RB per-lane partials across a warp.  On return the lane holds the
// warp total of row slot (lane >> (5 - log2 RB)).
template <int RB>
__device__ __forceinline__ float transpose_reduce(float (&v)[RB], int lane) {
  constexpr int P = Log2<RB>::value;
#pragma unroll
  for (int s = 0; s < P; ++s) {
    const int n = RB >> s;
    const int off = 16 >> s;
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? v[i] : v[i + n / 2];
      const float keep = upper ? v[i + n / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  float r = v[0];
#pragma unroll
  for (int off = 16 >> P; off >= 1; off >>= 1) r += __shfl_xor_sync(0xffffffffu, r, off);
  return r;
}

// sum over the 32 weights of one 16-byte code chunk of cb[code] * x, exact
// fp32 levels.  Per code byte: one PRMT (table address), one LDS.64 (both
// levels) and two FFMAs.  (A packed fma.rn.f32x2 per byte issues fewer
// instructions but measured slower inside the kernels: 53.5 against 49.3 us
// on the 151936 x 2048 projection.)
__device__ __forceinline__ float chunk_dot(const uint4 c, const float (&xv)[32], uint32_t laneoff,
                                           const uint8_t* lut) {
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      // byte 0 <- lane*8, byte 1 <- code byte j of word q, bytes 2-3 <- 0
      const uint32_t off = __byte_perm(w[q], laneoff, 0x5504u | (j << 4));
      const float2 v = *reinterpret_cast<const float2*>(lut + off);
      acc[j] = fmaf(v.x, xv[8 * q + 2 * j], acc[j]);
      acc[j] = fmaf(v.y, xv[8 * q + 2 * j + 1], acc[j]);
    }
  }
  return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

// Order-preserving 64-bit argmax key: larger value wins, then lower index.
__device__ __forceinline__ unsigned long long argmax_key(float v, int64_t row) {
  if (v == 0.0f) v = 0.0f;  // +0 and -0 tie
  const uint32_t u = __float_as_uint(v);
  const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)ord << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)row);
}

template <int NCH, int RB, int NV>
struct Batch {
  uint4 c[NV][RB][NCH];
  float s[NV][RB][NCH];
};

template <int NCH, int RB, int EPI, bool XBF16>
__device__ __forceinline__ void gemv_body(const GemvArgs& a) {
  constexpr int NV = (EPI == EPI_SWIGLU) ? 2 : 1;  // matrices per row
  constexpr int P = Log2<RB>::value;
  static_assert(EPI != EPI_GLU || RB % 2 == 0, "gate/up pairs need an even number of rows per batch");
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float cbs[16];
  __shared__ unsigned long long warp_keys[32];

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int G = a.G;
  const int group = tid / G;
  const int t = tid - group * G;
  const int wig = t >> 5;
  const int WPG = G >> 5;
  const int H = a.K >> 5;  // 16-byte chunks per row
  const int64_t NG = (int64_t)gridDim.x * a.gpc;
  const int64_t gg = (int64_t)blockIdx.x * a.gpc + group;
  const int64_t r0 = part_first_row<EPI>(gg, NG, a.M);
  const int64_t r1 = part_first_row<EPI>(gg + 1, NG, a.M);
  const int64_t row_bytes = a.K >> 1;
  const int64_t nblk = a.K >> 6;

  int cidx[NCH];
  bool cval[NCH];
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    cidx[j] = t + G * j;
    cval[j] = cidx[j] < H;
  }

  const uint8_t* codes[NV];
  const float* scales[NV];
  codes[0] = a.codes;
  scales[0] = a.scales;
  if (NV == 2) {
    codes[NV - 1] = a.codes2;
    scales[NV - 1] = a.scales2;
  }

  auto load_batch = [&](Batch<NCH, RB, NV>& B, int64_t rb0) {
#pragma unroll
    for (int n = 0; n < NV; ++n)
#pragma unroll
      for (int i = 0; i < RB; ++i)
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          const int64_t row = rb0 + i;
          if (row < r1 && cval[j]) {
            const uint8_t* cp = codes[n];
            const float* sp = scales[n];
            int64_t lr = row;
            if (EPI == EPI_QKV) {  // the row's own matrix
              const int sg = qkv_seg(a, row);
              lr = row - qkv_first(a, sg);
              cp = qkv_pick(sg, a.seg_codes[0], a.seg_codes[1], a.seg_codes[2]);
              sp = qkv_pick(sg, a.seg_scales[0], a.seg_scales[1], a.seg_scales[2]);
            }
            B.c[n][i][j] = ld_stream_v4(cp + lr * row_bytes + (int64_t)cidx[j] * 16);
            B.s[n][i][j] = ld_nc_f32(sp + lr * nblk + (cidx[j] >> 1));
          } else {
            B.c[n][i][j] = make_uint4(0x77777777u, 0x77777777u, 0x77777777u, 0x77777777u);
            B.s[n][i][j] = 0.f;
          }
        }
  };

  Batch<NCH, RB, NV> A, Bn;
  load_batch(A, r0);

  // this thread's slice of x, widened to fp32 once
  float xv[NCH][32];
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    if (cval[j]) {
      if (XBF16) {
        const uint8_t* xp = reinterpret_cast<const uint8_t*>(a.x) + (int64_t)cidx[j] * 64;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 u = ld_nc_v4(xp + 16 * q);
          const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            xv[j][8 * q + 2 * e] = bf16lo_to_f32(w[e]);
            xv[j][8 * q + 2 * e + 1] = bf16hi_to_f32(w[e]);
          }
        }
      } else {
        const uint8_t* xp = reinterpret_cast<const uint8_t*>(a.x) + (int64_t)cidx[j] * 128;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 u = ld_nc_v4(xp + 16 * q);
          xv[j][4 * q + 0] = __uint_as_float(u.x);
          xv[j][4 * q + 1] = __uint_as_float(u.y);
          xv[j][4 * q + 2] = __uint_as_float(u.z);
          xv[j][4 * q + 3] = __uint_as_float(u.w);
        }
      }
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) xv[j][e] = 0.f;
    }
  }

  // pair table (built while the first batch is in flight)
  if (tid < 16) cbs[tid] = a.cb.v[tid];
  __syncthreads();
  for (int i = tid; i < LUT_BYTES / 8; i += blockDim.x) {
    const int b = i >> 5;
    reinterpret_cast<float2*>(smem)[i] = make_float2(cbs[b & 15], cbs[b >> 4]);
  }
  __syncthreads();

  const uint8_t* lut = smem;
  const uint32_t laneoff = (uint32_t)lane * 8u;
  float* red = reinterpret_cast<float*>(smem + LUT_BYTES) + group * (2 * NV * RB * WPG);
  int buf = 0;
  unsigned long long best = 0ull;

  auto process = [&](const Batch<NCH, RB, NV>& B, int64_t rb0) {
    float acc[NV][RB];
#pragma unroll
    for (int n = 0; n < NV; ++n)
#pragma unroll
      for (int i = 0; i < RB; ++i) {
        float r = 0.f;
#pragma unroll
        for (int j = 0; j < NCH; ++j) r = fmaf(chunk_dot(B.c[n][i][j], xv[j], laneoff, lut), B.s[n][i][j], r);
        acc[n][i] = r;
      }
    float v[NV];
#pragma unroll
    for (int n = 0; n < NV; ++n) v[n] = transpose_reduce<RB>(acc[n], lane);
    const int rs = (P == 0) ? 0 : (lane >> (5 - P));
    const bool rep = (lane & ((32 >> P) - 1)) == 0;

    int64_t row = -1;
    if (WPG == 1) {
      if (rep) row = rb0 + rs;
    } else {
      float* rb = red + buf * (NV * RB * WPG);
      if (rep) {
#pragma unroll
        for (int n = 0; n < NV; ++n) rb[(n * RB + rs) * WPG + wig] = v[n];
      }
      named_bar_sync(1 + group, G);
      if (t < RB) {
        row = rb0 + t;
#pragma unroll
        for (int n = 0; n < NV; ++n) {
          float s = 0.f;
          for (int w = 0; w < WPG; ++w) s += rb[(n * RB + t) * WPG + w];
          v[n] = s;
        }
      }
      buf ^= 1;
    }
    // interleaved gate/up: the up sum of an even (gate) row sits one row slot
    // further on (32 / RB lanes after the transpose reduction, the next lane
    // after the cross-warp sum); batches start on even rows
    float up = 0.f;
    if (EPI == EPI_GLU) up = __shfl_down_sync(0xffffffffu, v[0], WPG == 1 ? (32 >> P) : 1);
    if (row >= 0 && row < r1) {
      if (EPI == EPI_PLAIN) {
        a.y[row] = v[0];
      } else if (EPI == EPI_RESID) {
        a.y[row] = v[0] + a.resid[row];
      } else if (EPI == EPI_SWIGLU) {
        const float g = v[0];
        const float u = v[NV - 1];
        const float silu = g / (1.0f + expf(-g));
        a.out_bf16[row] = __bfloat16_as_ushort(__float2bfloat16_rn(silu * u));
      } else if (EPI == EPI_QKV) {
        qkv_store(a, row, v[0]);
      } else if (EPI == EPI_GLU) {
        if (((row - rb0) & 1) == 0) {
          const float g = v[0];
          const float silu = g / (1.0f + expf(-g));
          a.out_bf16[row >> 1] = __bfloat16_as_ushort(__float2bfloat16_rn(silu * up));
        }
      } else {
        a.y[row] = v[0];
        const unsigned long long k = argmax_key(v[0], row);
        best = k > best ? k : best;
      }
    }
  };

  for (int64_t rb0 = r0; rb0 < r1; rb0 += 2 * RB) {
    load_batch(Bn, rb0 + RB);
    process(A, rb0);
    load_batch(A, rb0 + 2 * RB);
    if (rb0 + RB < r1) process(Bn, rb0 + RB);
  }

  if (EPI == EPI_ARGMAX) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, off);
      best = o > best ? o : best;
    }
    if (lane == 0) warp_keys[tid >> 5] = best;
    __syncthreads();
    if (tid < 32) {
      unsigned long long k = (tid < (int)(blockDim.x >> 5)) ? warp_keys[tid] : 0ull;
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, k, off);
        k = o > k ? o : k;
      }
      if (tid == 0) {
        if (k) atomicMax(&a.ws[0], k);
        __threadfence();
        const unsigned int prev = atomicAdd(reinterpret_cast<unsigned int*>(&a.ws[1]), 1u);
        if (prev == gridDim.x - 1) {
          const unsigned long long fin = atomicExch(&a.ws[0], 0ull);
          *a.index = (int64_t)(0xFFFFFFFFu - (uint32_t)(fin & 0xFFFFFFFFull));
          atomicExch(reinterpret_cast<unsigned int*>(&a.ws[1]), 0u);
        }
      }
    }
  }
}

// The register allocation is left free (up to 255 per thread) ...
template <int NCH, int RB, int EPI, bool XBF16>
__global__ void gemv_kernel(const __grid_constant__ GemvArgs a) {
  gemv_body<NCH, RB, EPI, XBF16>(a);
}

// ... or capped at 64 so that one row group can span a 1024-thread block for
// very long rows (K above ~20k).
template <int NCH, int RB, int EPI, bool XBF16>
__global__ void __launch_bounds__(1024) gemv_kernel_big(const __grid_constant__ GemvArgs a) {
  gemv_body<NCH, RB, EPI, XBF16>(a);
}

template <int NCH, int RB, int EPI, bool XBF16, bool BIG>
const void* gemv_instance_ptr() {
  return BIG ? reinterpret_cast<const void*>(&gemv_kernel_big<NCH, RB, EPI, XBF16>)
             : reinterpret_cast<const void*>(&gemv_kernel<NCH, RB, EPI, XBF16>);
}

// Launch one instantiation with the given configuration.
template <int NCH, int RB, int EPI, bool XBF16, bool BIG>
cudaError_t launch_gemv_instance(const GemvArgs& a, const GemvConfig& cfg, cudaStream_t s) {
  return checked_launch(gemv_instance_ptr<NCH, RB, EPI, XBF16, BIG>(), cfg.G * cfg.gpc, cfg.smem, [&] {
    if (BIG)
      gemv_kernel_big<NCH, RB, EPI, XBF16><<<cfg.blocks, cfg.G * cfg.gpc, cfg.smem, s>>>(a);
    else
      gemv_kernel<NCH, RB, EPI, XBF16><<<cfg.blocks, cfg.G * cfg.gpc, cfg.smem, s>>>(a);
  });
}

}  // namespace nf4k
