// gemv_tma.cuh -- N=1 NF4 GEMV with bulk-copy (TMA engine) weight streaming.
//
// Same arithmetic and epilogues as gemv_kernel.cuh (source: "Decode V2 --
// resident executor", section 6 "Linear primitive"), different data movement:
//  * each block owns a contiguous range of rows, whose codes and scales are
//    contiguous in memory; one producer thread streams them, RB rows per
//    stage, into a ring of S shared-memory stages with 1-D cp.async.bulk
//    copies completing on mbarriers ("full"), marked evict-first in L2 since
//    every weight is read once; a stage holds RB rows for each of GPS row
//    groups and the stages go round robin over the gpc / GPS sets of groups
//    (GPS = gpc: every group reads every stage; GPS = 1: small per-group
//    stages, for long rows or two matrices); a stage's rows complete on NB
//    "full" barriers of SUBR rows each, so the consumers start on the first
//    rows of a large stage while the rest are still in flight;
//  * consumer warps are x-stationary as before (thread t of a row group always
//    owns chunks t + G*j of a row, its x slice lives in registers) and read the
//    codes of each staged row from shared memory (conflict-free 16-byte loads),
//    then release the stage ("empty") for the producer to refill.
// Bytes in flight per SM are set by the ring (tens of KB), not by how many
// registers the consumers can spare, which is what bounded the register-
// prefetch kernel.  Every barrier wait is bounded (mbar_wait_bounded).
//
// Dequantization modes (LUTM):
//  LUT_F32     pair table of exact fp32 levels: per code byte one PRMT, one
//              conflict-free LDS.64 and two FFMAs.  Bound by
//              shared-memory bandwidth (8 bytes per two weights).  The default
//              for every activation dtype.
//  LUT_F16MIX  opt-in for bf16 activations (NF4_LUT=1): pair table of
//              fp16-rounded levels (relative error up to 2^-12 per level):
//              one LDS.32 per code byte halves the shared-memory traffic, and
//              each weight costs one mixed-precision FMA (f16 x f16 -> f32
//              accumulate; the product is exact in fp32).  The thread's x
//              slice is held as fp16 after scaling by a power of two that puts
//              its largest magnitude in [2^14, 2^15); the scale is undone
//              exactly with the block scale.  A bf16 value converts exactly
//              only while its scaled exponent is at least -17: values more
//              than 2^31 below the slice's largest magnitude land in fp16
//              subnormals and lose bits, or round to zero.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gemv_kernel.cuh"

namespace nf4k {

enum LutMode : int { LUT_F32 = 0, LUT_F16MIX = 1 };

// Shared-memory plan of one launch (host-computed).
struct TmaPlan {
  int SR;          // rows per stage (= GPS * RB)
  int GPS;         // row groups sharing one stage (a divisor of gpc)
  int S;           // stages
  int stage_bytes; // bytes of one stage (all matrices: codes then scales)
  int codes_bytes; // SR * K/2, one matrix
  int scales_bytes;// SR * K/64 * 4, one matrix
  int bar_off;     // offset of the S*(NB+1) mbarriers
  int red_off;     // offset of the reduction buffers
  int SUBR;        // rows per full barrier: SUB, or SR (one per stage)
  int NB;          // full barriers per stage (SR / SUBR)
};

// Two mixed-precision FMAs: acc0 += lo(h) * lo(x), acc1 += hi(h) * hi(x),
// f16 operands, f32 accumulation.
__device__ __forceinline__ void fma2_f16_f32(float& acc0, float& acc1, uint32_t h, uint32_t x) {
  asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\t"
      "mov.b32 {a0, a1}, %2;\n\t"
      "mov.b32 {b0, b1}, %3;\n\t"
      "fma.rn.f32.f16 %0, a0, b0, %0;\n\t"
      "fma.rn.f32.f16 %1, a1, b1, %1;\n\t}"
      : "+f"(acc0), "+f"(acc1)
      : "r"(h), "r"(x));
}

// sum over the 32 weights of one chunk of level(code) * x, fp16 levels and
// fp16 x pairs (xh[i] holds x[2i] in its low half, x[2i+1] in its high half).
__device__ __forceinline__ float chunk_dot_f16mix(const uint4 c, const uint32_t (&xh)[16], uint32_t laneoff,
                                                  const uint8_t* lut) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t off = __byte_perm(w[q], laneoff, 0x5504u | (j << 4));
      const uint32_t h = *reinterpret_cast<const uint32_t*>(lut + off);
      fma2_f16_f32(acc[2 * j], acc[2 * j + 1], h, xh[4 * q + j]);
    }
  }
  return ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
}

template <int NCH, int RB, int SUB, int EPI, bool XBF16, int LUTM>
__global__ void gemv_tma_kernel(const __grid_constant__ GemvArgs a, const __grid_constant__ TmaPlan P) {
  static_assert(SUB >= 1 && RB % SUB == 0, "SUB rows per full barrier must divide RB");
  static_assert(EPI != EPI_GLU || RB % 2 == 0, "gate/up pairs need an even number of rows per group");
  constexpr int NV = (EPI == EPI_SWIGLU) ? 2 : 1;
  constexpr int PL = Log2<RB>::value;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ float cbs[16];
  __shared__ unsigned long long warp_keys[32];
  __shared__ int s_abort;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int G = a.G;
  const int NC = G * a.gpc;  // consumer threads; the last warp produces
  const bool is_producer = tid >= NC;
  const int group = is_producer ? 0 : tid / G;
  const int t = tid - group * G;
  const int wig = t >> 5;
  const int WPG = G >> 5;
  const int H = a.K >> 5;
  const int64_t R0 = part_first_row<EPI>(blockIdx.x, gridDim.x, a.M);
  const int64_t R1 = part_first_row<EPI>(blockIdx.x + 1, gridDim.x, a.M);
  const int n_it = (int)((R1 - R0 + P.SR - 1) / P.SR);
  const int row_bytes = a.K >> 1;
  const int nblk = a.K >> 6;

  uint8_t* stages = smem + LUT_BYTES;
  // full[s][b] at bar0 + 8(s NB + b), empty[s] at bar0 + 8(S NB + s)
  const uint32_t bar0 = smem_addr(smem + P.bar_off);
  auto full_bar = [&](int s, int b) { return bar0 + 8u * (uint32_t)(s * P.NB + b); };
  auto empty_bar = [&](int s) { return bar0 + 8u * (uint32_t)(P.S * P.NB + s); };

  // Reduction slots: per group, S + 1 slots of NV x RB x WPG partial sums and
  // one arrival counter each (see the stage loop).
  const int R = P.S + 1;
  const int slot_floats = NV * RB * WPG;
  float* red = reinterpret_cast<float*>(smem + P.red_off);
  int* red_cnt = reinterpret_cast<int*>(smem + P.red_off) + a.gpc * R * slot_floats;

  // Barrier ids: 13 = consumers only, 15 = consumers + producer (initialized
  // barriers, complete pair table).  The producer never waits on either.
  if (is_producer) {
    if (lane == 0) {
      for (int s = 0; s < P.S; ++s) {
        for (int b = 0; b < P.NB; ++b) mbar_init(full_bar(s, b), 1);
        mbar_init(empty_bar(s), (uint32_t)(P.GPS * WPG));  // the owning groups' warps release it
      }
      mbar_init_fence();
      s_abort = 0;
    }
    __syncwarp();
    named_bar_arrive(15, NC + 32);
  } else {
    if (tid < 16) cbs[tid] = a.cb.v[tid];
    for (int i = tid; i < a.gpc * R; i += NC) red_cnt[i] = 0;
    named_bar_sync(13, NC);
  }

  // producer: issue the first S stages before anything else
  uint64_t policy = 0;
  const uint8_t* mcodes[NV];
  const float* mscales[NV];
  mcodes[0] = a.codes;
  mscales[0] = a.scales;
  if (NV == 2) {
    mcodes[NV - 1] = a.codes2;
    mscales[NV - 1] = a.scales2;
  }
  // Rows [g, g + n) of the row space as contiguous pieces of one matrix each:
  // fn(codes, scales, first row in that matrix, first stage row, rows).  Only
  // the fused q/k/v row space has more than one piece (segment boundaries).
  auto for_pieces = [&](int n_mat, int64_t g, int n, int srow, auto&& fn) {
    if (EPI != EPI_QKV) {
      fn(mcodes[n_mat], mscales[n_mat], g, srow, n);
      return;
    }
    while (n > 0) {
      const int sg = qkv_seg(a, g);
      const int64_t first = qkv_first(a, sg);
      const int64_t end = qkv_end(a, sg);
      const int piece = (int)((end - g) < n ? (end - g) : n);
      fn(qkv_pick(sg, a.seg_codes[0], a.seg_codes[1], a.seg_codes[2]),
         qkv_pick(sg, a.seg_scales[0], a.seg_scales[1], a.seg_scales[2]), g - first, srow, piece);
      g += piece;
      srow += piece;
      n -= piece;
    }
  };
  // one stage: per full barrier, the codes and scales of its SUBR rows (rows
  // are contiguous in memory and in the stage, so one copy per matrix each);
  // a barrier whose rows lie past the block's end is completed by a plain
  // arrival, so every barrier completes every phase
  auto issue = [&](int it) {
    const int s = it % P.S;
    const int64_t rb = R0 + (int64_t)it * P.SR;
    const int rows = (int)((R1 - rb) < P.SR ? (R1 - rb) : P.SR);
    uint8_t* st = stages + (size_t)s * P.stage_bytes;
    for (int b = 0; b < P.NB; ++b) {
      const int r0 = b * P.SUBR;
      const int nr = rows - r0 < P.SUBR ? rows - r0 : P.SUBR;
      const uint32_t fb = full_bar(s, b);
      if (nr <= 0) {
        mbar_arrive(fb);
        continue;
      }
      const uint32_t cb = (uint32_t)nr * (uint32_t)row_bytes;
      const uint32_t sb = (uint32_t)nr * (uint32_t)nblk * 4u;
      mbar_arrive_expect_tx(fb, NV * (cb + sb));
#pragma unroll
      for (int n = 0; n < NV; ++n)
        for_pieces(n, rb + r0, nr, r0, [&](const uint8_t* cp, const float* sp, int64_t lr, int sr, int pr) {
          bulk_g2s(smem_addr(st + n * P.codes_bytes + sr * row_bytes), cp + lr * row_bytes,
                   (uint32_t)pr * (uint32_t)row_bytes, fb, policy);
          bulk_g2s(smem_addr(st + NV * P.codes_bytes + n * P.scales_bytes + sr * nblk * 4), sp + lr * nblk,
                   (uint32_t)pr * (uint32_t)nblk * 4u, fb, policy);
        });
    }
  };
  // Before the previous kernel on the stream has finished (programmatic
  // dependent launch) only shared memory and L2 prefetches are touched.
  pdl_launch_dependents();
  int issued = 0;
  if (is_producer && lane == 0) {
    policy = policy_evict_first();
    for (int it = 0; it < n_it && it < P.S; ++it) {
      const int64_t rb = R0 + (int64_t)it * P.SR;
      const int rows = (int)((R1 - rb) < P.SR ? (R1 - rb) : P.SR);
#pragma unroll
      for (int n = 0; n < NV; ++n)
        for_pieces(n, rb, rows, 0, [&](const uint8_t* cp, const float* sp, int64_t lr, int, int pr) {
          bulk_prefetch_l2(cp + lr * row_bytes, (uint32_t)pr * (uint32_t)row_bytes);
          bulk_prefetch_l2(sp + lr * nblk, (uint32_t)pr * (uint32_t)nblk * 4u);
        });
    }
  }

  // The producer goes straight to its copies (the first bytes are on the
  // critical path of short kernels); the consumers build the pair table:
  // byte b, lane l -> (cb[b & 15], cb[b >> 4]) at b * 256 + l * (4 or 8),
  // written 16 bytes (4 or 2 identical lane replicas) at a time.
  if (is_producer) {
    pdl_wait();  // global reads and writes follow the previous kernel's completion
    if (lane == 0)
      for (; issued < n_it && issued < P.S; ++issued) issue(issued);
  } else {
    if (LUTM == LUT_F16MIX) {
      for (int i = tid; i < 256 * 8; i += NC) {
        const int b = i >> 3, q = i & 7;
        const __half2 h = __floats2half2_rn(cbs[b & 15], cbs[b >> 4]);
        const uint32_t u = *reinterpret_cast<const uint32_t*>(&h);
        *reinterpret_cast<uint4*>(smem + b * 256 + q * 16) = make_uint4(u, u, u, u);
      }
    } else {
      for (int i = tid; i < 256 * 16; i += NC) {
        const int b = i >> 4, q = i & 15;
        const uint32_t lo = __float_as_uint(cbs[b & 15]), hi = __float_as_uint(cbs[b >> 4]);
        *reinterpret_cast<uint4*>(smem + b * 256 + q * 16) = make_uint4(lo, hi, lo, hi);
      }
    }
    pdl_wait();
  }

  // consumers: x slice to registers (fp32, or scaled fp16 pairs for LUT_F16MIX)
  int cidx[NCH];
  bool cval[NCH];
  float xv[NCH][32];
  uint32_t xh[NCH][16];
  float xinv[NCH];  // 1 / (power-of-two scale of the fp16 slice)
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    cidx[j] = t + G * j;
    cval[j] = !is_producer && cidx[j] < H;
    xinv[j] = 1.f;
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
    if (LUTM == LUT_F16MIX) {
      // largest magnitude of the slice -> scale 2^(14 - e), e its exponent
      uint32_t mbits = 0;
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const uint32_t b = __float_as_uint(xv[j][e]) & 0x7FFFFFFFu;
        mbits = b > mbits ? b : mbits;
      }
      int ex = (int)(mbits >> 23) - 127;
      ex = ex < -100 ? -100 : ex;
      const float sig = __uint_as_float((uint32_t)(127 + 14 - ex) << 23);
      xinv[j] = __uint_as_float((uint32_t)(127 - 14 + ex) << 23);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const __half2 h = __floats2half2_rn(xv[j][2 * e] * sig, xv[j][2 * e + 1] * sig);
        xh[j][e] = *reinterpret_cast<const uint32_t*>(&h);
      }
    }
  }

  // consumers: the barriers are initialized and the pair table is complete
  if (!is_producer) named_bar_sync(15, NC + 32);

  volatile int* abort = &s_abort;
  unsigned long long best = 0ull;

  if (is_producer) {
    if (lane == 0) {
      for (; issued < n_it; ++issued) {
        const int s = issued % P.S;
        // the consumers released this stage's previous use (iteration issued - S)
        if (!mbar_wait_bounded(empty_bar(s), (uint32_t)(((issued / P.S) - 1) & 1), abort, a.wait_polls)) break;
        issue(issued);
      }
      if (*abort) {
        // drain: wait (bounded, ignoring the abort flag) for every copy that
        // may still be in flight, so none lands after the block has exited
        for (int it = (issued > P.S ? issued - P.S : 0); it < issued; ++it)
          for (int b = 0; b < P.NB; ++b)
            for (uint32_t i = 0; i < kWaitPolls; ++i)
              if (mbar_try_wait(full_bar(it % P.S, b), (uint32_t)((it / P.S) & 1))) break;
      }
    }
  } else {
    const uint8_t* lut = smem;
    const uint32_t laneoff = (uint32_t)lane * (LUTM == LUT_F16MIX ? 4u : 8u);
    int cidx_c[NCH];
#pragma unroll
    for (int j = 0; j < NCH; ++j) cidx_c[j] = cval[j] ? cidx[j] : 0;
    int li = 0;  // this group's stage count
    // stage it belongs to the GPS groups of set it % (gpc / GPS); within the
    // stage, group g reads rows (g % GPS) * RB .. + RB
    const int sets = a.gpc / P.GPS;
    const int pos = group % P.GPS;
    // after the warp transpose reduction, lane holds row slot rs; one lane
    // per slot (rep) carries it on
    const int rs = (PL == 0) ? 0 : (lane >> (5 - PL));
    const bool rep = (lane & ((32 >> PL) - 1)) == 0;
    for (int it = group / P.GPS; it < n_it; it += sets) {
      const int s = it % P.S;
      const uint32_t par = (uint32_t)((it / P.S) & 1);
      const int64_t rb = R0 + (int64_t)it * P.SR;
      const int rows = (int)((R1 - rb) < P.SR ? (R1 - rb) : P.SR);
      // the residual of the row this thread will write, fetched now so its
      // latency hides under the stage's arithmetic
      float resid_v = 0.f;
      if (EPI == EPI_RESID) {
        const int my = (WPG == 1) ? (rep ? pos * RB + rs : -1) : (lane < RB ? pos * RB + lane : -1);
        if (my >= 0 && my < rows) resid_v = a.resid[rb + my];
      }
      const uint8_t* st = stages + (size_t)s * P.stage_bytes;
      // Branch-free: every thread computes all RB rows of its group.  Chunks a
      // thread does not own read chunk 0 with x = 0 and add exactly zero; rows
      // past the end of the last stage compute garbage that is never stored.
      // The group's RB rows are taken SUB at a time: wait for the full barrier
      // that covers them, read all their codes and scales (the loads issue
      // back to back), then multiply them out.
      float acc[NV][RB];
#pragma unroll
      for (int sb = 0; sb < RB / SUB; ++sb) {
        const int lr0 = pos * RB + sb * SUB;
        mbar_wait_bounded(full_bar(s, lr0 / P.SUBR), par, abort, a.wait_polls);
        uint4 c[NV][SUB][NCH];
        float scl[NV][SUB][NCH];
#pragma unroll
        for (int n = 0; n < NV; ++n) {
          const uint8_t* sc = st + n * P.codes_bytes;
          const float* ss = reinterpret_cast<const float*>(st + NV * P.codes_bytes + n * P.scales_bytes);
#pragma unroll
          for (int i = 0; i < SUB; ++i)
#pragma unroll
            for (int j = 0; j < NCH; ++j) {
              c[n][i][j] = lds128(sc + (lr0 + i) * row_bytes + cidx_c[j] * 16);
              scl[n][i][j] = ss[(lr0 + i) * nblk + (cidx_c[j] >> 1)];
            }
        }
#pragma unroll
        for (int n = 0; n < NV; ++n)
#pragma unroll
          for (int i = 0; i < SUB; ++i) {
            float r = 0.f;
#pragma unroll
            for (int j = 0; j < NCH; ++j) {
              if (LUTM == LUT_F16MIX)
                r = fmaf(chunk_dot_f16mix(c[n][i][j], xh[j], laneoff, lut), scl[n][i][j] * xinv[j], r);
              else
                r = fmaf(chunk_dot(c[n][i][j], xv[j], laneoff, lut), scl[n][i][j], r);
            }
            acc[n][sb * SUB + i] = r;
          }
      }
      // the stage's shared memory is no longer read by this warp
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(s));

      float v[NV];
#pragma unroll
      for (int n = 0; n < NV; ++n) v[n] = transpose_reduce<RB>(acc[n], lane);
      int lr = -1;
      if (WPG == 1) {
        if (rep) lr = pos * RB + rs;
      } else {
        // Every warp leaves its partial sums in the group's slot and counts
        // itself in; the last warp to arrive adds the WPG partials in warp
        // order (deterministic) and writes the rows, while the others go on
        // to their next stage without waiting.  A slot is reused S + 1 stages
        // later: no warp can get that far ahead of the warp still reducing it,
        // because the producer refills a stage only after every warp has
        // released it.
        float* slot = red + (group * R + li % R) * slot_floats;
        int* cnt = red_cnt + group * R + li % R;
        if (rep) {
#pragma unroll
          for (int n = 0; n < NV; ++n) slot[(n * RB + rs) * WPG + wig] = v[n];
        }
        __syncwarp();
        int last = 0;
        if (lane == 0) {
          __threadfence_block();
          last = (atomicAdd(cnt, 1) == WPG - 1) ? 1 : 0;
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
          __threadfence_block();
          if (lane < RB) {
            lr = pos * RB + lane;
#pragma unroll
            for (int n = 0; n < NV; ++n) {
              float sum = 0.f;
              for (int w = 0; w < WPG; ++w) sum += slot[(n * RB + lane) * WPG + w];
              v[n] = sum;
            }
          }
          __syncwarp();
          if (lane == 0) *cnt = 0;
        }
      }
      ++li;
      // interleaved gate/up: the up sum of an even (gate) row sits one row
      // slot further on, RB-row slots apart in lanes (32 / RB) after the
      // transpose reduction, or in the next lane after the cross-warp sum
      float up = 0.f;
      if (EPI == EPI_GLU) up = __shfl_down_sync(0xffffffffu, v[0], WPG == 1 ? (32 >> PL) : 1);
      if (lr >= 0 && lr < rows && !*abort) {
        const int64_t row = rb + lr;
        if (EPI == EPI_PLAIN) {
          a.y[row] = v[0];
        } else if (EPI == EPI_RESID) {
          a.y[row] = v[0] + resid_v;
        } else if (EPI == EPI_SWIGLU) {
          const float g = v[0];
          const float u = v[NV - 1];
          const float silu = g / (1.0f + expf(-g));
          a.out_bf16[row] = __bfloat16_as_ushort(__float2bfloat16_rn(silu * u));
        } else if (EPI == EPI_QKV) {
          qkv_store(a, row, v[0]);
        } else if (EPI == EPI_GLU) {
          if ((lr & 1) == 0) {  // stages and groups start on even rows
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
    }
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

template <int NCH, int RB, int SUB, int EPI, bool XBF16, int LUTM>
const void* gemv_tma_ptr() {
  return reinterpret_cast<const void*>(&gemv_tma_kernel<NCH, RB, SUB, EPI, XBF16, LUTM>);
}

template <int NCH, int RB, int SUB, int EPI, bool XBF16, int LUTM>
cudaError_t launch_gemv_tma_instance(const GemvArgs& a, const TmaPlan& p, int blocks, int threads, int smem,
                                     cudaStream_t s) {
  return checked_launch(gemv_tma_ptr<NCH, RB, SUB, EPI, XBF16, LUTM>(), threads, smem, [&] {
    // one wave of persistent blocks: the next kernel may launch early
    // (programmatic dependent launch) and overlap its prologue with our tail
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    cudaLaunchKernelEx(&cfg, gemv_tma_kernel<NCH, RB, SUB, EPI, XBF16, LUTM>, a, p);
  });
}

}  // namespace nf4k
