// chunk.cu -- prefill chunk (N <= 32 tokens) on the tcgen05 tensor cores.
//
// Y[n][m] = sum_k X[n][k] * bf16(W_hat[m][k]), fp32 accumulation.
// Source: "Decode V2 -- resident executor", section 0 "Goals" item 1 and
// section 5 (the prompt is consumed in chunks of LIVE_MAX_N = 32 through the
// tensor-core GEMM so each weight is read once per chunk); the page's kernel
// is a desktop mma design, this one is written for sm_103a:
//
//  * one block owns a 128-row tile of W (the MMA's M) and a K range;
//  * eight producer warps stream the tile's NF4 codes (two lanes per 32-byte
//    row segment, 16-byte loads), dequantize them through the lane-replicated
//    pair table (fp32 level * fp32 scale, rounded once to bf16) and store the
//    bf16 tile straight into shared memory in the K-major 128-byte-swizzled
//    layout the tensor core reads; they also stage the matching 64-column
//    slice of X (rows n >= N are zero) the same way;
//  * one thread issues tcgen05.mma (M = 128, N = 32, K = 16 per instruction,
//    4 per 64-column stage) into a 32-column fp32 accumulator in TMEM, and
//    releases each stage with tcgen05.commit;
//  * after the last stage, four warps read the accumulator back with
//    tcgen05.ld (warp w owns TMEM lanes 32w..32w+31 = tile rows) and store Y
//    coalesced along m.
// Stages form a ring of S buffers guarded by mbarriers; every wait is bounded
// and the block always frees its TMEM.  With K split into P ranges, the P
// partial tiles of one row tile are summed in a fixed order by the last block
// to finish that tile (a per-tile ticket in the caller's workspace), so the
// result is deterministic.
#include <cstdio>
#include <string>

#include "gemv_kernel.cuh"

namespace nf4k {

namespace {

constexpr int TILE_M = 128;    // MMA M: rows of W per block
constexpr int TILE_N = 32;     // MMA N: tokens (X rows, zero padded)
constexpr int KT = 64;         // K columns per stage (one NF4 block, one 128-byte swizzle atom)
constexpr int NPW = 8;         // producer warps
constexpr int NTHREADS = NPW * 32 + 32;  // + the MMA warp
constexpr int A_BYTES = TILE_M * KT * 2;  // 16 KB
constexpr int B_BYTES = TILE_N * KT * 2;  // 4 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 32;

struct ChunkArgs {
  const uint8_t* codes;
  const float* scales;
  const uint16_t* X;
  float* Y;
  float* partial;         // [P][N][M] when P > 1
  unsigned int* tickets;  // [tiles] when P > 1
  int M, K, N;
  int P;                  // K ranges
  int S;                  // stages
  Codebook cb;
};

// Byte offset of (row r, 16-byte chunk c) inside a K-major 128-byte-swizzled
// tile whose rows are 128 bytes (64 bf16): 8-row groups 1024 B apart, rows
// 128 B apart, chunk index XOR (r % 8).
__device__ __forceinline__ uint32_t sw128_offset(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

__global__ void __launch_bounds__(NTHREADS, 1) chunk_kernel(const __grid_constant__ ChunkArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ float cbs[16];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ unsigned long long s_bars[2 * 8 + 1];
  __shared__ unsigned int s_last;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int tile = blockIdx.x / a.P;
  const int part = blockIdx.x % a.P;
  const int m0 = tile * TILE_M;
  const int nkt_all = a.K / KT;
  const int kt0 = (int)((int64_t)part * nkt_all / a.P);
  const int kt1 = (int)((int64_t)(part + 1) * nkt_all / a.P);
  const int nkt = kt1 - kt0;
  const int S = a.S;

  // stages start 1024-aligned after the pair table
  uint8_t* stage0 = smem + LUT_BYTES;
  const uint32_t bar_full = smem_addr(&s_bars[0]);
  const uint32_t bar_empty = smem_addr(&s_bars[8]);
  const uint32_t bar_done = smem_addr(&s_bars[16]);
  auto full_bar = [&](int s) { return bar_full + 8u * s; };
  auto empty_bar = [&](int s) { return bar_empty + 8u * s; };

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), NPW);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(bar_done, 1);
    mbar_init_fence();
    s_abort = 0;
  }
  if (tid < 16) cbs[tid] = a.cb.v[tid];
  if (warp == NPW) {  // the MMA warp owns the accumulator
    tmem_alloc(smem_addr(&s_tmem), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = s_tmem;

  for (int i = tid; i < LUT_BYTES / 8; i += NTHREADS) {
    const int b = i >> 5;
    reinterpret_cast<float2*>(smem)[i] = make_float2(cbs[b & 15], cbs[b >> 4]);
  }
  __syncthreads();

  volatile int* abort = &s_abort;
  // the swizzled operand tiles must sit on 1024-byte boundaries
  if (tid == 0 && (smem_addr(stage0) & 1023u) != 0) {
    s_abort = 1;
    atomicOr(&g_nf4_device_error, kErrWaitTimeout);
  }
  __syncthreads();
  const int row_bytes = a.K >> 1;
  const int nblk = a.K >> 6;

  if (warp < NPW) {
    // ---------------------------------------------------------- producers
    const int pt = tid;                  // 0..255
    const int r = pt >> 1;               // tile row 0..127
    const int h = pt & 1;                // half of the 64-column stage
    const int64_t grow = (int64_t)m0 + r;
    const bool rvalid = grow < a.M;
    const uint32_t laneoff = (uint32_t)lane * 8u;
    // X chunk handled by this thread: row n = pt >> 3, 16-byte chunk c = pt & 7
    const int xn = pt >> 3, xc = pt & 7;
    for (int it = 0; it < nkt; ++it) {
      const int s = it % S;
      const int kt = kt0 + it;
      uint4 code = make_uint4(0x77777777u, 0x77777777u, 0x77777777u, 0x77777777u);
      float sc = 0.f;
      if (rvalid) {
        code = ld_stream_v4(a.codes + grow * row_bytes + (int64_t)kt * 32 + h * 16);
        sc = ld_nc_f32(a.scales + grow * nblk + kt);
      }
      uint4 xv = make_uint4(0u, 0u, 0u, 0u);
      if (xn < a.N) xv = ld_nc_v4(a.X + (int64_t)xn * a.K + (int64_t)kt * KT + xc * 8);
      if (it >= S) mbar_wait_bounded(empty_bar(s), (uint32_t)(((it / S) - 1) & 1), abort);
      uint8_t* A = stage0 + s * STAGE_BYTES;
      uint8_t* B = A + A_BYTES;
      // 16 code bytes -> 32 bf16 = four 16-byte chunks (c = 4h .. 4h+3)
      const uint32_t w[4] = {code.x, code.y, code.z, code.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t packed[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t off = __byte_perm(w[q], laneoff, 0x5504u | (j << 4));
          const float2 v = *reinterpret_cast<const float2*>(smem + off);
          packed[j] = pack_bf16x2(v.x * sc, v.y * sc);
        }
        *reinterpret_cast<uint4*>(A + sw128_offset(r, 4 * h + q)) =
            make_uint4(packed[0], packed[1], packed[2], packed[3]);
      }
      *reinterpret_cast<uint4*>(B + sw128_offset(xn, xc)) = xv;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(full_bar(s));
    }
  } else if (lane == 0) {
    // ------------------------------------------------------ MMA issuer
    const uint32_t idesc = idesc_bf16_f32(TILE_M, TILE_N);
    for (int it = 0; it < nkt; ++it) {
      const int s = it % S;
      mbar_wait_bounded(full_bar(s), (uint32_t)((it / S) & 1), abort);
      tc_fence_after_sync();
      if (!*abort) {
        const uint32_t A = smem_addr(stage0 + s * STAGE_BYTES);
        const uint32_t B = A + A_BYTES;
#pragma unroll
        for (int kk = 0; kk < KT / 16; ++kk)
          tc_mma_bf16(tmem, smem_desc_sw128(A + kk * 32), smem_desc_sw128(B + kk * 32), idesc,
                      (it > 0 || kk > 0) ? 1u : 0u);
      }
      tc_commit(empty_bar(s));
    }
    tc_commit(bar_done);
  }

  // ------------------------------------------------------------ epilogue
  if (warp < 4) {
    const bool ok = mbar_wait_bounded(bar_done, 0, abort);
    tc_fence_after_sync();
    uint32_t acc[32];
    tmem_ld_32x32b_x32(tmem + ((uint32_t)(warp * 32) << 16), acc);
    tmem_ld_wait();
    const int64_t m = (int64_t)m0 + warp * 32 + lane;
    if (ok && !*abort && m < a.M) {
      if (a.P == 1) {
#pragma unroll
        for (int n = 0; n < TILE_N; ++n)
          if (n < a.N) a.Y[(int64_t)n * a.M + m] = __uint_as_float(acc[n]);
      } else {
        float* dst = a.partial + (int64_t)part * a.N * a.M;
#pragma unroll
        for (int n = 0; n < TILE_N; ++n)
          if (n < a.N) dst[(int64_t)n * a.M + m] = __uint_as_float(acc[n]);
        __threadfence();  // the partial tile is visible device-wide before the ticket
      }
    }
  }
  if (warp == NPW && *abort) {
    // make sure no tensor-core op is still writing TMEM before it is freed
    for (uint32_t i = 0; i < kWaitPolls; ++i)
      if (mbar_try_wait(bar_done, 0)) break;
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == NPW) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, TMEM_COLS);
  }

  if (a.P > 1) {
    // the last block of this row tile sums the P partial tiles in order
    if (tid == 0) {
      __threadfence();
      const unsigned int prev = atomicAdd(&a.tickets[tile], 1u);
      s_last = (prev == (unsigned int)a.P - 1) ? 1u : 0u;
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
      const int rows = (a.M - m0) < TILE_M ? (a.M - m0) : TILE_M;
      // eight outputs per thread at a time, every partial loaded before any
      // store (independent loads, not one round trip per output); parts added
      // in order
      constexpr int OB = 8;
      for (int i0 = tid * OB; i0 < a.N * rows; i0 += NTHREADS * OB) {
        float sum[OB];
#pragma unroll
        for (int o = 0; o < OB; ++o) sum[o] = 0.f;
        for (int p = 0; p < a.P; ++p) {
          float v[OB];
#pragma unroll
          for (int o = 0; o < OB; ++o) {
            const int i = i0 + o;
            const int n = i / rows, rr = i - n * rows;
            v[o] = i < a.N * rows ? __ldcg(a.partial + (int64_t)p * a.N * a.M + (int64_t)n * a.M + m0 + rr) : 0.f;
          }
#pragma unroll
          for (int o = 0; o < OB; ++o) sum[o] += v[o];
        }
#pragma unroll
        for (int o = 0; o < OB; ++o) {
          const int i = i0 + o;
          const int n = i / rows, rr = i - n * rows;
          if (i < a.N * rows && !*abort) a.Y[(int64_t)n * a.M + m0 + rr] = sum[o];
        }
      }
      if (tid == 0) a.tickets[tile] = 0u;  // leave the workspace zeroed
    }
  }
}

// K ranges per row tile: enough blocks to fill the GPU in whole waves.
// (Planned for a 152-SM GB300 on every device, so that the workspace size
// depends only on the shape.)
int choose_parts(int M, int K, int sms = 152) {
  const int tiles = (M + TILE_M - 1) / TILE_M;
  const int nkt = K / KT;
  int best = 1;
  double best_t = 1e30;
  for (int p = 1; p <= 16 && p <= nkt; ++p) {
    const int64_t units = (int64_t)tiles * p;
    const int64_t waves = (units + sms - 1) / sms;
    const double t = (double)waves * ((double)nkt / p + 2.0);  // +2: per-block fill and epilogue
    if (t < best_t - 1e-9) {
      best_t = t;
      best = p;
    }
  }
  return best;
}

size_t fallback_partial_bytes(int64_t M, int64_t K, int N) {
  const int P = choose_parts((int)M, (int)K);
  return P <= 1 ? 0 : (size_t)P * N * M * 4;
}

}  // namespace

// chunk_tma.cu: the stream-K kernel, used when K % 256 == 0 and the operands
// are 16-byte aligned; this file's kernel serves every other shape.
bool chunk_tma_usable(int64_t K, const void* codes, const void* scales, const void* X);
size_t chunk_tma_partial_bytes(int64_t M, int64_t K, int N);
cudaError_t launch_chunk_tma(const uint8_t* codes, const float* scales, int M, int K, const uint16_t* X, int N,
                             float* Y, float* partial, unsigned int* tickets, const Codebook& cb, cudaStream_t s);
std::string describe_chunk_tma(int64_t M, int64_t K, int N);

// Workspace layout, either kernel: split-tile partials from the start, one
// ticket per 128-row tile at the end followed by 16 spare bytes.  Sized for
// the larger of the two kernels' needs (which one runs also depends on the
// pointers' alignment, not known here); split plans are made for a 152-SM
// GB300 on every device, so the size depends only on the shape.
size_t chunk_workspace_bytes(int64_t M, int64_t K, int N) {
  const size_t a = fallback_partial_bytes(M, K, N), b = chunk_tma_partial_bytes(M, K, N);
  const size_t part = a > b ? a : b;
  if (part == 0) return 16;
  const int64_t tiles = (M + TILE_M - 1) / TILE_M;
  return ((part + 255) / 256) * 256 + (size_t)tiles * 4 + 16;
}

cudaError_t launch_chunk(const uint8_t* codes, const float* scales, int M, int K, const uint16_t* X, int N, float* Y,
                         void* workspace, const Codebook& cb, cudaStream_t s, int device) {
  const size_t ws_bytes = chunk_workspace_bytes(M, K, N);
  const int64_t tiles_all = (M + TILE_M - 1) / TILE_M;
  unsigned int* tickets =
      ws_bytes > 16 ? reinterpret_cast<unsigned int*>(reinterpret_cast<uint8_t*>(workspace) + ws_bytes - 16 - tiles_all * 4)
                    : nullptr;
  if (chunk_tma_usable(K, codes, scales, X))
    return launch_chunk_tma(codes, scales, M, K, X, N, Y, reinterpret_cast<float*>(workspace), tickets, cb, s);
  ChunkArgs a{};
  a.codes = codes;
  a.scales = scales;
  a.X = X;
  a.Y = Y;
  a.M = M;
  a.K = K;
  a.N = N;
  a.cb = cb;
  (void)device;
  a.P = choose_parts(M, K);
  if (a.P > 1) {
    a.partial = reinterpret_cast<float*>(workspace);
    a.tickets = tickets;
  }
  a.S = 4;
  const int smem = LUT_BYTES + a.S * STAGE_BYTES;
  const int tiles = (M + TILE_M - 1) / TILE_M;
  return checked_launch(reinterpret_cast<const void*>(&chunk_kernel), NTHREADS, smem,
                        [&] { chunk_kernel<<<tiles * a.P, NTHREADS, smem, s>>>(a); });
}

std::string describe_chunk(int64_t M, int64_t K, int N, int device) {
  (void)device;
  if (K % 256 == 0) return describe_chunk_tma(M, K, N) + " (16-byte aligned operands)";
  const int P = choose_parts((int)M, (int)K);
  char buf[256];
  std::snprintf(buf, sizeof buf,
                "chunk M=%lld K=%lld N=%d: tcgen05 M=%d N=%d K=16, %d row tiles x %d K range(s), %d stages of %d "
                "columns, %d threads",
                (long long)M, (long long)K, N, TILE_M, TILE_N, (int)((M + TILE_M - 1) / TILE_M), P, 4, KT, NTHREADS);
  return buf;
}

}  // namespace nf4k
