// chunk_tma.cu -- prefill chunk (N <= 32 tokens), persistent stream-K kernel fed
// by the tensor-memory-access (TMA) engine.
//
// Y[n][m] = sum_k X[n][k] * bf16(W_hat[m][k]), fp32 accumulation, the same
// definition as chunk.cu (source: "Decode V2 -- resident executor", section 0
// item 1 and section 5: prompt chunks of up to 32 tokens through the
// tensor-core GEMM, each weight read once per chunk).  This kernel is the one
// used when K is a multiple of 256 and the operands are 16-byte aligned:
//
//  * work units are (128-row tile, 256-column slice) pairs, tile-major; each of
//    min(units, 152) persistent blocks takes one contiguous, equal share of them
//    (stream-K), so every SM streams the same number of bytes; a block whose
//    last tile continues in the next block processes that tile's units first;
//  * two producer warps load each unit with 2-D TMA copies into two rings: one
//    the codes (128 rows x 128 bytes, 128-byte swizzled so the dequantizing
//    threads read them without bank conflicts) and the 128 x 4 fp32 scales into
//    a ring of code stages that the dequantizing warps release as soon as they
//    hold their bytes in registers; the other the four 64-column slices of
//    X (32 rows, rows >= N zero-filled by the copy, already in the swizzled
//    K-major layout the tensor core reads) into a ring of X stages that the
//    MMA commit releases.  Code stages thus never wait for the tensor core, and
//    the code ring runs several units ahead of the dequantization;
//  * eight dequantizing warps turn each 64-column k-tile of codes into the bf16
//    A operand (fp32 level x fp32 scale from the lane-replicated pair table,
//    rounded once) and store it straight into tensor memory (tcgen05.st; row m
//    in TMEM lane m), a ring of three stages of four k-tiles: the A operand never passes
//    through shared memory, which the pair-table reads alone keep busy;
//  * two issuer warps (one thread each) issue tcgen05.mma (M = 128, N = 32,
//    K = 16, A from TMEM, X from shared memory) into one of two TMEM
//    accumulator buffers, so four epilogue warps can drain one tile while the
//    next accumulates; within a tile the units alternate between the issuers,
//    each accumulating into its own 32-column chain of the buffer, and the
//    epilogue adds the two chains;
//  * a tile whose K range is split over several blocks is finished by the last of
//    them to arrive (a per-tile ticket), which adds the partial tiles in block
//    order: the result does not depend on timing.  The last of two that finds
//    the other's partial already published does not publish its own.
// Every wait is bounded; on a timeout the block stops issuing work, waits for its
// copies and tensor-core operations, frees its TMEM and reports the error word.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <mutex>
#include <string>

#include "gemv_kernel.cuh"

namespace nf4k {

namespace {

constexpr int TM = 128;        // MMA M: rows of W per tile
constexpr int TN = 32;         // MMA N: tokens
constexpr int KT = 64;         // columns per k-tile (one NF4 block, one swizzle atom of bf16)
constexpr int KQ = 4;          // k-tiles per unit (256 columns, 128 code bytes per row)
constexpr int NDQ = 8;        // dequantizing warps
constexpr int CPW = 16 / NDQ;  // column groups per dequantizing warp
constexpr int EPI_WARPS = 4;   // warps 0-3: epilogue (TMEM lanes 32w .. 32w + 31)
constexpr int PROD_WARP = 4;
constexpr int MMA_WARP = 5;
constexpr int DQ_WARP0 = 6;
constexpr int XPROD_WARP = DQ_WARP0 + NDQ;       // 14: the X-ring producer
constexpr int MMA2_WARP = XPROD_WARP + 1;        // 15: the second MMA issuer
constexpr int NTHREADS = (MMA2_WARP + 1) * 32;   // 512
#ifndef NF4_CHUNK_SC
#define NF4_CHUNK_SC 3
#endif
#ifndef NF4_CHUNK_SX
#define NF4_CHUNK_SX 6
#endif
#ifndef NF4_CHUNK_SA
#define NF4_CHUNK_SA 3
#endif
#ifndef NF4_DQ_SLEEP
#define NF4_DQ_SLEEP 0
#endif
constexpr int SC = NF4_CHUNK_SC;  // code stages (codes + scales of a unit) in shared memory
constexpr int SX = NF4_CHUNK_SX;  // X stages (the unit's four X slices) in shared memory
constexpr int SA = NF4_CHUNK_SA;  // A stages in tensor memory, KS k-tiles each
// k-tiles per A stage: one barrier wait, KS x 4 MMAs and one commit per stage.
// Measured alone, a wait + fence costs about 190 cycles and a commit 44
// against 45 per M=128 N=32 K=16 MMA, so one handshake per k-tile would cost
// more than the k-tile's tensor-core work.
#ifndef NF4_CHUNK_KS
#define NF4_CHUNK_KS 4
#endif
constexpr int KS = NF4_CHUNK_KS;
static_assert(KQ % KS == 0, "A stages tile a unit");
constexpr int CODES_BYTES = TM * KQ * KT / 2;    // 16 KB
constexpr int XT_BYTES = TN * KT * 2;            // 4 KB per k-tile
constexpr int SCL_BYTES = TM * KQ * 4;           // 2 KB
constexpr int CST_BYTES = CODES_BYTES + SCL_BYTES;  // 18 KB code stage
constexpr int XST_BYTES = KQ * XT_BYTES;            // 16 KB X stage
constexpr int SMEM_BYTES = LUT_BYTES + SC * CST_BYTES + SX * XST_BYTES;
static_assert(SMEM_BYTES + 1024 <= 232448, "shared memory per block");
// TMEM columns: two 32-column fp32 accumulators, then SA A stages of KS x 32
// columns (64 bf16 of each row per k-tile, two per 32-bit column)
constexpr int A_COLS = KS * KT / 2;
// Accumulators: two buffers (one tile accumulates while the epilogue drains
// the other) of CH = 2 chains, one per MMA issuer warp: columns
// (buf * CH + issuer) * TN.
constexpr int CH = 2;
constexpr int A_COL0 = 2 * CH * TN;
constexpr int TMEM_COLS = (A_COL0 + SA * A_COLS) <= 256 ? 256 : 512;  // a power of two; one block per SM
static_assert(A_COL0 + SA * A_COLS <= TMEM_COLS, "tensor memory per block");
constexpr int PLAN_SMS = 152;  // blocks planned for a 152-SM GB300 (the workspace depends on the shape only)

static_assert(CST_BYTES % 1024 == 0 && XST_BYTES % 1024 == 0, "stages must keep 1024-byte alignment");
static_assert(NDQ == 8 || NDQ == 16, "dequantizing warps: whole lane quarters");

struct StreamKArgs {
  float* Y;
  float* partial;         // [tiles][maxseg][N][128]
  unsigned int* tickets;  // [tiles]
  int M, K, N;
  int tiles, NQ;          // row tiles, units per tile (K / 256)
  long long U;            // units = tiles * NQ
  int B;                  // blocks
  int maxseg;             // partial slots per tile (0: whole tiles per block)
  uint32_t wait_polls;    // limit of the pipeline waits (free stages, staged codes, dequantized operands)
};

// First unit of block b: an equal share of the units, or, when there are at
// least four tiles per block, an equal share of whole tiles (no tile is split,
// no partials).
__host__ __device__ inline long long unit_start(long long b, const StreamKArgs& a) {
  return a.maxseg == 0 ? (b * a.tiles / a.B) * a.NQ : b * a.U / a.B;
}

// the block whose unit range holds unit u
__host__ __device__ inline int block_of(long long u, const StreamKArgs& a) {
  long long b = u * a.B / a.U;
  while (b + 1 < a.B && unit_start(b + 1, a) <= u) ++b;
  while (b > 0 && unit_start(b, a) > u) --b;
  return (int)b;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ uint2 lds64(const void* p) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(smem_addr(p)));
  return v;
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T, bf16 inputs, fp32 accumulate; A is
// M rows in TMEM lanes, each row's K values packed two per 32-bit column.
// The B descriptor comes as its two 32-bit halves: the issuer precomputes the
// high half (layout constants) and the low half of a stage's first k-step,
// so each MMA of a stage costs one 32-bit add (the start-address field, bits
// 0-13, never carries: shared addresses are below 256 KB).
__device__ __forceinline__ void tc_mma_bf16_ta2(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 bd;\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "mov.b64 bd, {%2, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], bd, %4, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Warp-wide store of 8 consecutive 32-bit columns into this warp's 32 TMEM
// lanes (lane l of the warp writes TMEM lane base + l).
__device__ __forceinline__ void tmem_st_32x32b_x8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}
__device__ __forceinline__ void mul2_f32(float& r0, float& r1, float a0, float a1, float b) {
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %4};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(r0), "=f"(r1)
      : "f"(a0), "f"(a1), "f"(b));
}

// Bounded wait that sleeps `ns` nanoseconds between polls (waits that are long
// by design leave the barrier unit to the threads on the critical path).
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity, volatile int* abort, uint32_t ns,
                                                uint32_t polls = kWaitPolls) {
  for (uint32_t i = 0; i < polls; ++i) {
    if (polls == kWaitPolls ? mbar_try_wait(bar, parity) : mbar_test_wait(bar, parity)) return true;
    if (*abort) return false;
    if (ns) __nanosleep(ns);
  }
  *abort = 1;
  atomicOr(&g_nf4_device_error, kErrWaitTimeout);
  return false;
}

// Warp-wide wait: lane 0 polls, the other lanes wait at the warp barrier, which
// orders their later accesses after the phase lane 0 observed (one poller per
// warp instead of 32).
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, volatile int* abort, int lane,
                                               uint32_t ns, uint32_t polls = kWaitPolls) {
  int ok = 1;
  if (lane == 0) ok = mbar_wait_sleep(bar, parity, abort, ns, polls) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

// Warp-wide load of 16 consecutive fp32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// Release and acquire at GPU scope (orders this thread's, and by cumulativity
// the CTA-barrier-ordered, memory operations around a ticket atomic).
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// Load with acquire semantics at GPU scope (a ticket read before the partials
// it guards).
__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__global__ void __launch_bounds__(NTHREADS, 1)
    chunk_tma_kernel(const __grid_constant__ CUtensorMap tm_codes, const __grid_constant__ CUtensorMap tm_scales,
                     const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ StreamKArgs a,
                     const __grid_constant__ Codebook cbk) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ float cbs[16];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ unsigned int s_last;
  __shared__ unsigned long long s_bar[2 * SC + 2 * SX + 2 * SA + 4 + 1];

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const long long u0 = unit_start(blockIdx.x, a);
  const long long u1 = unit_start(blockIdx.x + 1, a);
  const int nq = (int)(u1 - u0);
  // Processing order.  When the block's last tile continues in the next
  // block, this block takes that tile's units (its head) first, so their
  // partial is published early and the next block, which reaches the rest of
  // that tile at its own end, finds it published and needs not publish its
  // own.  All roles walk the units in this order: the q-th unit processed is
  // slice kq_of(q) of tile tile_of(q), and seg_end(q) ends the run of units
  // of the same tile that holds q (32-bit arithmetic per unit).
  const int tB = nq > 0 ? (int)((u1 - 1) / a.NQ) : 0;
  const long long uB = (long long)tB * a.NQ;
  const int nh = (a.maxseg != 0 && uB > u0 && (u1 % a.NQ) != 0) ? (int)(u1 - uB) : 0;
  const int t0 = (int)(u0 / a.NQ), r0 = (int)(u0 % a.NQ);
  auto kq_of = [&](int q) -> int { return q < nh ? q : (r0 + q - nh) % a.NQ; };
  auto tile_of = [&](int q) -> int { return q < nh ? tB : t0 + (r0 + q - nh) / a.NQ; };
  auto seg_end = [&](int q) -> int {
    if (q < nh) return nh;
    const int e = q + a.NQ - (r0 + q - nh) % a.NQ;
    return e < nq ? e : nq;
  };

  uint8_t* cst0 = smem + LUT_BYTES;         // SC code stages: codes, then scales
  uint8_t* xst0 = cst0 + SC * CST_BYTES;     // SX X stages
  const uint32_t bar0 = smem_addr(&s_bar[0]);
  constexpr int B_CE = SC, B_XF = 2 * SC, B_XE = 2 * SC + SX, B_AF = 2 * SC + 2 * SX, B_AE = B_AF + SA,
                B_ACC = B_AE + SA;
  auto c_full = [&](int s) { return bar0 + 8u * (uint32_t)s; };
  auto c_empty = [&](int s) { return bar0 + 8u * (uint32_t)(B_CE + s); };
  auto x_full = [&](int s) { return bar0 + 8u * (uint32_t)(B_XF + s); };
  auto x_empty = [&](int s) { return bar0 + 8u * (uint32_t)(B_XE + s); };
  auto a_full = [&](int s) { return bar0 + 8u * (uint32_t)(B_AF + s); };
  auto a_empty = [&](int s) { return bar0 + 8u * (uint32_t)(B_AE + s); };
  auto acc_full = [&](int b) { return bar0 + 8u * (uint32_t)(B_ACC + b); };
  auto acc_empty = [&](int b) { return bar0 + 8u * (uint32_t)(B_ACC + 2 + b); };
  const uint32_t mma_done = bar0 + 8u * (uint32_t)(B_ACC + 4);

  if (tid == 0) {
    for (int s = 0; s < SC; ++s) {
      mbar_init(c_full(s), 1);
      mbar_init(c_empty(s), NDQ);  // the dequantizing warps, once their codes are in registers
    }
    for (int s = 0; s < SX; ++s) {
      mbar_init(x_full(s), 1);
      mbar_init(x_empty(s), 1);  // the MMA commit of the unit
    }
    for (int s = 0; s < SA; ++s) {
      mbar_init(a_full(s), NDQ);
      mbar_init(a_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full(b), 2);  // one commit per MMA issuer
      mbar_init(acc_empty(b), EPI_WARPS);
    }
    mbar_init(mma_done, 2);
    mbar_init_fence();
    s_abort = 0;
  }
  if (tid < 16) cbs[tid] = cbk.v[tid];
  pdl_launch_dependents();  // the next kernel may start its prologue on SMs this grid has left
  if (warp == MMA_WARP) {
    tmem_alloc(smem_addr(&s_tmem), TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == PROD_WARP && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_codes) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_scales) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_x) : "memory");
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = s_tmem;

  // producers: a unit is the codes and scales of a 128-row x 256-column slice
  // (code ring) and the four 64-column slices of X it multiplies (X ring),
  // each completing on its stage's full barrier
  auto issue_codes = [&](int q) {
    const int s = q % SC;
    const int tile = tile_of(q), kq = kq_of(q);
    uint8_t* st = cst0 + s * CST_BYTES;
    mbar_arrive_expect_tx(c_full(s), CST_BYTES);
    tma_load_2d(smem_addr(st), &tm_codes, kq * 128, tile * TM, c_full(s));
    tma_load_2d(smem_addr(st + CODES_BYTES), &tm_scales, kq * KQ, tile * TM, c_full(s));
  };
  auto issue_x = [&](int q) {
    const int s = q % SX;
    const int kq = kq_of(q);
    uint8_t* st = xst0 + s * XST_BYTES;
    mbar_arrive_expect_tx(x_full(s), XST_BYTES);
#pragma unroll
    for (int i = 0; i < KQ; ++i) tma_load_2d(smem_addr(st + i * XT_BYTES), &tm_x, (kq * KQ + i) * KT, 0, x_full(s));
  };
  // the first code stages go out before the pair table is built, so the
  // table build hides under their latency
  const bool aligned1k = (smem_addr(cst0) & 1023u) == 0;
  const int pre_c = aligned1k ? (nq < SC ? nq : SC) : 0;
  if (warp == PROD_WARP && lane == 0)
    for (int q = 0; q < pre_c; ++q) issue_codes(q);
  // (X is the previous kernel's output: its first slices go out after the
  // dependency wait, in the X producer's loop below)
  // pair table: byte b, lane l -> (cb[b & 15], cb[b >> 4]) at b * 256 + l * 8
  for (int i = tid; i < LUT_BYTES / 8; i += NTHREADS) {
    const int b = i >> 5;
    reinterpret_cast<float2*>(smem)[i] = make_float2(cbs[b & 15], cbs[b >> 4]);
  }
  if (tid == 0 && !aligned1k) {  // swizzled tiles need 1024-byte alignment
    s_abort = 1;
    atomicOr(&g_nf4_device_error, kErrWaitTimeout);
  }
  __syncthreads();
  volatile int* abort = &s_abort;

  if (warp == PROD_WARP || warp == XPROD_WARP) {
    // ------------------------------------------------------------ producers
    // lane 0 of one warp fills the code ring, lane 0 of the other the X ring,
    // each waiting only for its own ring's stages to be released
    if (lane == 0) {
      const bool codes_lane = warp == PROD_WARP;
      const int ring = codes_lane ? SC : SX;
      // programmatic dependent launch: the weights never depend on the
      // previous kernel, X does
      if (!codes_lane) pdl_wait();
      int issued = codes_lane ? pre_c : 0;
      for (int q = issued; q < nq; ++q) {
        const int s = q % ring;
        if (q >= ring &&
            !mbar_wait_sleep(codes_lane ? c_empty(s) : x_empty(s), (uint32_t)(((q / ring) - 1) & 1), abort, 64,
                             a.wait_polls))
          break;
        if (*abort) break;
        if (codes_lane)
          issue_codes(q);
        else
          issue_x(q);
        issued = q + 1;
      }
      if (*abort) {
        // wait (bounded, ignoring the flag) for this lane's copies still in flight
        for (int q = (issued > ring ? issued - ring : 0); q < issued; ++q) {
          const uint32_t fb = codes_lane ? c_full(q % ring) : x_full(q % ring);
          for (uint32_t i = 0; i < kWaitPolls; ++i)
            if (mbar_try_wait(fb, (uint32_t)((q / ring) & 1))) break;
        }
      }
    }
    __syncwarp();
  } else if (warp == MMA_WARP || warp == MMA2_WARP) {
    // ------------------------------------------------------- MMA issuers
    // Two issuer warps: within a tile, units alternate between them (unit
    // qs + 2i + me goes to issuer me), each into its own accumulator chain, so
    // while one warp waits out an MMA issue the other issues.  The whole warp
    // runs the loop; lane 0 issues the tensor-core operations.
    {
      const int me = warp == MMA_WARP ? 0 : 1;
      const uint32_t idesc = idesc_bf16_f32(TM, TN);
      int g = 0;
      for (int q = 0; q < nq;) {
        const int qs = q;
        const int qe = seg_end(q);
        const int buf = g & 1;
        if (g >= 2) mbar_wait_warp(acc_empty(buf), (uint32_t)(((g >> 1) - 1) & 1), abort, lane, 0);
        tc_fence_after_sync();
        const uint32_t dtm = tmem + (uint32_t)((buf * CH + me) * TN);
        bool first = true;  // this issuer's first k-step of the tile starts its chain at 0
        for (q = qs + me; q < qe; q += CH) {
          const int s = q % SX;
          mbar_wait_warp(x_full(s), (uint32_t)((q / SX) & 1), abort, lane, 0);
          const uint32_t xb = smem_addr(xst0 + s * XST_BYTES);
#pragma unroll 1
          for (int h = 0; h < KQ / KS; ++h) {
            const int j = q * (KQ / KS) + h;  // A stages are filled in unit order
            const int as = j % SA;
            mbar_wait_warp(a_full(as), (uint32_t)((j / SA) & 1), abort, lane, 0, a.wait_polls);
            tc_fence_after_sync();
            if (lane == 0) {
              if (!*abort) {
                const uint32_t at = tmem + (uint32_t)(A_COL0 + as * A_COLS);
                const uint64_t d0 = smem_desc_sw128(xb + h * KS * XT_BYTES);
                const uint32_t blo = (uint32_t)d0, bhi = (uint32_t)(d0 >> 32);
#pragma unroll
                for (int i2 = 0; i2 < KS; ++i2)
#pragma unroll
                  for (int kk = 0; kk < KT / 16; ++kk)
                    tc_mma_bf16_ta2(dtm, at + i2 * (KT / 2) + kk * 8, blo + (uint32_t)((i2 * XT_BYTES + kk * 32) >> 4),
                                    bhi, idesc, (!first || i2 > 0 || kk > 0) ? 1u : 0u);
              }
              tc_commit(a_empty(as));
            }
            first = false;
            __syncwarp();
          }
          if (lane == 0) tc_commit(x_empty(s));  // X of this unit is read once these MMAs complete
          __syncwarp();
        }
        q = qe;
        if (lane == 0) tc_commit(acc_full(buf));  // both issuers arrive once per tile
        __syncwarp();
        ++g;
      }
      // every tensor-core operation has completed before TMEM is freed
      if (lane == 0) {
        tc_commit(mma_done);  // both issuers arrive
        for (uint32_t i = 0; i < kWaitPolls; ++i)
          if (mbar_try_wait(mma_done, 0)) break;
      }
      __syncwarp();
    }
  } else if (warp >= DQ_WARP0 && warp < DQ_WARP0 + NDQ) {
    // ---------------------------------------------------- dequantization
    // A warp may reach only TMEM lanes 32 (warp % 4) .. + 31, so each thread owns
    // one tile row (its TMEM lane) and CPW 16-column groups of every k-tile
    // (the NDQ / 4 warps of a lane quarter share its four groups; eight warps
    // measured 22.00 against 22.11 us for sixteen, four 23.36).
    const int r = 32 * (warp & 3) + lane;          // tile row = TMEM lane
    const int cg0 = ((warp - DQ_WARP0) >> 2) * CPW;  // first column group
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t laneoff = (uint32_t)lane * 8u;  // pair-table replica
    int j = 0;
    for (int q = 0; q < nq; ++q) {
      const int s = q % SC;
      mbar_wait_warp(c_full(s), (uint32_t)((q / SC) & 1), abort, lane, NF4_DQ_SLEEP, a.wait_polls);
      const uint8_t* cst = cst0 + s * CST_BYTES;
      // this thread's codes (8 bytes of each k-tile) and scales, into
      // registers; then the code stage goes back to the producer at once
      const float4 sc4 = *reinterpret_cast<const float4*>(cst + CODES_BYTES + r * 16);
      const float scl[4] = {sc4.x, sc4.y, sc4.z, sc4.w};
      uint2 cw4[CPW][KQ];
#pragma unroll
      for (int c = 0; c < CPW; ++c)
#pragma unroll
        for (int i = 0; i < KQ; ++i)
          cw4[c][i] = lds64(cst + r * 128 + (((2 * i + ((cg0 + c) >> 1)) ^ (r & 7)) << 4) + ((cg0 + c) & 1) * 8);
      __syncwarp();
      if (lane == 0) mbar_arrive(c_empty(s));
#pragma unroll
      for (int h = 0; h < KQ / KS; ++h, ++j) {
        const int as = j % SA;
        // the tensor core has finished with this A stage's previous contents
        if (j >= SA) mbar_wait_warp(a_empty(as), (uint32_t)(((j / SA) - 1) & 1), abort, lane, NF4_DQ_SLEEP);
        tc_fence_after_sync();
#pragma unroll
        for (int i2 = 0; i2 < KS; ++i2) {
#pragma unroll
          for (int c = 0; c < CPW; ++c) {
            const int cg = cg0 + c;
            const int i = h * KS + i2;
            uint32_t p[8];
            const uint32_t w2[2] = {cw4[c][i].x, cw4[c][i].y};
#pragma unroll
            for (int e = 0; e < 2; ++e)
#pragma unroll
              for (int jj = 0; jj < 4; ++jj) {
                const uint32_t off = __byte_perm(w2[e], laneoff, 0x5504u | (jj << 4));
                const float2 v = *reinterpret_cast<const float2*>(smem + off);
                float w0, w1;
                mul2_f32(w0, w1, v.x, v.y, scl[i]);  // two IEEE products, as v.x * s and v.y * s
                p[4 * e + jj] = pack_bf16x2(w0, w1);
              }
            tmem_st_32x32b_x8(tmem + lane_base + (uint32_t)(A_COL0 + as * A_COLS + i2 * (KT / 2) + cg * 8), p);
          }
        }
        tmem_st_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(a_full(as));
      }
    }
  } else {
    // --------------------------------------------------------- epilogue
    const int er = warp * 32 + lane;  // tile row = TMEM lane
    pdl_wait();  // Y and the workspace are written only after the previous kernel has finished
    int g = 0;
    for (int q = 0; q < nq; ++g) {
      const long long tile = tile_of(q);
      const int qe = seg_end(q);
      const bool two = qe - q >= 2;  // the second issuer's chain holds units of this tile
      q = qe;
      const int buf = g & 1;
      // the tile's segment count and this block's place among them (the
      // block_of searches) are worked out while the accumulators fill, not
      // after: on a block's last tile they would delay its end
      const long long m = tile * TM + er;
      const int bf = a.maxseg == 0 ? (int)blockIdx.x : block_of(tile * a.NQ, a);
      const int nseg = a.maxseg == 0 ? 1 : block_of(tile * a.NQ + a.NQ - 1, a) - bf + 1;
      const int si = (int)blockIdx.x - bf;
      const bool ok = mbar_wait_warp(acc_full(buf), (uint32_t)((g >> 1) & 1), abort, lane, 128);
      tc_fence_after_sync();
      uint32_t acc[32];
      tmem_ld_32x32b_x32(tmem + (uint32_t)(buf * CH * TN) + ((uint32_t)(warp * 32) << 16), acc);
      if (two) {  // the two issuers' chains, added once (the second in halves)
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t acc1[16];
          tmem_ld_32x32b_x16(tmem + (uint32_t)((buf * CH + 1) * TN + 16 * half) + ((uint32_t)(warp * 32) << 16), acc1);
          tmem_ld_wait();
#pragma unroll
          for (int n = 0; n < 16; ++n)
            acc[16 * half + n] = __float_as_uint(__uint_as_float(acc[16 * half + n]) + __uint_as_float(acc1[n]));
        }
      }
      tmem_ld_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty(buf));
      if (nseg == 1) {
        if (ok && !*abort && m < a.M) {
#pragma unroll
          for (int n = 0; n < TN; ++n)
            if (n < a.N) a.Y[(long long)n * a.M + m] = __uint_as_float(acc[n]);
        }
        continue;
      }
      // partial tile: the last of the tile's blocks to arrive adds all of them in block order
      // A tile of two segments whose other partial is already published
      // (ticket = 1, read with acquire by thread 0; the barrier orders that
      // read before every thread's loads of the partial): this block is the
      // last and finishes the tile without publishing its own (s_last = 2).
      if (tid == 0) s_last = (nseg == 2 && ld_acquire_gpu(a.tickets + tile) == 1u) ? 2u : 0u;
      named_bar_sync(1, EPI_WARPS * 32);
      if (s_last == 0u) {
        float* slot = a.partial + ((long long)tile * a.maxseg + si) * a.N * TM;
        if (ok && !*abort) {
#pragma unroll
          for (int n = 0; n < TN; ++n)
            if (n < a.N) slot[n * TM + er] = __uint_as_float(acc[n]);
        }
        // Publish the partial: the barrier orders every epilogue thread's
        // stores before thread 0, whose release fence (cumulative) then
        // precedes its ticket; the last arriver's acquire fence follows its
        // ticket, and the barrier orders it before every thread's loads of
        // the other partials.
        named_bar_sync(1, EPI_WARPS * 32);
        if (tid == 0) {
          fence_acq_rel_gpu();
          const unsigned int prev = atomicAdd(&a.tickets[tile], 1u);
          s_last = (prev == (unsigned int)nseg - 1) ? 1u : 0u;
          if (s_last) fence_acq_rel_gpu();
        }
        named_bar_sync(1, EPI_WARPS * 32);
      }
      if (s_last) {
        // all of a slot's values are loaded before any store (32 independent
        // loads per slot, not one round trip per value); slots added in order
        const float* base = a.partial + (long long)tile * a.maxseg * a.N * TM;
        float sum[TN];
        if (nseg == 2) {
          // the usual split: this block's own partial is still in registers,
          // so one slot is loaded; added in block order from 0 as below
          float v[TN];
#pragma unroll
          for (int n = 0; n < TN; ++n) v[n] = n < a.N ? __ldcg(base + ((long long)(1 - si) * a.N + n) * TM + er) : 0.f;
#pragma unroll
          for (int n = 0; n < TN; ++n)
            sum[n] = si == 0 ? (0.f + __uint_as_float(acc[n])) + v[n] : (0.f + v[n]) + __uint_as_float(acc[n]);
        } else {
#pragma unroll
          for (int n = 0; n < TN; ++n) sum[n] = 0.f;
          for (int k = 0; k < nseg; ++k) {
            float v[TN];
#pragma unroll
            for (int n = 0; n < TN; ++n) v[n] = n < a.N ? __ldcg(base + ((long long)k * a.N + n) * TM + er) : 0.f;
#pragma unroll
            for (int n = 0; n < TN; ++n) sum[n] += v[n];
          }
        }
        if (!*abort && m < a.M) {
#pragma unroll
          for (int n = 0; n < TN; ++n)
            if (n < a.N) a.Y[(long long)n * a.M + m] = sum[n];
        }
        if (tid == 0) a.tickets[tile] = 0u;  // leave the workspace zeroed
      }
      named_bar_sync(1, EPI_WARPS * 32);  // s_last is read before the next tile rewrites it
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

using EncodeTiled = PFN_cuTensorMapEncodeTiled_v12000;

EncodeTiled encode_fn() {
  static std::once_flag once;
  static EncodeTiled fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
    cudaGetLastError();
  });
  return fn;
}

struct Plan {
  int tiles, NQ, B, maxseg;
  long long U;
};

Plan plan_for(int64_t M, int64_t K) {
  Plan p{};
  p.tiles = (int)((M + TM - 1) / TM);
  p.NQ = (int)(K / (KT * KQ));
  p.U = (long long)p.tiles * p.NQ;
  p.B = (int)(p.U < PLAN_SMS ? p.U : PLAN_SMS);
  if (p.B < 1) p.B = 1;
  if (p.tiles >= 4 * p.B) {  // whole tiles per block: at most 1 tile in 4 of imbalance
    p.maxseg = 0;
    return p;
  }
  const long long min_units = p.U / p.B;  // >= 1
  long long ms = (p.NQ + min_units - 1) / min_units + 1;
  p.maxseg = (int)(ms < p.B ? ms : p.B);
  return p;
}

}  // namespace

bool chunk_tma_usable(int64_t K, const void* codes, const void* scales, const void* X) {
  auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  return K % (KT * KQ) == 0 && a16(codes) && a16(scales) && a16(X) && encode_fn() != nullptr;
}

// Bytes of the split-tile partials (tickets are placed by the caller).
size_t chunk_tma_partial_bytes(int64_t M, int64_t K, int N) {
  if (K % (KT * KQ) != 0) return 0;
  const Plan p = plan_for(M, K);
  return (size_t)p.tiles * (size_t)p.maxseg * N * TM * sizeof(float);
}

cudaError_t launch_chunk_tma(const uint8_t* codes, const float* scales, int M, int K, const uint16_t* X, int N,
                             float* Y, float* partial, unsigned int* tickets, const Codebook& cb, cudaStream_t s) {
  EncodeTiled enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const Plan p = plan_for(M, K);
  CUtensorMap mc, ms, mx;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)K / 2, (cuuint64_t)M};
    const cuuint64_t strides[1] = {(cuuint64_t)K / 2};
    const cuuint32_t box[2] = {128, TM};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&mc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(codes), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)K / 64, (cuuint64_t)M};
    const cuuint64_t strides[1] = {(cuuint64_t)K / 64 * 4};
    const cuuint32_t box[2] = {KQ, TM};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&ms, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(scales), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)N};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {KT, TN};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(X), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  StreamKArgs a{};
  a.Y = Y;
  a.partial = partial;
  a.tickets = tickets;
  a.M = M;
  a.K = K;
  a.N = N;
  a.tiles = p.tiles;
  a.NQ = p.NQ;
  a.U = p.U;
  a.B = p.B;
  a.maxseg = p.maxseg;
  a.wait_polls = data_wait_polls();
  return checked_launch(reinterpret_cast<const void*>(&chunk_tma_kernel), NTHREADS, SMEM_BYTES, [&] {
    // programmatic dependent launch: blocks may start (TMEM, barriers, pair
    // table, the first code stages) while the previous kernel finishes
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)p.B);
    cfg.blockDim = dim3((unsigned)NTHREADS);
    cfg.dynamicSmemBytes = (size_t)SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    cudaLaunchKernelEx(&cfg, chunk_tma_kernel, mc, ms, mx, a, cb);
  });
}

std::string describe_chunk_tma(int64_t M, int64_t K, int N) {
  const Plan p = plan_for(M, K);
  char buf[448];
  std::snprintf(buf, sizeof buf,
                "chunk M=%lld K=%lld N=%d: tcgen05 M=%d N=%d K=16, %s over %lld units of 128 rows x 256 "
                "columns on %d persistent blocks (%d threads: %d dequantizing warps, 2 TMA producers, 2 MMA issuers, 4 "
                "epilogue warps), %d code + %d X + %d operand stages, 2 TMEM accumulator buffers of 2 chains, %s",
                (long long)M, (long long)K, N, TM, TN, p.maxseg == 0 ? "whole tiles per block" : "stream-K", p.U, p.B,
                NTHREADS, NDQ, SC, SX, SA, pdl_enabled() ? "programmatic dependent launch" : "plain launch");
  return buf;
}

}  // namespace nf4k
