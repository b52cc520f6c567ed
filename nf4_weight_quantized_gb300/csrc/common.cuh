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

// ---- shared-memory barriers and bulk copies (sm_90+ async proxy) ----------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make initialized barriers visible to the async proxy (bulk copies, MMA).
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of one barrier phase (never suspends the thread).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Upper bound on polls of one barrier phase (each poll may itself block for a
// short hardware-defined time); past it the kernel gives up (see WaitGuard).
constexpr uint32_t kWaitPolls = 1u << 22;

// Error word set by kernels whose bounded waits ran out (0 = none).  Device
// code is compiled per translation unit (no relocatable device linking), so
// every unit that includes this header has its own word; a static initializer
// registers the unit's reader with the library (nf4_check_device_errors).
static __device__ unsigned int g_nf4_device_error;
constexpr unsigned int kErrWaitTimeout = 1u;
constexpr unsigned int kErrBadIndex = 2u;  // a token id outside its table (nf4_dequant_rows)

using DeviceErrorReader = unsigned int (*)();
void register_device_error_reader(DeviceErrorReader f);  // abi.cu

namespace {
// Reads and clears this unit's error word on the current device (synchronous).
unsigned int read_and_clear_device_error() {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_nf4_device_error, sizeof v) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (v) {
    const unsigned int z = 0;
    cudaMemcpyToSymbol(g_nf4_device_error, &z, sizeof z);
  }
  return v;
}
struct DeviceErrorRegistration {
  DeviceErrorRegistration() { register_device_error_reader(&read_and_clear_device_error); }
};
const DeviceErrorRegistration g_device_error_registration;
}  // namespace

// Bounded wait on one barrier phase.  `abort` is a block-shared flag: once any
// wait in the block has timed out, later waits return at once, so the block
// runs to its end (keeping every block-level barrier matched) without hanging.
// `polls` is the limit (kWaitPolls unless a failure-detection test shortened
// the waits for data to arrive, see data_wait_polls; a shortened wait polls
// without suspending, so its limit is a count of tests, not of time slices).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort,
                                                  uint32_t polls = kWaitPolls) {
  for (uint32_t i = 0; i < polls; ++i) {
    if (polls == kWaitPolls ? mbar_try_wait(bar, parity) : mbar_test_wait(bar, parity)) return true;
    if (*abort) return false;
  }
  *abort = 1;
  atomicOr(&g_nf4_device_error, kErrWaitTimeout);
  return false;
}

// 1-D bulk copy global -> shared, completing `bytes` on the barrier's tx count.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// L2 policy for data read exactly once (weights): evict first.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---- programmatic dependent launch ----------------------------------------
// A kernel launched with programmatic stream serialization may start while
// the previous kernel on the stream is still running.  It must not touch
// global memory that kernel writes (or reads, for its own outputs) before
// pdl_wait(), which returns once the previous grid has completed and its
// writes are visible; without a programmatic dependency it returns at once.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Bring global data into L2 without touching shared memory.  Safe before
// pdl_wait(): L2 is the point of coherence, so later reads still see writes
// the previous kernel makes after the prefetch.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Host: programmatic dependent launch for the streaming kernels (NF4_PDL=0
// turns it off).
bool pdl_enabled();

// Host: poll limit of the pipeline waits between producers and consumers (a
// producer's wait for a free stage, a consumer's wait for staged weights or
// dequantized operands): kWaitPolls unless nf4_debug_set_wait_limit set
// another.  Waits that drain copies or tensor-core work already in flight
// always keep kWaitPolls.
uint32_t data_wait_polls();

__device__ __forceinline__ uint4 lds128(const void* p) {
  return *reinterpret_cast<const uint4*>(p);
}

// d0 += a0 * b0, d1 += a1 * b1 with one packed fp32x2 FMA (sm_100+).
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%0, %1};\n\t"
      "fma.rn.f32x2 rc, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rc;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// ---- tcgen05 (5th-generation tensor cores, TMEM accumulators) -------------

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy reads (tensor-core operand fetch) that another thread triggers.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Whole-warp TMEM allocation of `ncols` columns (power of two >= 32); the
// base address is written to shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the barrier when all previously issued tcgen05 ops of this
// thread have completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// Warp-wide load of 32 consecutive fp32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor for a K-major operand in the 128-byte
// swizzled layout: 8-row groups of 128-byte rows (1024 B apart), 16-byte
// chunks XOR-swizzled by (row % 8).  Fields: start address >> 4 (bits 0-13),
// leading-dimension offset >> 4 (16-29, unused for this layout), stride
// offset >> 4 (32-45), descriptor version 1 (46-47), layout type 2 =
// SWIZZLE_128B (61-63).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B bf16
// (bits 7-9 = 1, 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 in bits
// 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Two fp32 -> packed bf16x2 (round to nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Raise a kernel's dynamic shared-memory limit to `bytes` if it is lower
// (host; once per function and size, thread-safe).
cudaError_t ensure_smem_limit(const void* fn, int bytes);

// Launch helper used by every kernel wrapper: raises the shared-memory limit,
// launches, and on failure records what failed (attribute or launch, the
// function's attributes) for the caller's error message, then re-applies the
// limit and retries the launch once.
template <typename Launch>
cudaError_t checked_launch(const void* fn, int threads, int smem, Launch&& launch);
void note_launch_failure(const void* fn, int threads, int smem, cudaError_t set_err, cudaError_t launch_err,
                         cudaError_t retry_err);
std::string take_launch_note();
void note_stale_error(const void* fn, cudaError_t stale);  // NF4_DEBUG_LAUNCH=1 prints it

template <typename Launch>
cudaError_t checked_launch(const void* fn, int threads, int smem, Launch&& launch) {
  const cudaError_t stale = cudaGetLastError();  // launch errors below are this launch's own
  if (stale != cudaSuccess) note_stale_error(fn, stale);
  const cudaError_t set_err = ensure_smem_limit(fn, smem);
  cudaError_t e = set_err;
  if (e == cudaSuccess) {
    launch();
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) return e;
  // re-apply the limit unconditionally and retry once
  cudaError_t retry = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (retry == cudaSuccess) {
    launch();
    retry = cudaGetLastError();
  } else {
    cudaGetLastError();
  }
  note_launch_failure(fn, threads, smem, set_err, e, retry);
  return retry;
}

// Arrive on a named barrier without waiting (count threads take part).
__device__ __forceinline__ void named_bar_arrive(int id, int count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier over `count` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Epilogue kinds of the N=1 kernel.  EPI_GLU: one matrix whose rows alternate
// gate and up (row 2c the gate, row 2c + 1 the up of output c), SwiGLU of
// each pair.
enum Epi : int { EPI_PLAIN = 0, EPI_RESID = 1, EPI_SWIGLU = 2, EPI_ARGMAX = 3, EPI_QKV = 4, EPI_GLU = 5 };

// First row of part p of n equal parts of M rows.  With interleaved gate/up
// rows the split falls on even rows, so that an output's two rows stay in one
// part (every kernel variant also keeps an even number of rows per group).
template <int EPI>
__host__ __device__ __forceinline__ int64_t part_first_row(int64_t p, int64_t n, int64_t M) {
  return EPI == EPI_GLU ? 2 * (p * (M >> 1) / n) : p * M / n;
}

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
  uint32_t wait_polls;  // limit of the pipeline waits between producer and consumers (data_wait_polls)
  Codebook cb;
  // fused q/k/v (EPI_QKV): one row space over three matrices sharing x; rows
  // [0, seg_end[0]) are matrix 0's, [seg_end[0], seg_end[1]) matrix 1's,
  // [seg_end[1], seg_end[2]) matrix 2's.  Bias pointers may be null.
  const uint8_t* seg_codes[3];
  const float* seg_scales[3];
  const float* seg_bias[3];
  float* seg_out[3];
  int seg_end[3];
};

// Segment of a row of the fused q/k/v row space, its first row, and its
// members (selected without indexing the parameter arrays at run time).
__device__ __forceinline__ int qkv_seg(const GemvArgs& a, int64_t row) {
  return row < a.seg_end[0] ? 0 : (row < a.seg_end[1] ? 1 : 2);
}
__device__ __forceinline__ int64_t qkv_first(const GemvArgs& a, int s) {
  return s == 0 ? 0 : (s == 1 ? a.seg_end[0] : a.seg_end[1]);
}
__device__ __forceinline__ int64_t qkv_end(const GemvArgs& a, int s) {
  return s == 0 ? a.seg_end[0] : (s == 1 ? a.seg_end[1] : a.seg_end[2]);
}
template <typename T>
__device__ __forceinline__ T qkv_pick(int s, T v0, T v1, T v2) {
  return s == 0 ? v0 : (s == 1 ? v1 : v2);
}
// fused q/k/v epilogue: y = sum + bias, into the segment's own output
__device__ __forceinline__ void qkv_store(const GemvArgs& a, int64_t row, float v) {
  const int s = qkv_seg(a, row);
  const int64_t lr = row - qkv_first(a, s);
  const float* b = qkv_pick(s, a.seg_bias[0], a.seg_bias[1], a.seg_bias[2]);
  float* o = qkv_pick(s, a.seg_out[0], a.seg_out[1], a.seg_out[2]);
  o[lr] = b ? v + b[lr] : v;
}

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

// Bulk-copy (TMA-engine) N=1 configuration (gemv_host.cu).
struct TmaConfig {
  bool ok;       // the shape and alignment allow the bulk-copy kernel
  int nch, rb, lut, G, gpc, blocks, threads, smem;
  int SR, GPS, S, stage_bytes, codes_bytes, scales_bytes, bar_off, red_off;
  int sub;       // rows per full barrier within a group's rb rows (compiled variant)
  int subr, nb;  // rows per full barrier in the stage, full barriers per stage
};
TmaConfig choose_tma_config(int epi, bool x_bf16, int64_t M, int64_t K, int device);

// Cluster split-K kernel for few rows (gemv_cluster.cu).
struct ClusterConfig {
  bool ok;       // the epilogue and shape qualify
  int CL;        // blocks per cluster (K split)
  int RPC;       // rows per cluster
  int clusters, threads, smem;
};
ClusterConfig choose_cluster_config(int epi, int64_t M, int64_t K, int device);
cudaError_t launch_gemv_cluster(int epi, bool x_bf16, const GemvArgs& a, const ClusterConfig& c, cudaStream_t s);
cudaError_t launch_gemv_tma(int epi, bool x_bf16, const GemvArgs& a, const TmaConfig& c, cudaStream_t s);

// Host launchers (gemv.cu / quantize.cu).
cudaError_t launch_gemv(int epi, bool x_bf16, const GemvArgs& a, GemvConfig cfg, cudaStream_t s);
GemvConfig choose_gemv_config(int epi, int64_t M, int64_t K, int device);
cudaError_t launch_quantize(const float* W, int64_t M, int64_t K, uint8_t* codes, float* scales,
                            const Codebook& cb, cudaStream_t s, int device);

// RMSNorm, one block per row (rmsnorm.cu).
cudaError_t launch_rmsnorm(const float* x, const uint16_t* w, int64_t rows, int64_t K, float eps, void* y,
                           bool y_bf16, cudaStream_t s);

// Prefill chunk (chunk.cu).
cudaError_t launch_embed_rows(const uint8_t* codes, const float* scales, int64_t V, int64_t K, const int64_t* ids,
                              int64_t n, void* out, bool out_bf16, const Codebook& cb, cudaStream_t s);
cudaError_t launch_chunk(const uint8_t* codes, const float* scales, int M, int K, const uint16_t* X, int N,
                         float* Y, void* workspace, const Codebook& cb, cudaStream_t s, int device);
size_t chunk_workspace_bytes(int64_t M, int64_t K, int N);
std::string describe_chunk(int64_t M, int64_t K, int N, int device);

}  // namespace nf4k
