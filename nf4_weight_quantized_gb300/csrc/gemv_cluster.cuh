// gemv_cluster.cuh -- N=1 NF4 GEMV for few rows: K split across a thread-block
// cluster, partial sums added through distributed shared memory.
//
// Same definition and epilogues as gemv_kernel.cuh (source: "Decode V2 --
// resident executor", section 6 "Linear primitive"; the page measures its
// q/k/v/o projections at 4-41 GB/s and notes that small shapes need many
// CTAs per row).  With M of a few hundred or thousand rows, one block per row
// group leaves most SMs idle and every block's work is one long latency chain.
// Here a cluster of CL blocks (CL SMs) owns a range of rows; block `rank` of
// the cluster reads only the chunks [rank * H / CL, (rank + 1) * H / CL) of
// each row (H = K / 32 chunks of 32 weights), so the bytes of a row are
// fetched by CL SMs at once.
//  * inside a block, TPR = the next power of two >= that chunk count threads
//    share a row (one chunk each, x-stationary: the thread's x chunk is in
//    registers), 32 / TPR rows per warp, a shuffle reduction per row;
//  * each block leaves its row partials in shared memory; after a cluster
//    barrier, block q of the cluster adds, for rows r with r % CL == q, the CL
//    partials in rank order (distributed shared-memory loads), then applies
//    the epilogue; a second cluster barrier keeps every block's shared memory
//    alive until all remote loads are done.  Every block executes both
//    barriers (no early exit), and nothing else waits.
//  * the weights do not depend on the previous kernel: every thread loads the
//    codes and scales of all its rows (at most NP passes) into registers
//    before the programmatic-dependent-launch wait, so after the previous
//    kernel ends only the x load (an L2 hit) and the arithmetic remain;
//  * levels come from a 16-entry shared table (one bank each, lanes reading
//    the same level share the word), so there is no per-block table build.
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"

namespace nf4k {

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// fp32 load from the shared memory of block `rank` of this cluster, at the
// address `p` has in this block's shared window
__device__ __forceinline__ float ld_dsmem_f32(const float* p, uint32_t rank) {
  uint32_t local = smem_addr(p), remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

constexpr int kClusterThreads = 512;
constexpr int kClusterPasses = 4;  // NP: rows per cluster <= NP x rows per pass

template <int EPI, bool XBF16>
__global__ void __launch_bounds__(kClusterThreads, 1) gemv_cluster_kernel(const __grid_constant__ GemvArgs a, int CL,
                                                                        int RPC) {
  constexpr int NP = kClusterPasses;
  extern __shared__ float part[];  // [RPC] this block's partial sum per row
  __shared__ float lv[16];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rank = (int)cluster_ctarank();
  const int64_t cl = blockIdx.x / CL;
  const int64_t r0 = cl * RPC;
  const int rows = (int)((a.M - r0) < RPC ? (a.M - r0) : RPC);  // may be <= 0 for a trailing cluster
  const int H = a.K >> 5;
  const int c0 = (int)((int64_t)rank * H / CL), c1 = (int)((int64_t)(rank + 1) * H / CL);
  const int hr = c1 - c0;  // chunks of this block's K slice (<= 32)
  int TPR = 1;
  while (TPR < hr) TPR <<= 1;
  const int RPW = 32 / TPR;               // rows per warp
  const int RPP = RPW * (blockDim.x >> 5);  // rows per pass of the block
  const int sub = lane / TPR, ci = lane % TPR;
  const bool cval = ci < hr;
  const int chunk = c0 + (cval ? ci : 0);
  const int64_t row_bytes = a.K >> 1, nblk = a.K >> 6;

  if (tid < 16) lv[tid] = a.cb.v[tid];
  // codes and scales of this thread's rows, all passes, before the wait
  uint4 cbuf[NP];
  float sbuf[NP];
#pragma unroll
  for (int p = 0; p < NP; ++p) {
    const int lr = p * RPP + warp * RPW + sub;
    cbuf[p] = make_uint4(0x77777777u, 0x77777777u, 0x77777777u, 0x77777777u);
    sbuf[p] = 0.f;
    if (cval && lr < rows) {
      const int64_t row = r0 + lr;
      const uint8_t* cp = a.codes;
      const float* sp = a.scales;
      int64_t mr = row;
      if (EPI == EPI_QKV) {
        const int sg = qkv_seg(a, row);
        mr = row - qkv_first(a, sg);
        cp = qkv_pick(sg, a.seg_codes[0], a.seg_codes[1], a.seg_codes[2]);
        sp = qkv_pick(sg, a.seg_scales[0], a.seg_scales[1], a.seg_scales[2]);
      }
      cbuf[p] = ld_stream_v4(cp + mr * row_bytes + (int64_t)chunk * 16);
      sbuf[p] = ld_nc_f32(sp + mr * nblk + (chunk >> 1));
    }
  }
  pdl_launch_dependents();
  pdl_wait();  // x (and the residual) come from the previous kernel
  // this thread's x chunk, widened exactly to fp32
  float xv[32];
  if (cval) {
    if (XBF16) {
      const uint8_t* xp = reinterpret_cast<const uint8_t*>(a.x) + (int64_t)chunk * 64;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 u = ld_nc_v4(xp + 16 * q);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          xv[8 * q + 2 * e] = bf16lo_to_f32(w[e]);
          xv[8 * q + 2 * e + 1] = bf16hi_to_f32(w[e]);
        }
      }
    } else {
      const uint8_t* xp = reinterpret_cast<const uint8_t*>(a.x) + (int64_t)chunk * 128;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint4 u = ld_nc_v4(xp + 16 * q);
        xv[4 * q + 0] = __uint_as_float(u.x);
        xv[4 * q + 1] = __uint_as_float(u.y);
        xv[4 * q + 2] = __uint_as_float(u.z);
        xv[4 * q + 3] = __uint_as_float(u.w);
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < 32; ++e) xv[e] = 0.f;
  }
  __syncthreads();  // level table

  // partial sums of this block's K slice, RPP rows per pass
#pragma unroll
  for (int p = 0; p < NP; ++p) {
    const int lr = p * RPP + warp * RPW + sub;  // row within the cluster's range
    float acc = 0.f;
    if (cval && lr < rows) {
      const uint4 c = cbuf[p];
      const float s = sbuf[p];
      const uint32_t w[4] = {c.x, c.y, c.z, c.w};
      float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int b = 0; b < 8; ++b) d[j] = fmaf(lv[(w[j] >> (4 * b)) & 15u], xv[8 * j + b], d[j]);
      acc = ((d[0] + d[1]) + (d[2] + d[3])) * s;
    }
    // sum over the TPR lanes of the row (fixed butterfly order)
    for (int off = TPR >> 1; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (ci == 0 && lr < rows) part[lr] = acc;
  }

  cluster_sync_all();  // every block's partials are written
  for (int lr = rank + CL * tid; lr < rows; lr += CL * (int)blockDim.x) {
    float v = 0.f;
    for (int q = 0; q < CL; ++q) v += ld_dsmem_f32(&part[lr], (uint32_t)q);  // rank order
    const int64_t row = r0 + lr;
    if (EPI == EPI_PLAIN) {
      a.y[row] = v;
    } else if (EPI == EPI_RESID) {
      a.y[row] = v + a.resid[row];
    } else if (EPI == EPI_QKV) {
      qkv_store(a, row, v);
    }
  }
  cluster_sync_all();  // no block leaves while its shared memory may still be read
}

}  // namespace nf4k
