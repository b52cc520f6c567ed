// chunk_noalloc.cu -- nf4_gemm_chunk for callers that cannot allocate device memory.
//
// nf4_gemm_chunk needs a caller-allocated workspace for its split-K partial
// tiles and per-tile tickets.  Some callers cannot provide one: code embedded
// in a host program that owns every device allocation (a serving process with
// its own memory pool, a plugin handed only input and output pointers), or a
// real-time loop that must not call cudaMalloc because it synchronizes the
// device and can stall the whole pipeline.  For them this file keeps the
// scratch in one file-scope static device array, allocated when the module is
// loaded and held by every GPU that loads the library until the process exits.
//
// The array's host-side name is only a stand-in for the device symbol: host
// code must never hand it to a kernel.  Its device address is looked up once
// per device with cudaGetSymbolAddress (with that device current) on the first
// call made on that device; make that first call before any stream capture.
// The address is cached for the life of the process, so it goes stale if the
// device's primary context is destroyed and recreated (cudaDeviceReset): the
// entry point must not be used again in such a process.
// Every call on a device shares the one array and leaves its last contents in
// it, so calls whose kernels overlap on the GPU (other streams, other host
// threads) race on it.  The part that must start at zero (the per-tile
// tickets of the split-K fixup) is cleared by every call before its launch.
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "nf4.h"

namespace nf4k {
void set_last_error(const char* msg);  // abi.cu
}

namespace {

constexpr size_t kScratchBytes = (size_t)8 << 20;  // 8 MiB
static __device__ __align__(256) unsigned char g_chunk_scratch[kScratchBytes];

std::mutex g_mu;
void* g_addr[64];

nf4_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    nf4k::set_last_error("nf4_gemm_chunk_noalloc: no current CUDA device");
    return NF4_ECUDA;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_chunk_scratch);
    if (e != cudaSuccess || !p) {
      char buf[256];
      std::snprintf(buf, sizeof buf, "nf4_gemm_chunk_noalloc: cudaGetSymbolAddress failed: %s",
                    cudaGetErrorString(e));
      cudaGetLastError();
      nf4k::set_last_error(buf);
      return NF4_ECUDA;
    }
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return NF4_OK;
}

}  // namespace

extern "C" nf4_status nf4_gemm_chunk_noalloc(const nf4_weight* W, const uint16_t* X, int N, float* Y,
                                             nf4_stream stream) {
  // shape, pointer and alignment errors are reported exactly as nf4_gemm_chunk
  // reports them, before anything is launched
  const size_t need = W ? nf4_workspace_bytes(W->M, W->K, N) : 0;
  if (!W || need == 0 || !X || !Y || (reinterpret_cast<uintptr_t>(X) & 15) || (reinterpret_cast<uintptr_t>(Y) & 3) ||
      !W->codes || !W->scales)
    return nf4_gemm_chunk(W, X, N, Y, nullptr, stream);
  if (need > kScratchBytes) {
    char buf[256];
    std::snprintf(buf, sizeof buf,
                  "nf4_gemm_chunk_noalloc: an %lldx%lld weight at N = %d needs %zu bytes of scratch; the static "
                  "scratch holds %zu (use nf4_gemm_chunk with a caller workspace)",
                  (long long)W->M, (long long)W->K, N, need, kScratchBytes);
    nf4k::set_last_error(buf);
    return NF4_EINVAL;
  }
  void* scratch = nullptr;
  nf4_status st = scratch_address(&scratch);
  if (st) return st;
  // the tickets (one per 128-row tile) and the padding after them end the
  // workspace; they must read zero when the kernel starts
  const int64_t tiles = (W->M + 127) / 128;
  const size_t tail = need > 16 ? (size_t)tiles * 4 + 16 : need;
  cudaError_t e = cudaMemsetAsync(static_cast<unsigned char*>(scratch) + (need - tail), 0, tail,
                                  reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    char buf[256];
    std::snprintf(buf, sizeof buf, "nf4_gemm_chunk_noalloc: clearing the scratch failed: %s", cudaGetErrorString(e));
    cudaGetLastError();
    nf4k::set_last_error(buf);
    return NF4_ECUDA;
  }
  return nf4_gemm_chunk(W, X, N, Y, scratch, stream);
}
