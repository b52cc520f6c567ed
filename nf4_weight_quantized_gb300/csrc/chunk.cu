// chunk.cu -- prefill chunk (N <= 32) on the tcgen05 tensor cores.
#include "common.cuh"

namespace nf4k {

cudaError_t launch_chunk(const uint8_t*, const float*, int, int, const uint16_t*, int, float*, void*, const Codebook&,
                         cudaStream_t, int) {
  return cudaErrorNotSupported;
}

size_t chunk_workspace_bytes(int64_t, int64_t, int) { return 0; }

std::string describe_chunk(int64_t, int64_t, int, int) { return "chunk: not available"; }

}  // namespace nf4k
