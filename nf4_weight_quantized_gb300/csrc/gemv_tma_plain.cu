// gemv_tma_plain.cu -- instantiations of the bulk-copy N=1 kernel, PLAIN epilogue.
#include "gemv_tma_dispatch.cuh"

namespace nf4k {
NF4_GEMV_TMA_DEFINE_DISPATCH(EPI_PLAIN)
}  // namespace nf4k
