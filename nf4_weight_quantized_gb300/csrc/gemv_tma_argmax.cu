// gemv_tma_argmax.cu -- instantiations of the bulk-copy N=1 kernel, ARGMAX epilogue.
#include "gemv_tma_dispatch.cuh"

namespace nf4k {
NF4_GEMV_TMA_DEFINE_DISPATCH(EPI_ARGMAX)
}  // namespace nf4k
