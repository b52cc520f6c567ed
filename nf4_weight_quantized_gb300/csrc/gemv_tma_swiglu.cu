// gemv_tma_swiglu.cu -- instantiations of the bulk-copy N=1 kernel, SWIGLU epilogue.
#include "gemv_tma_dispatch.cuh"

namespace nf4k {
NF4_GEMV_TMA_DEFINE_DISPATCH(EPI_SWIGLU)
}  // namespace nf4k
