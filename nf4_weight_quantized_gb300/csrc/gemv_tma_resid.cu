// gemv_tma_resid.cu -- instantiations of the bulk-copy N=1 kernel, RESID epilogue.
#include "gemv_tma_dispatch.cuh"

namespace nf4k {
NF4_GEMV_TMA_DEFINE_DISPATCH(EPI_RESID)
}  // namespace nf4k
