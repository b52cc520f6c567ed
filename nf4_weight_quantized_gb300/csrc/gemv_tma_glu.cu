// gemv_tma_glu.cu -- instantiations of the bulk-copy N=1 kernel, interleaved
// gate/up SwiGLU epilogue.
#include "gemv_tma_dispatch.cuh"

namespace nf4k {
NF4_GEMV_TMA_DEFINE_DISPATCH(EPI_GLU)
}  // namespace nf4k
