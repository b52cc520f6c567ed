// gemv_glu.cu -- instantiations of the N=1 kernel with the interleaved gate/up
// SwiGLU epilogue.
#include "gemv_dispatch.cuh"

namespace nf4k {
NF4_GEMV_DEFINE_DISPATCH(EPI_GLU)
}  // namespace nf4k
