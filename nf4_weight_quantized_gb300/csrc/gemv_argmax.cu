// gemv_argmax.cu -- instantiations of the N=1 kernel with the ARGMAX epilogue.
#include "gemv_dispatch.cuh"

namespace nf4k {
NF4_GEMV_DEFINE_DISPATCH(EPI_ARGMAX)
}  // namespace nf4k
