// gemv_plain.cu -- instantiations of the N=1 kernel with the PLAIN epilogue.
#include "gemv_dispatch.cuh"

namespace nf4k {
NF4_GEMV_DEFINE_DISPATCH(EPI_PLAIN)
}  // namespace nf4k
