// gemv_swiglu.cu -- instantiations of the N=1 kernel with the SWIGLU epilogue.
#include "gemv_dispatch.cuh"

namespace nf4k {
NF4_GEMV_DEFINE_DISPATCH(EPI_SWIGLU)
}  // namespace nf4k
