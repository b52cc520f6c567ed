// gemv_resid.cu -- instantiations of the N=1 kernel with the RESID epilogue.
#include "gemv_dispatch.cuh"

namespace nf4k {
NF4_GEMV_DEFINE_DISPATCH(EPI_RESID)
}  // namespace nf4k
