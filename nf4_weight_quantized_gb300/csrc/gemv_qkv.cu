// gemv_qkv.cu -- instantiations of the N=1 kernel with the fused q/k/v epilogue.
#include "gemv_dispatch.cuh"

namespace nf4k {
NF4_GEMV_DEFINE_DISPATCH(EPI_QKV)
}  // namespace nf4k
