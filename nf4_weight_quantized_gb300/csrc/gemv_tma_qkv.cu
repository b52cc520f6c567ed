// gemv_tma_qkv.cu -- instantiations of the bulk-copy N=1 kernel, fused q/k/v epilogue.
#include "gemv_tma_dispatch.cuh"

namespace nf4k {
NF4_GEMV_TMA_DEFINE_DISPATCH(EPI_QKV)
}  // namespace nf4k
