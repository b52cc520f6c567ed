// gemv_tma_dispatch.cuh -- runtime (nch, rb, sub, x dtype, lut mode) -> instantiation.
#pragma once

#include "gemv_tma.cuh"

namespace nf4k {

// Compiled (nch, rb, sub): (1, 2, 2), (1, 4, 4), (1, 4, 2), (1, 8, 8),
// (1, 8, 4), (1, 8, 2), (2, 2, 2), (2, 4, 4).  The fp16-level loop is compiled
// for bf16 activations only (fp32 activations always take the fp32 table).
inline bool gemv_tma_variant_exists(int nch, int rb, int sub) {
  if (nch == 1) return (rb == 2 && sub == 2) || (rb == 4 && (sub == 4 || sub == 2)) || (rb == 8 && (sub == 8 || sub == 4 || sub == 2));
  return nch == 2 && (rb == 2 || rb == 4) && sub == rb;
}

template <int EPI>
struct GemvTmaDispatch {
  static const void* ptr(int nch, int rb, int sub, bool xb, int lut);
  static cudaError_t launch(int nch, int rb, int sub, bool xb, int lut, const GemvArgs& a, const TmaPlan& p,
                            int blocks, int threads, int smem, cudaStream_t s);
};

#define NF4_TMA_CASE(E, N, R, U)                                                                    \
  if (nch == N && rb == R && sub == U) {                                                            \
    if (lut == LUT_F16MIX) return xb ? gemv_tma_ptr<N, R, U, E, true, LUT_F16MIX>() : nullptr;      \
    return xb ? gemv_tma_ptr<N, R, U, E, true, LUT_F32>() : gemv_tma_ptr<N, R, U, E, false, LUT_F32>(); \
  }
#define NF4_TMA_LAUNCH(E, N, R, U)                                                                  \
  if (nch == N && rb == R && sub == U) {                                                            \
    if (lut == LUT_F16MIX)                                                                          \
      return xb ? launch_gemv_tma_instance<N, R, U, E, true, LUT_F16MIX>(a, p, blocks, threads, smem, s) \
                : cudaErrorInvalidValue;                                                            \
    return xb ? launch_gemv_tma_instance<N, R, U, E, true, LUT_F32>(a, p, blocks, threads, smem, s)   \
              : launch_gemv_tma_instance<N, R, U, E, false, LUT_F32>(a, p, blocks, threads, smem, s); \
  }
#define NF4_TMA_VARIANTS(M, E) \
  M(E, 1, 2, 2) M(E, 1, 4, 4) M(E, 1, 4, 2) M(E, 1, 8, 8) M(E, 1, 8, 4) M(E, 1, 8, 2) M(E, 2, 2, 2) M(E, 2, 4, 4)

#define NF4_GEMV_TMA_DEFINE_DISPATCH(E)                                                             \
  template <>                                                                                       \
  const void* GemvTmaDispatch<E>::ptr(int nch, int rb, int sub, bool xb, int lut) {                 \
    NF4_TMA_VARIANTS(NF4_TMA_CASE, E)                                                               \
    return nullptr;                                                                                 \
  }                                                                                                 \
  template <>                                                                                       \
  cudaError_t GemvTmaDispatch<E>::launch(int nch, int rb, int sub, bool xb, int lut, const GemvArgs& a, \
                                         const TmaPlan& p, int blocks, int threads, int smem,       \
                                         cudaStream_t s) {                                          \
    NF4_TMA_VARIANTS(NF4_TMA_LAUNCH, E)                                                             \
    return cudaErrorInvalidValue;                                                                   \
  }

}  // namespace nf4k
