// gemv_tma_dispatch.cuh -- runtime (nch, rb, x dtype, lut mode) -> instantiation.
#pragma once

#include "gemv_tma.cuh"

namespace nf4k {

// Compiled (nch, rb): (1, 2), (1, 4), (1, 8), (2, 2), (2, 4).
inline bool gemv_tma_variant_exists(int nch, int rb) {
  return (nch == 1 && (rb == 2 || rb == 4 || rb == 8)) || (nch == 2 && (rb == 2 || rb == 4));
}

template <int EPI>
struct GemvTmaDispatch {
  static const void* ptr(int nch, int rb, bool xb, int lut);
  static cudaError_t launch(int nch, int rb, bool xb, int lut, const GemvArgs& a, const TmaPlan& p, int blocks,
                            int threads, int smem, cudaStream_t s);
};

#define NF4_TMA_CASE_L(E, N, R, L)                                                                  \
  if (nch == N && rb == R && lut == L)                                                              \
    return xb ? gemv_tma_ptr<N, R, E, true, L>() : gemv_tma_ptr<N, R, E, false, L>();
#define NF4_TMA_LAUNCH_L(E, N, R, L)                                                                \
  if (nch == N && rb == R && lut == L)                                                              \
    return xb ? launch_gemv_tma_instance<N, R, E, true, L>(a, p, blocks, threads, smem, s)          \
              : launch_gemv_tma_instance<N, R, E, false, L>(a, p, blocks, threads, smem, s);
#define NF4_TMA_CASES(M, E, N, R) M(E, N, R, LUT_F32) M(E, N, R, LUT_F16MIX)

#define NF4_GEMV_TMA_DEFINE_DISPATCH(E)                                                             \
  template <>                                                                                       \
  const void* GemvTmaDispatch<E>::ptr(int nch, int rb, bool xb, int lut) {                          \
    NF4_TMA_CASES(NF4_TMA_CASE_L, E, 1, 2)                                                          \
    NF4_TMA_CASES(NF4_TMA_CASE_L, E, 1, 4)                                                          \
    NF4_TMA_CASES(NF4_TMA_CASE_L, E, 1, 8)                                                          \
    NF4_TMA_CASES(NF4_TMA_CASE_L, E, 2, 2)                                                          \
    NF4_TMA_CASES(NF4_TMA_CASE_L, E, 2, 4)                                                          \
    return nullptr;                                                                                 \
  }                                                                                                 \
  template <>                                                                                       \
  cudaError_t GemvTmaDispatch<E>::launch(int nch, int rb, bool xb, int lut, const GemvArgs& a,      \
                                         const TmaPlan& p, int blocks, int threads, int smem,       \
                                         cudaStream_t s) {                                          \
    NF4_TMA_CASES(NF4_TMA_LAUNCH_L, E, 1, 2)                                                        \
    NF4_TMA_CASES(NF4_TMA_LAUNCH_L, E, 1, 4)                                                        \
    NF4_TMA_CASES(NF4_TMA_LAUNCH_L, E, 1, 8)                                                        \
    NF4_TMA_CASES(NF4_TMA_LAUNCH_L, E, 2, 2)                                                        \
    NF4_TMA_CASES(NF4_TMA_LAUNCH_L, E, 2, 4)                                                        \
    return cudaErrorInvalidValue;                                                                   \
  }

}  // namespace nf4k
