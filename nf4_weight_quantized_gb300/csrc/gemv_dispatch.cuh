// gemv_dispatch.cuh -- maps a runtime (nch, rb, x dtype) to a compiled instantiation.
#pragma once

#include "gemv_kernel.cuh"

namespace nf4k {

// Compiled (nch, rb, big) triples: nch = 1 with rb in {2, 4, 8}; nch = 2 with
// rb in {2, 4}; and the register-capped big-row variants (1, 2) and (2, 2).
inline bool gemv_variant_exists(int nch, int rb, bool big) {
  if (big) return rb == 2 && (nch == 1 || nch == 2);
  return (nch == 1 && (rb == 2 || rb == 4 || rb == 8)) || (nch == 2 && (rb == 2 || rb == 4));
}

template <int EPI>
struct GemvDispatch {
  static const void* ptr(int nch, int rb, bool big, bool xb);
  static cudaError_t launch(int nch, int rb, bool big, bool xb, const GemvArgs& a, const GemvConfig& c,
                            cudaStream_t s);
};

#define NF4_PTR_CASE(E, N, R, B, T)                                                    \
  if (nch == N && rb == R && big == B)                                                 \
    return xb ? gemv_instance_ptr<N, R, E, true, T>() : gemv_instance_ptr<N, R, E, false, T>();
#define NF4_LAUNCH_CASE(E, N, R, B, T)                                                 \
  if (nch == N && rb == R && big == B)                                                 \
    return xb ? launch_gemv_instance<N, R, E, true, T>(a, c, s)                        \
              : launch_gemv_instance<N, R, E, false, T>(a, c, s);

// Defines the dispatch of one epilogue; each epilogue lives in its own
// translation unit so the instantiations compile in parallel.
#define NF4_GEMV_DEFINE_DISPATCH(E)                                                               \
  template <>                                                                                     \
  const void* GemvDispatch<E>::ptr(int nch, int rb, bool big, bool xb) {                          \
    NF4_PTR_CASE(E, 1, 2, false, false) NF4_PTR_CASE(E, 1, 4, false, false)                           \
    NF4_PTR_CASE(E, 1, 8, false, false) NF4_PTR_CASE(E, 2, 2, false, false)                           \
    NF4_PTR_CASE(E, 2, 4, false, false) NF4_PTR_CASE(E, 1, 2, true, true)                           \
    NF4_PTR_CASE(E, 2, 2, true, true)                                                             \
    return nullptr;                                                                               \
  }                                                                                               \
  template <>                                                                                     \
  cudaError_t GemvDispatch<E>::launch(int nch, int rb, bool big, bool xb, const GemvArgs& a,      \
                                      const GemvConfig& c, cudaStream_t s) {                      \
    NF4_LAUNCH_CASE(E, 1, 2, false, false) NF4_LAUNCH_CASE(E, 1, 4, false, false)                     \
    NF4_LAUNCH_CASE(E, 1, 8, false, false) NF4_LAUNCH_CASE(E, 2, 2, false, false)                     \
    NF4_LAUNCH_CASE(E, 2, 4, false, false) NF4_LAUNCH_CASE(E, 1, 2, true, true)                     \
    NF4_LAUNCH_CASE(E, 2, 2, true, true)                                                          \
    return cudaErrorInvalidValue;                                                                 \
  }

}  // namespace nf4k
