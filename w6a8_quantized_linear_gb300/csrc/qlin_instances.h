// The forward-kernel variants this library builds, by prologue kind:
// X(BITS, KIND, G, MOE) for every group size the format allows (4 and 8 for
// 4-bit codes only) and, for expert banks, G >= 32.  The kernels are
// instantiated in one translation unit per prologue kind (compiled in
// parallel) and declared extern where the host code takes their addresses.
#pragma once

#define QLIN_KERNELS_OF_KIND(X, KIND)                                                                      \
  X(4, KIND, 4, false) X(4, KIND, 8, false) X(4, KIND, 16, false) X(4, KIND, 32, false)                     \
  X(4, KIND, 64, false) X(4, KIND, 128, false) X(4, KIND, 256, false)                                       \
  X(6, KIND, 16, false) X(6, KIND, 32, false) X(6, KIND, 64, false) X(6, KIND, 128, false)                  \
  X(6, KIND, 256, false)                                                                                    \
  X(4, KIND, 32, true) X(4, KIND, 64, true) X(4, KIND, 128, true) X(4, KIND, 256, true)                     \
  X(6, KIND, 32, true) X(6, KIND, 64, true) X(6, KIND, 128, true) X(6, KIND, 256, true)

#define QLIN_INSTANTIATE(B, K, G, M) template __global__ void qlin::qlin_forward_kernel<B, K, G, M>(qlin::FwdParams);
#define QLIN_DECLARE_EXTERN(B, K, G, M) \
  extern template __global__ void qlin::qlin_forward_kernel<B, K, G, M>(qlin::FwdParams);
