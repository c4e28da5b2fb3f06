// The forward-kernel variants this library builds, by prologue kind:
// X(BITS, KIND, G, MODE) for every group size the format allows (4 and 8 for
// 4-bit codes only) in mode 0 (plain), G >= 32 for expert banks (mode 1), and
// 4-bit codes with G >= 32 for codebook levels (mode 2).  The kernels are
// instantiated in one translation unit per prologue kind (compiled in
// parallel) and declared extern where the host code takes their addresses.
#pragma once

#define QLIN_KERNELS_OF_KIND(X, KIND)                                                                      \
  X(4, KIND, 4, 0) X(4, KIND, 8, 0) X(4, KIND, 16, 0) X(4, KIND, 32, 0)                                     \
  X(4, KIND, 64, 0) X(4, KIND, 128, 0) X(4, KIND, 256, 0)                                                   \
  X(6, KIND, 16, 0) X(6, KIND, 32, 0) X(6, KIND, 64, 0) X(6, KIND, 128, 0) X(6, KIND, 256, 0)               \
  X(4, KIND, 32, 1) X(4, KIND, 64, 1) X(4, KIND, 128, 1) X(4, KIND, 256, 1)                                 \
  X(6, KIND, 32, 1) X(6, KIND, 64, 1) X(6, KIND, 128, 1) X(6, KIND, 256, 1)                                 \
  X(4, KIND, 32, 2) X(4, KIND, 64, 2) X(4, KIND, 128, 2) X(4, KIND, 256, 2)

#define QLIN_INSTANTIATE(B, K, G, M) template __global__ void qlin::qlin_forward_kernel<B, K, G, M>(qlin::FwdParams);
#define QLIN_DECLARE_EXTERN(B, K, G, M) \
  extern template __global__ void qlin::qlin_forward_kernel<B, K, G, M>(qlin::FwdParams);
