// The forward-kernel variants this library builds: X(BITS, G, MODE) for every
// group size the format allows (4 and 8 for 4-bit codes only) in mode 0
// (plain weight table), mode 3 (the same with the test exports) and mode 4
// (the same for one activation row), G >= 32 for expert banks (modes 1 and 5,
// the latter for one row), and 4-bit codes with G >= 32 for codebook levels
// (modes 2 and 6).  The prologue kind is a runtime parameter, so consecutive
// launches of different prologues run the same code.  The variants are
// instantiated in several translation units (compiled in parallel) and
// declared extern where the host code takes their addresses.
#pragma once

#define QLIN_KERNELS_W4(X) X(4, 4, 0) X(4, 8, 0) X(4, 16, 0) X(4, 32, 0) X(4, 64, 0) X(4, 128, 0) X(4, 256, 0)
#define QLIN_KERNELS_W6(X) X(6, 16, 0) X(6, 32, 0) X(6, 64, 0) X(6, 128, 0) X(6, 256, 0)
#define QLIN_KERNELS_CODEBOOK(X) X(4, 32, 2) X(4, 64, 2) X(4, 128, 2) X(4, 256, 2)
#define QLIN_KERNELS_MOE_W4(X) X(4, 32, 1) X(4, 64, 1) X(4, 128, 1) X(4, 256, 1)
#define QLIN_KERNELS_MOE_W6(X) X(6, 32, 1) X(6, 64, 1) X(6, 128, 1) X(6, 256, 1)
#define QLIN_KERNELS_EXPORT_W4(X) X(4, 4, 3) X(4, 8, 3) X(4, 16, 3) X(4, 32, 3) X(4, 64, 3) X(4, 128, 3) X(4, 256, 3)
#define QLIN_KERNELS_EXPORT_W6(X) X(6, 16, 3) X(6, 32, 3) X(6, 64, 3) X(6, 128, 3) X(6, 256, 3)
// mode 4: the plain weight table for one activation row
#define QLIN_KERNELS_ONE_ROW_W4(X) X(4, 4, 4) X(4, 8, 4) X(4, 16, 4) X(4, 32, 4) X(4, 64, 4) X(4, 128, 4) X(4, 256, 4)
#define QLIN_KERNELS_ONE_ROW_W6(X) X(6, 16, 4) X(6, 32, 4) X(6, 64, 4) X(6, 128, 4) X(6, 256, 4)
// modes 5 and 6: expert banks and codebook levels for one activation row
#define QLIN_KERNELS_MOE_ONE_ROW(X) \
  X(4, 32, 5) X(4, 64, 5) X(4, 128, 5) X(4, 256, 5) X(6, 32, 5) X(6, 64, 5) X(6, 128, 5) X(6, 256, 5)
#define QLIN_KERNELS_CODEBOOK_ONE_ROW(X) X(4, 32, 6) X(4, 64, 6) X(4, 128, 6) X(4, 256, 6)
#define QLIN_KERNELS_ALL(X)                                                                                 \
  QLIN_KERNELS_W4(X) QLIN_KERNELS_W6(X) QLIN_KERNELS_CODEBOOK(X) QLIN_KERNELS_MOE_W4(X) QLIN_KERNELS_MOE_W6(X) \
  QLIN_KERNELS_EXPORT_W4(X) QLIN_KERNELS_EXPORT_W6(X) QLIN_KERNELS_ONE_ROW_W4(X) QLIN_KERNELS_ONE_ROW_W6(X)   \
  QLIN_KERNELS_MOE_ONE_ROW(X) QLIN_KERNELS_CODEBOOK_ONE_ROW(X)

// The tcgen05 main loop (qlin_tc_kernel): groups of 32 k and more, the weight
// table without (mode 0) and with (mode 3) the test hooks.
#define QLIN_TC_KERNELS(X) X(4, 32, 0) X(4, 64, 0) X(4, 128, 0) X(4, 256, 0) X(6, 32, 0) X(6, 64, 0) X(6, 128, 0) X(6, 256, 0)
#define QLIN_TC_KERNELS_EXPORT(X) \
  X(4, 32, 3) X(4, 64, 3) X(4, 128, 3) X(4, 256, 3) X(6, 32, 3) X(6, 64, 3) X(6, 128, 3) X(6, 256, 3)
#define QLIN_TC_ALL(X) QLIN_TC_KERNELS(X) QLIN_TC_KERNELS_EXPORT(X)

#define QLIN_INSTANTIATE(B, G, M) template __global__ void qlin::qlin_forward_kernel<B, G, M>(qlin::FwdParams);
#define QLIN_DECLARE_EXTERN(B, G, M) \
  extern template __global__ void qlin::qlin_forward_kernel<B, G, M>(qlin::FwdParams);
#define QLIN_TC_INSTANTIATE(B, G, M) template __global__ void qlin::qlin_tc_kernel<B, G, M>(qlin::FwdParams);
#define QLIN_TC_DECLARE_EXTERN(B, G, M) extern template __global__ void qlin::qlin_tc_kernel<B, G, M>(qlin::FwdParams);
