// Forward-kernel variants: 6-bit codes, plain weight table; 4-bit codes with a codebook (see qlin_instances.h).
#include "qlin_forward.cuh"
#include "qlin_instances.h"

QLIN_KERNELS_W6_CODEBOOK(QLIN_INSTANTIATE)
