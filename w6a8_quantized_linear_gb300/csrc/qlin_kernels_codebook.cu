// Forward-kernel variants: 4-bit codes with a codebook (see qlin_instances.h).
#include "qlin_forward.cuh"
#include "qlin_instances.h"

QLIN_KERNELS_CODEBOOK(QLIN_INSTANTIATE)
