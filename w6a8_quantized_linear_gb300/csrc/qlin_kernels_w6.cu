// Forward-kernel variants: 6-bit codes, plain weight table (see qlin_instances.h).
#include "qlin_forward.cuh"
#include "qlin_instances.h"

QLIN_KERNELS_W6(QLIN_INSTANTIATE)
