// Forward-kernel variants: 4-bit codes, plain weight table (see qlin_instances.h).
#include "qlin_forward.cuh"
#include "qlin_instances.h"

QLIN_KERNELS_W4(QLIN_INSTANTIATE)
