// Forward-kernel variants: expert banks of 4-bit codes (see qlin_instances.h).
#include "qlin_forward.cuh"
#include "qlin_instances.h"

QLIN_KERNELS_MOE_W4(QLIN_INSTANTIATE)
