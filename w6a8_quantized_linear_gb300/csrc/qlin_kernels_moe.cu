// Forward-kernel variants: expert banks (see qlin_instances.h).
#include "qlin_forward.cuh"
#include "qlin_instances.h"

QLIN_KERNELS_MOE(QLIN_INSTANTIATE)
