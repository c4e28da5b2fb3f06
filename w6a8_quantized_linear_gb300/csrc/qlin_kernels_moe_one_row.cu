// Forward-kernel variants: expert banks, one activation row (see qlin_instances.h).
#include "qlin_forward.cuh"
#include "qlin_instances.h"

QLIN_KERNELS_MOE_ONE_ROW(QLIN_INSTANTIATE)
