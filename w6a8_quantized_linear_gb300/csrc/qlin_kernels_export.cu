// Forward-kernel variants with the test exports (see qlin_instances.h).
#include "qlin_forward.cuh"
#include "qlin_instances.h"

QLIN_KERNELS_EXPORT(QLIN_INSTANTIATE)
