// Forward-kernel variants: 6-bit codes with the test hooks (see qlin_instances.h).
#include "qlin_forward.cuh"
#include "qlin_instances.h"

QLIN_KERNELS_EXPORT_W6(QLIN_INSTANTIATE)
