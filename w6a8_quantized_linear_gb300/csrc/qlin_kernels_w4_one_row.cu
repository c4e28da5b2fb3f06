// Forward-kernel variants: 4-bit codes, plain weight table, one activation row (see qlin_instances.h).
#include "qlin_forward.cuh"
#include "qlin_instances.h"

QLIN_KERNELS_ONE_ROW_W4(QLIN_INSTANTIATE)
