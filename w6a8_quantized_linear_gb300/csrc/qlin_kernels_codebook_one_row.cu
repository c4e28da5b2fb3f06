// Forward-kernel variants: codebook levels, one activation row (see qlin_instances.h).
#include "qlin_forward.cuh"
#include "qlin_instances.h"

QLIN_KERNELS_CODEBOOK_ONE_ROW(QLIN_INSTANTIATE)
