// Forward-kernel variants with the swiglu prologue (see qlin_instances.h).
#include "qlin_forward.cuh"
#include "qlin_instances.h"

QLIN_KERNELS_OF_KIND(QLIN_INSTANTIATE, 2)
