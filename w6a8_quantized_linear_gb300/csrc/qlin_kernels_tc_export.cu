// Forward-kernel variants on the tcgen05 main loop: weight table with the test hooks (see qlin_instances.h).
#include "qlin_forward_tc.cuh"
#include "qlin_instances.h"

QLIN_TC_KERNELS_EXPORT(QLIN_TC_INSTANTIATE)
