// Forward-kernel variants on the tcgen05 main loop: weight table (see qlin_instances.h).
#include "qlin_forward_tc.cuh"
#include "qlin_instances.h"

QLIN_TC_KERNELS(QLIN_TC_INSTANTIATE)
