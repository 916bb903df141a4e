// tensor-core kernels (added with the tcgen05 path)
#include "device_common.cuh"
