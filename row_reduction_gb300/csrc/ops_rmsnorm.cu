// ops_rmsnorm.cu -- instantiates the rmsnorm kernels (register and loop paths).
#include "mt_kernels.cuh"

MT_DEFINE_LAUNCHER(launch_rmsnorm, OP_RMSNORM)
