// ops_rmsnorm_f16.cu -- instantiates the rmsnorm kernels for FP16 storage
// (register and loop paths).
#include "mt_kernels.cuh"

MT_DEFINE_LAUNCHER(launch_rmsnorm_f16, OP_RMSNORM, __half)
