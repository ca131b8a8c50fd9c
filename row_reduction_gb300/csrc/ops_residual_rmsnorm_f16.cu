// ops_residual_rmsnorm_f16.cu -- instantiates the residual_rmsnorm kernels for FP16 storage
// (register and loop paths).
#include "mt_kernels.cuh"

MT_DEFINE_LAUNCHER(launch_residual_rmsnorm_f16, OP_RESIDUAL_RMSNORM, __half)
