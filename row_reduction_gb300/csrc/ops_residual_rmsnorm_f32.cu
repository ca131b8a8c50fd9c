// ops_residual_rmsnorm_f32.cu -- instantiates the residual_rmsnorm kernels for FP32 storage
// (register and loop paths).
#include "mt_kernels.cuh"

MT_DEFINE_LAUNCHER(launch_residual_rmsnorm_f32, OP_RESIDUAL_RMSNORM, float)
