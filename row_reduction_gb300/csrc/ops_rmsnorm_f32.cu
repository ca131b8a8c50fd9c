// ops_rmsnorm_f32.cu -- instantiates the rmsnorm kernels for FP32 storage
// (register and loop paths).
#include "mt_kernels.cuh"

MT_DEFINE_LAUNCHER(launch_rmsnorm_f32, OP_RMSNORM, float)
