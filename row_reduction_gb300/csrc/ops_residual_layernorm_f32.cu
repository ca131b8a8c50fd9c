// ops_residual_layernorm_f32.cu -- instantiates the residual_layernorm kernels for FP32 storage
// (register and loop paths).
#include "mt_kernels.cuh"

MT_DEFINE_LAUNCHER(launch_residual_layernorm_f32, OP_RESIDUAL_LAYERNORM, float)
