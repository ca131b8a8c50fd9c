// ops_layernorm_f32.cu -- instantiates the layernorm kernels for FP32 storage
// (register and loop paths).
#include "mt_kernels.cuh"

MT_DEFINE_LAUNCHER(launch_layernorm_f32, OP_LAYERNORM, float)
