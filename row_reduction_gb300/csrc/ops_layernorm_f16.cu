// ops_layernorm_f16.cu -- instantiates the layernorm kernels for FP16 storage
// (register and loop paths).
#include "mt_kernels.cuh"

MT_DEFINE_LAUNCHER(launch_layernorm_f16, OP_LAYERNORM, __half)
