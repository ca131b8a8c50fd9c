// ops_residual_layernorm.cu -- instantiates the residual_layernorm kernels (register and loop paths).
#include "mt_kernels.cuh"

MT_DEFINE_LAUNCHER(launch_residual_layernorm, OP_RESIDUAL_LAYERNORM)
