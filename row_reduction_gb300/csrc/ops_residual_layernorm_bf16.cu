// ops_residual_layernorm_bf16.cu -- instantiates the residual_layernorm kernels for BF16 storage
// (register and loop paths).
#include "mt_kernels.cuh"

MT_DEFINE_LAUNCHER(launch_residual_layernorm_bf16, OP_RESIDUAL_LAYERNORM, __nv_bfloat16)
