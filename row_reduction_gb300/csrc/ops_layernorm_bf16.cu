// ops_layernorm_bf16.cu -- instantiates the layernorm kernels for BF16 storage
// (register and loop paths).
#include "mt_kernels.cuh"

MT_DEFINE_LAUNCHER(launch_layernorm_bf16, OP_LAYERNORM, __nv_bfloat16)
