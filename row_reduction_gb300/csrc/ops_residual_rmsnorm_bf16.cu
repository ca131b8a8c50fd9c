// ops_residual_rmsnorm_bf16.cu -- instantiates the residual_rmsnorm kernels for BF16 storage
// (register and loop paths).
#include "mt_kernels.cuh"

MT_DEFINE_LAUNCHER(launch_residual_rmsnorm_bf16, OP_RESIDUAL_RMSNORM, __nv_bfloat16)
