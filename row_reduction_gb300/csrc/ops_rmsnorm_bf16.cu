// ops_rmsnorm_bf16.cu -- instantiates the rmsnorm kernels for BF16 storage
// (register and loop paths).
#include "mt_kernels.cuh"

MT_DEFINE_LAUNCHER(launch_rmsnorm_bf16, OP_RMSNORM, __nv_bfloat16)
