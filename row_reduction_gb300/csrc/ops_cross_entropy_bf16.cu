// ops_cross_entropy_bf16.cu -- instantiates the cross_entropy kernels for BF16 storage
// (register and loop paths).
#include "mt_kernels.cuh"

MT_DEFINE_LAUNCHER(launch_cross_entropy_bf16, OP_CROSS_ENTROPY, __nv_bfloat16)
