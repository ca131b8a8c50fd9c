// ops_cross_entropy_f16.cu -- instantiates the cross_entropy kernels for FP16 storage
// (register and loop paths).
#include "mt_kernels.cuh"

MT_DEFINE_LAUNCHER(launch_cross_entropy_f16, OP_CROSS_ENTROPY, __half)
