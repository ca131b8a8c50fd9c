// ops_cross_entropy_f32.cu -- instantiates the cross_entropy kernels for FP32 storage
// (register and loop paths).
#include "mt_kernels.cuh"

MT_DEFINE_LAUNCHER(launch_cross_entropy_f32, OP_CROSS_ENTROPY, float)
