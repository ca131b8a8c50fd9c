// ops_softmax_f32.cu -- instantiates the softmax kernels for FP32 storage
// (register and loop paths).
#include "mt_kernels.cuh"

MT_DEFINE_LAUNCHER(launch_softmax_f32, OP_SOFTMAX, float)
