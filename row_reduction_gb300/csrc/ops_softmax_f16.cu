// ops_softmax_f16.cu -- instantiates the softmax kernels for FP16 storage
// (register and loop paths).
#include "mt_kernels.cuh"

MT_DEFINE_LAUNCHER(launch_softmax_f16, OP_SOFTMAX, __half)
