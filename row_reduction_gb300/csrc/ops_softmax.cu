// ops_softmax.cu -- instantiates the softmax kernels (register and loop paths).
#include "mt_kernels.cuh"

MT_DEFINE_LAUNCHER(launch_softmax, OP_SOFTMAX)
