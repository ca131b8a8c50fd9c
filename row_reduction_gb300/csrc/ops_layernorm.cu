// ops_layernorm.cu -- instantiates the layernorm kernels (register and loop paths).
#include "mt_kernels.cuh"

MT_DEFINE_LAUNCHER(launch_layernorm, OP_LAYERNORM)
