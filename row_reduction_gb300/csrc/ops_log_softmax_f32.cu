// ops_log_softmax_f32.cu -- instantiates the log_softmax kernels for FP32 storage
// (register and loop paths).
#include "mt_kernels.cuh"

MT_DEFINE_LAUNCHER(launch_log_softmax_f32, OP_LOG_SOFTMAX, float)
