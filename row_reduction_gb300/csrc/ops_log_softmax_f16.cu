// ops_log_softmax_f16.cu -- instantiates the log_softmax kernels for FP16 storage
// (register and loop paths).
#include "mt_kernels.cuh"

MT_DEFINE_LAUNCHER(launch_log_softmax_f16, OP_LOG_SOFTMAX, __half)
