// ops_log_softmax_bf16.cu -- instantiates the log_softmax kernels for BF16 storage
// (register and loop paths).
#include "mt_kernels.cuh"

MT_DEFINE_LAUNCHER(launch_log_softmax_bf16, OP_LOG_SOFTMAX, __nv_bfloat16)
