// ops_row_sum_f32.cu -- instantiates the row_sum kernels for FP32 storage
// (register and loop paths).
#include "mt_kernels.cuh"

MT_DEFINE_LAUNCHER(launch_row_sum_f32, OP_ROW_SUM, float)
