// ops_row_sum_bf16.cu -- instantiates the row_sum kernels for BF16 storage
// (register and loop paths).
#include "mt_kernels.cuh"

MT_DEFINE_LAUNCHER(launch_row_sum_bf16, OP_ROW_SUM, __nv_bfloat16)
