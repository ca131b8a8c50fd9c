// ops_row_sum.cu -- instantiates the row_sum kernels (register and loop paths).
#include "mt_kernels.cuh"

MT_DEFINE_LAUNCHER(launch_row_sum, OP_ROW_SUM)
