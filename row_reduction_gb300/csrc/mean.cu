// mean.cu -- the one-CTA kernel that averages the per-row cross-entropy
// losses.
#include "mt_kernels.cuh"

namespace mt {

// mean = (sum of loss[0..rows)) / rows.  One CTA; each thread sums a strided
// subset in index order with compensated arithmetic, then the block combines
// the partials in a fixed shuffle/shared-memory order, so the result does not
// depend on timing (no atomics).
__global__ void __launch_bounds__(1024)
    mean_kernel(const float *loss, float *mean, int64_t rows) {
    // Launched as a programmatic dependent of the loss kernel: wait until
    // that grid has completed and its losses are visible.
    grid_wait_prerequisites();
    grid_launch_dependents();
    __shared__ RedScratch red;
    int parity = 0;
    float s = 0.f, c = 0.f;
    for (int64_t i = threadIdx.x; i < rows; i += blockDim.x) {
        float t, err;
        two_sum(s, loss[i], t, err);
        s = t;
        c += err;
    }
    row_allreduce_compensated(s, c, (int)blockDim.x, red, parity);
    if (threadIdx.x == 0)
        *mean = (float)((double)(s + c) / (double)rows);
}

cudaError_t launch_mean(const float *loss, float *mean, int64_t rows,
                        cudaStream_t stream) {
    // Programmatic dependent launch lets this one-CTA kernel start while the
    // loss kernel finishes; it waits for that grid before reading.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(1024);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, mean_kernel, loss, mean, rows);
}

}  // namespace mt
