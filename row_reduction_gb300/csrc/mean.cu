// mean.cu -- the one-CTA kernel that averages the per-row cross-entropy
// losses.
#include "mt_kernels.cuh"

namespace mt {

// mean = (sum of loss[0..rows)) / n, n = rows, or with an ignore index the
// number of rows whose label is not it (ignored rows hold loss 0; no such
// row gives 0/0 = NaN).  One CTA; each thread sums a strided subset in index
// order with compensated arithmetic (kMeanInFlight loads in flight per
// thread), then the block combines the partials in a fixed shuffle/shared-
// memory order, so the result does not depend on timing (no atomics).
constexpr int kMeanThreads = 256;
constexpr int kMeanInFlight = 4;   // loads in flight per thread

__global__ void __launch_bounds__(kMeanThreads)
    mean_kernel(const float *loss, float *mean, int64_t rows,
                const int32_t *labels, int32_t ignore_index,
                int32_t has_ignore) {
    // Launched as a programmatic dependent of the loss kernel.  Let the next
    // kernel on the stream launch now (it waits for this grid to complete
    // before it touches memory), then wait until the loss grid has
    // completed and its losses are visible.
    grid_launch_dependents();
    grid_wait_prerequisites();
    __shared__ RedScratch red;
    int parity = 0;
    __shared__ long long ignored_part[32];
    float s = 0.f, c = 0.f;
    long long ignored = 0;
    const int64_t T = blockDim.x;
    for (int64_t i0 = threadIdx.x; i0 < rows; i0 += kMeanInFlight * T) {
        float t[kMeanInFlight];
#pragma unroll
        for (int u = 0; u < kMeanInFlight; ++u)
            t[u] = i0 + u * T < rows ? loss[i0 + u * T] : 0.f;
#pragma unroll
        for (int u = 0; u < kMeanInFlight; ++u) {
            float sum, err;
            two_sum(s, t[u], sum, err);
            s = sum;
            c += err;
            if (has_ignore && i0 + u * T < rows &&
                labels[i0 + u * T] == ignore_index)
                ++ignored;
        }
    }
    row_allreduce_compensated(s, c, (int)blockDim.x, red, parity);
    long long total = 0;
    if (has_ignore) {
        // Exact count of ignored rows: warp sums, then thread 0 adds the
        // warps'.
        for (int off = 16; off > 0; off >>= 1)
            ignored += __shfl_xor_sync(kFull, ignored, off);
        if ((threadIdx.x & 31) == 0) ignored_part[threadIdx.x >> 5] = ignored;
        __syncthreads();
        if (threadIdx.x == 0)
            for (int w = 0; w < (int)(blockDim.x >> 5); ++w)
                total += ignored_part[w];
    }
    // One FP32 rounding of the compensated sum, one of the count (exact up
    // to 2^24 rows) and one of the quotient.
    if (threadIdx.x == 0) *mean = (s + c) / (float)(rows - total);
}

cudaError_t launch_mean(const float *loss, float *mean, int64_t rows,
                        const int32_t *labels, int32_t ignore_index,
                        int32_t has_ignore, cudaStream_t stream) {
    // Programmatic dependent launch lets this one-CTA kernel start while the
    // loss kernel finishes; it waits for that grid before reading.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kMeanThreads);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, mean_kernel, loss, mean, rows, labels,
                              ignore_index, has_ignore);
}

}  // namespace mt
