// probe.cu -- measurement aids: a plain vectorised device-to-device copy, a
// read of the same shape, and an empty kernel.  All three launch the way the
// row-reduction kernels do (as programmatic dependents of the previous
// kernel on the stream, one wave of resident CTAs), so a benchmark can put a
// row-reduction launch beside the
// floor of a launch that moves the same bytes with no arithmetic (in and
// out, or in only), or no bytes at all, timed by the same method on the
// same buffers.
#include "mt_kernels.cuh"

namespace mt {

// Copies n 16-byte words from src to dst.  CTA b copies the contiguous
// slice [b*per, min(n, (b+1)*per)) of per = ceil(n / grid) words, the way a
// row-reduction CTA owns its rows; its threads stride over the slice with U
// predicated loads in flight before the U stores.  With `prefetch`, thread 0
// first asks L2 for the CTA's slice, before the wait on the previous grid,
// as the operators' MT_PLAN_PDL launches do.
template <int U>
__global__ void __launch_bounds__(1024)
    probe_copy_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                      int64_t n, int prefetch) {
    const int64_t per = (n + gridDim.x - 1) / gridDim.x;
    const int64_t lo = (int64_t)blockIdx.x * per;
    const int64_t hi = lo + per < n ? lo + per : n;
    if (prefetch && threadIdx.x == 0 && lo < hi)
        prefetch_l2(src + lo, (hi - lo) * 16);
    grid_launch_dependents();
    grid_wait_prerequisites();
    const int64_t T = blockDim.x;
    for (int64_t i = lo + threadIdx.x; i < hi; i += (int64_t)U * T) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (i + u * T < hi) v[u] = src[i + u * T];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (i + u * T < hi) dst[i + u * T] = v[u];
    }
}

// Reads n 16-byte words from src with the same slices, threads and loads in
// flight as probe_copy_kernel, and writes one 32-bit word per CTA: the XOR
// of every word of its slice (so no load can be elided) to dst[blockIdx.x].
// The floor of an operator that reads a matrix and writes one value per row.
template <int U>
__global__ void __launch_bounds__(1024)
    probe_read_kernel(const uint4 *__restrict__ src, unsigned *__restrict__ dst,
                      int64_t n, int prefetch) {
    __shared__ unsigned part[32];
    const int64_t per = (n + gridDim.x - 1) / gridDim.x;
    const int64_t lo = (int64_t)blockIdx.x * per;
    const int64_t hi = lo + per < n ? lo + per : n;
    if (prefetch && threadIdx.x == 0 && lo < hi)
        prefetch_l2(src + lo, (hi - lo) * 16);
    grid_launch_dependents();
    grid_wait_prerequisites();
    const int64_t T = blockDim.x;
    unsigned acc = 0;
    for (int64_t i = lo + threadIdx.x; i < hi; i += (int64_t)U * T) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            v[u] = i + u * T < hi ? src[i + u * T] : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int u = 0; u < U; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        acc ^= __shfl_xor_sync(kFull, acc, off);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned t = 0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t ^= part[w];
        dst[blockIdx.x] = t;
    }
}

// Does nothing but take part in the dependent-launch chain.
__global__ void __launch_bounds__(1024) probe_empty_kernel() {
    grid_launch_dependents();
    grid_wait_prerequisites();
}

namespace {

typedef void (*CopyFn)(const uint4 *, uint4 *, int64_t, int);

typedef void (*ReadFn)(const uint4 *, unsigned *, int64_t, int);

ReadFn read_kernel_for(int unroll) {
    switch (unroll) {
        case 1: return probe_read_kernel<1>;
        case 2: return probe_read_kernel<2>;
        case 4: return probe_read_kernel<4>;
        case 8: return probe_read_kernel<8>;
    }
    return nullptr;
}

CopyFn copy_kernel_for(int unroll) {
    switch (unroll) {
        case 1: return probe_copy_kernel<1>;
        case 2: return probe_copy_kernel<2>;
        case 4: return probe_copy_kernel<4>;
        case 8: return probe_copy_kernel<8>;
    }
    return nullptr;
}

cudaError_t launch_pdl(const void *fn, int grid, int threads, void **args,
                       cudaStream_t stream) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

// grid == 0: every CTA the device holds at once (SMs x resident CTAs).
cudaError_t resolve_grid(const void *fn, int threads, int *grid) {
    if (*grid > 0) return cudaSuccess;
    int dev = 0, sms = 0, bps = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, fn, threads,
                                                          0);
    if (e != cudaSuccess) return e;
    *grid = sms * (bps > 0 ? bps : 1);
    return cudaSuccess;
}

bool bad_block(int threads) {
    return threads < 32 || threads > 1024 || threads % 32 != 0;
}

}  // namespace
}  // namespace mt

using namespace mt;

extern "C" {

mt_status mt_probe_copy(const void *src, void *dst, int64_t bytes,
                        int32_t threads, int32_t unroll, int32_t grid,
                        int32_t flags, mt_stream_t stream) {
    if (bytes < 0 || bytes % 16 != 0 || bad_block(threads) || grid < 0 ||
        (flags & ~MT_PLAN_PDL) != 0)
        return MT_ERR_INVALID_ARGUMENT;
    CopyFn fn = copy_kernel_for(unroll);
    if (fn == nullptr) return MT_ERR_INVALID_ARGUMENT;
    if (bytes == 0) return MT_OK;
    if (src == nullptr || dst == nullptr ||
        (reinterpret_cast<uintptr_t>(src) & 15) != 0 ||
        (reinterpret_cast<uintptr_t>(dst) & 15) != 0)
        return MT_ERR_INVALID_ARGUMENT;
    const char *s = static_cast<const char *>(src);
    char *d = static_cast<char *>(dst);
    if (s < d + bytes && d < s + bytes) return MT_ERR_INVALID_ARGUMENT;
    int g = grid;
    cudaError_t e =
        resolve_grid(reinterpret_cast<const void *>(fn), threads, &g);
    if (e == cudaSuccess) {
        const uint4 *sp = static_cast<const uint4 *>(src);
        uint4 *dp = static_cast<uint4 *>(dst);
        int64_t n = bytes / 16;
        int prefetch = (flags & MT_PLAN_PDL) != 0;
        void *args[] = {&sp, &dp, &n, &prefetch};
        e = launch_pdl(reinterpret_cast<const void *>(fn), g, threads, args,
                       (cudaStream_t)stream);
    }
    return status_from_cuda(e);
}

mt_status mt_probe_read(const void *src, int64_t bytes, uint32_t *dst,
                        int64_t dst_words, int32_t threads, int32_t unroll,
                        int32_t grid, int32_t flags, mt_stream_t stream) {
    if (bytes < 0 || bytes % 16 != 0 || bad_block(threads) || grid < 0 ||
        dst_words < 0 || (flags & ~MT_PLAN_PDL) != 0)
        return MT_ERR_INVALID_ARGUMENT;
    ReadFn fn = read_kernel_for(unroll);
    if (fn == nullptr) return MT_ERR_INVALID_ARGUMENT;
    if (bytes == 0) return MT_OK;
    if (src == nullptr || dst == nullptr ||
        (reinterpret_cast<uintptr_t>(src) & 15) != 0 ||
        (reinterpret_cast<uintptr_t>(dst) & 3) != 0)
        return MT_ERR_INVALID_ARGUMENT;
    if (grid > 0 && grid > dst_words) return MT_ERR_INVALID_ARGUMENT;
    int g = grid;
    cudaError_t e =
        resolve_grid(reinterpret_cast<const void *>(fn), threads, &g);
    if (e != cudaSuccess) return status_from_cuda(e);
    if (g > dst_words) return MT_ERR_INVALID_ARGUMENT;
    const uint4 *sp = static_cast<const uint4 *>(src);
    unsigned *dp = dst;
    int64_t n = bytes / 16;
    int prefetch = (flags & MT_PLAN_PDL) != 0;
    void *args[] = {&sp, &dp, &n, &prefetch};
    return status_from_cuda(launch_pdl(reinterpret_cast<const void *>(fn),
                                       g, threads, args,
                                       (cudaStream_t)stream));
}

mt_status mt_probe_empty(int32_t threads, int32_t grid, mt_stream_t stream) {
    if (bad_block(threads) || grid < 0) return MT_ERR_INVALID_ARGUMENT;
    const void *fn = reinterpret_cast<const void *>(probe_empty_kernel);
    int g = grid;
    cudaError_t e = resolve_grid(fn, threads, &g);
    if (e == cudaSuccess)
        e = launch_pdl(fn, g, threads, nullptr, (cudaStream_t)stream);
    return status_from_cuda(e);
}

}  // extern "C"
