// api.cpp -- the C ABI: argument checks, plan choice, alignment mode, grid
// sizing and launch.  Calls allocate nothing and never synchronise.
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <mutex>
#include <unordered_map>

#include "mt_internal.h"

namespace mt {
namespace {

thread_local int g_last_cuda_error = 0;

mt_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return MT_OK;
    (void)cudaGetLastError();  // do not leave the error for the caller
    g_last_cuda_error = (int)e;
    return e == cudaErrorLaunchOutOfResources ? MT_ERR_OUT_OF_RESOURCES
                                              : MT_ERR_CUDA;
}

bool misaligned4(const void *p) {
    return (reinterpret_cast<uintptr_t>(p) & 3u) != 0;
}

// SM count per device, queried once.
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];

cudaError_t sm_count(int dev, int *out) {
    if (dev >= 0 && dev < kMaxDevices) {
        int v = g_sm_count[dev].load(std::memory_order_relaxed);
        if (v > 0) {
            *out = v;
            return cudaSuccess;
        }
    }
    int v = 0;
    cudaError_t e =
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices)
        g_sm_count[dev].store(v, std::memory_order_relaxed);
    *out = v;
    return cudaSuccess;
}

// Resident CTAs per SM for a (device, op, kernel variant, block size).
std::mutex g_occ_mu;
std::unordered_map<uint64_t, int> g_occ;

typedef cudaError_t (*LaunchFn)(const mt_plan_t &, const KArgs &, bool,
                                cudaStream_t, int *);
typedef cudaError_t (*OccFn)(const mt_plan_t &, bool, int *);

const LaunchFn kLaunch[OP_COUNT] = {
    launch_rmsnorm, launch_layernorm, launch_residual_layernorm,
    launch_softmax, launch_row_sum,   launch_cross_entropy};
const OccFn kOcc[OP_COUNT] = {
    launch_rmsnorm_occupancy,   launch_layernorm_occupancy,
    launch_residual_layernorm_occupancy, launch_softmax_occupancy,
    launch_row_sum_occupancy,   launch_cross_entropy_occupancy};

cudaError_t blocks_per_sm(int dev, int op, const mt_plan_t &p, bool aligned,
                          int *out) {
    const uint64_t key =
        ((uint64_t)(dev & 0xff) << 56) | ((uint64_t)op << 48) |
        ((uint64_t)p.path << 44) | ((uint64_t)p.values_per_thread << 40) |
        ((uint64_t)(p.chunks & 0xff) << 32) | ((uint64_t)aligned << 31) |
        (uint64_t)(p.threads_per_row * p.rows_per_block);
    {
        std::lock_guard<std::mutex> lk(g_occ_mu);
        auto it = g_occ.find(key);
        if (it != g_occ.end()) {
            *out = it->second;
            return cudaSuccess;
        }
    }
    int n = 0;
    cudaError_t e = kOcc[op](p, aligned, &n);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_occ_mu);
    g_occ[key] = n;
    *out = n;
    return cudaSuccess;
}

// Pointers accessed with V-wide vectors besides x (NULL entries ignored).
struct VecPtrs {
    const void *y = nullptr, *res = nullptr, *h = nullptr, *w = nullptr,
               *b = nullptr;
};

mt_status dispatch(int op, KArgs a, const VecPtrs &vp,
                   const mt_plan_t *forced, cudaStream_t stream) {
    mt_plan_t p;
    if (forced != nullptr) {
        p = *forced;
        const mt_status st = plan_check(op, a.cols, p);
        if (st != MT_OK) return st;
    } else {
        const mt_status st = plan_lookup(op, a.rows, a.cols, &p);
        if (st != MT_OK) return st;
    }
    if (a.rows == 0) return MT_OK;

    // Alignment mode: the "aligned" kernels need every row of every
    // vector-accessed pointer to start on a 4V-byte boundary.
    const int V = p.values_per_thread;
    const uintptr_t mask = (uintptr_t)(4 * V - 1);
    auto al = [&](const void *q) {
        return q == nullptr || (reinterpret_cast<uintptr_t>(q) & mask) == 0;
    };
    const bool aligned = V == 1 || (a.cols % V == 0 && al(a.x) && al(vp.y) &&
                                    al(vp.res) && al(vp.h) && al(vp.w) &&
                                    al(vp.b));
    // Unaligned kernels: a pointer keeps x's phase when its distance from x
    // is a multiple of 4V bytes; then its row bodies are aligned too.
    auto phase = [&](const void *q) -> int32_t {
        if (q == nullptr) return 0;
        return ((reinterpret_cast<uintptr_t>(q) -
                 reinterpret_cast<uintptr_t>(a.x)) & mask) == 0;
    };
    a.y_vec = phase(vp.y);
    a.h_vec = phase(vp.h);
    a.r_vec = phase(vp.res);
    a.W = p.threads_per_row;
    int l = 0;
    while ((1 << l) < a.W) ++l;
    a.log2W = l;
    a.B = p.rows_per_block;
    a.pdl = (p.flags & MT_PLAN_PDL) ? 1 : 0;
    a.prefetch_next = (p.flags & MT_PLAN_PREFETCH_NEXT) ? 1 : 0;

    const int64_t ngroups = (a.rows + a.B - 1) / a.B;
    int64_t grid = p.grid;
    if (grid == 0) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return cuda_status(e);
        int sms = 0, bps = 0;
        e = sm_count(dev, &sms);
        if (e != cudaSuccess) return cuda_status(e);
        e = blocks_per_sm(dev, op, p, aligned, &bps);
        if (e != cudaSuccess) return cuda_status(e);
        if (bps < 1) return MT_ERR_OUT_OF_RESOURCES;
        grid = (int64_t)sms * bps;
    }
    if (grid > ngroups) grid = ngroups;
    if (grid > 0x7fffffff) grid = 0x7fffffff;
    p.grid = (int32_t)grid;

    cudaError_t e = kLaunch[op](p, a, aligned, stream, nullptr);
    return cuda_status(e);
}

mt_status check_shape(int64_t rows, int64_t cols) {
    if (rows < 0 || cols < 1 || cols > 0x7fffffff) return MT_ERR_INVALID_ARGUMENT;
    if (rows > 0 && rows > INT64_MAX / cols) return MT_ERR_INVALID_ARGUMENT;
    return MT_OK;
}

KArgs base_args(const float *x, int64_t rows, int64_t cols) {
    KArgs a = {};
    a.x = x;
    a.rows = rows;
    a.cols = (int32_t)cols;
    return a;
}

}  // namespace
}  // namespace mt

using mt::check_shape;
using mt::dispatch;
using mt::misaligned4;
using mt::VecPtrs;

extern "C" {

mt_status mt_rmsnorm_f32_with_plan(const float *x, const float *weight,
                                   float *y, int64_t rows, int64_t cols,
                                   float eps, mt_stream_t stream,
                                   const mt_plan_t *plan) {
    if (mt_status st = check_shape(rows, cols)) return st;
    if (rows > 0 && (!x || !y))
        return MT_ERR_INVALID_ARGUMENT;
    if (misaligned4(x) ||
        misaligned4(y) ||
        misaligned4(weight))
        return MT_ERR_INVALID_ARGUMENT;
    mt::KArgs a = mt::base_args(x, rows, cols);
    a.w = weight;
    a.y = y;
    a.eps = eps;
    VecPtrs vp;
    vp.y = y;
    vp.w = weight;
    return dispatch(mt::OP_RMSNORM, a, vp, plan, (cudaStream_t)stream);
}

mt_status mt_rmsnorm_f32(const float *x, const float *weight, float *y,
                         int64_t rows, int64_t cols, float eps,
                         mt_stream_t stream) {
    return mt_rmsnorm_f32_with_plan(x, weight, y, rows, cols, eps, stream,
                                    nullptr);
}

mt_status mt_layernorm_f32_with_plan(const float *x, const float *gamma,
                                     const float *beta, float *y,
                                     int64_t rows, int64_t cols, float eps,
                                     mt_stream_t stream,
                                     const mt_plan_t *plan) {
    if (mt_status st = check_shape(rows, cols)) return st;
    if (rows > 0 && (!x || !y))
        return MT_ERR_INVALID_ARGUMENT;
    if (misaligned4(x) ||
        misaligned4(y) ||
        misaligned4(gamma) ||
        misaligned4(beta))
        return MT_ERR_INVALID_ARGUMENT;
    mt::KArgs a = mt::base_args(x, rows, cols);
    a.w = gamma;
    a.b = beta;
    a.y = y;
    a.eps = eps;
    VecPtrs vp;
    vp.y = y;
    vp.w = gamma;
    vp.b = beta;
    return dispatch(mt::OP_LAYERNORM, a, vp, plan, (cudaStream_t)stream);
}

mt_status mt_layernorm_f32(const float *x, const float *gamma,
                           const float *beta, float *y, int64_t rows,
                           int64_t cols, float eps, mt_stream_t stream) {
    return mt_layernorm_f32_with_plan(x, gamma, beta, y, rows, cols, eps,
                                      stream, nullptr);
}

mt_status mt_residual_layernorm_f32_with_plan(
    const float *x, const float *residual, const float *gamma,
    const float *beta, float *y, float *h_out, int64_t rows, int64_t cols,
    float eps, mt_stream_t stream, const mt_plan_t *plan) {
    if (mt_status st = check_shape(rows, cols)) return st;
    if (rows > 0 && (!x || !residual || !y))
        return MT_ERR_INVALID_ARGUMENT;
    if (misaligned4(x) ||
        misaligned4(residual) ||
        misaligned4(y) ||
        misaligned4(h_out) ||
        misaligned4(gamma) ||
        misaligned4(beta))
        return MT_ERR_INVALID_ARGUMENT;
    mt::KArgs a = mt::base_args(x, rows, cols);
    a.res = residual;
    a.w = gamma;
    a.b = beta;
    a.y = y;
    a.h = h_out;
    a.eps = eps;
    VecPtrs vp;
    vp.y = y;
    vp.res = residual;
    vp.h = h_out;
    vp.w = gamma;
    vp.b = beta;
    return dispatch(mt::OP_RESIDUAL_LAYERNORM, a, vp, plan,
                    (cudaStream_t)stream);
}

mt_status mt_residual_layernorm_f32(const float *x, const float *residual,
                                    const float *gamma, const float *beta,
                                    float *y, float *h_out, int64_t rows,
                                    int64_t cols, float eps,
                                    mt_stream_t stream) {
    return mt_residual_layernorm_f32_with_plan(x, residual, gamma, beta, y,
                                               h_out, rows, cols, eps, stream,
                                               nullptr);
}

mt_status mt_softmax_f32_with_plan(const float *x, float *y, int64_t rows,
                                   int64_t cols, mt_stream_t stream,
                                   const mt_plan_t *plan) {
    if (mt_status st = check_shape(rows, cols)) return st;
    if (rows > 0 && (!x || !y))
        return MT_ERR_INVALID_ARGUMENT;
    if (misaligned4(x) ||
        misaligned4(y))
        return MT_ERR_INVALID_ARGUMENT;
    mt::KArgs a = mt::base_args(x, rows, cols);
    a.y = y;
    VecPtrs vp;
    vp.y = y;
    return dispatch(mt::OP_SOFTMAX, a, vp, plan, (cudaStream_t)stream);
}

mt_status mt_softmax_f32(const float *x, float *y, int64_t rows,
                         int64_t cols, mt_stream_t stream) {
    return mt_softmax_f32_with_plan(x, y, rows, cols, stream, nullptr);
}

mt_status mt_row_sum_f32_with_plan(const float *x, float *out, int64_t rows,
                                   int64_t cols, mt_stream_t stream,
                                   const mt_plan_t *plan) {
    if (mt_status st = check_shape(rows, cols)) return st;
    if (rows > 0 && (!x || !out))
        return MT_ERR_INVALID_ARGUMENT;
    if (misaligned4(x) ||
        misaligned4(out))
        return MT_ERR_INVALID_ARGUMENT;
    mt::KArgs a = mt::base_args(x, rows, cols);
    a.out = out;
    return dispatch(mt::OP_ROW_SUM, a, VecPtrs(), plan,
                    (cudaStream_t)stream);
}

mt_status mt_row_sum_f32(const float *x, float *out, int64_t rows,
                         int64_t cols, mt_stream_t stream) {
    return mt_row_sum_f32_with_plan(x, out, rows, cols, stream, nullptr);
}

mt_status mt_cross_entropy_f32_with_plan(const float *logits,
                                         const int32_t *labels, float *loss,
                                         float *mean_loss, int64_t rows,
                                         int64_t cols, mt_stream_t stream,
                                         const mt_plan_t *plan) {
    if (mt_status st = check_shape(rows, cols)) return st;
    if (rows > 0 && (!logits || !labels || !loss))
        return MT_ERR_INVALID_ARGUMENT;
    if (misaligned4(logits) ||
        misaligned4(labels) ||
        misaligned4(loss) ||
        misaligned4(mean_loss))
        return MT_ERR_INVALID_ARGUMENT;
    mt::KArgs a = mt::base_args(logits, rows, cols);
    a.labels = labels;
    a.out = loss;
    const mt_status st = dispatch(mt::OP_CROSS_ENTROPY, a, VecPtrs(), plan,
                                  (cudaStream_t)stream);
    if (st != MT_OK || rows == 0 || mean_loss == nullptr) return st;
    return mt::cuda_status(
        mt::launch_mean(loss, mean_loss, rows, (cudaStream_t)stream));
}

mt_status mt_cross_entropy_f32(const float *logits, const int32_t *labels,
                               float *loss, float *mean_loss, int64_t rows,
                               int64_t cols, mt_stream_t stream) {
    return mt_cross_entropy_f32_with_plan(logits, labels, loss, mean_loss,
                                          rows, cols, stream, nullptr);
}

const char *mt_status_string(mt_status s) {
    switch (s) {
        case MT_OK: return "MT_OK";
        case MT_ERR_INVALID_ARGUMENT: return "MT_ERR_INVALID_ARGUMENT";
        case MT_ERR_UNSUPPORTED: return "MT_ERR_UNSUPPORTED";
        case MT_ERR_OUT_OF_RESOURCES: return "MT_ERR_OUT_OF_RESOURCES";
        case MT_ERR_CUDA: return "MT_ERR_CUDA";
    }
    return "MT_ERR_UNKNOWN";
}

int mt_last_cuda_error(void) { return mt::g_last_cuda_error; }

}  // extern "C"
