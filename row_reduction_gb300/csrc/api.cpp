// api.cpp -- the C ABI: argument checks, plan choice, alignment mode, grid
// sizing and launch.  Calls allocate nothing and never synchronise.
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <mutex>
#include <unordered_map>
#include <unordered_set>

#include "mt_internal.h"

namespace mt {
namespace {
thread_local int g_last_cuda_error = 0;
}  // namespace

mt_status status_from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return MT_OK;
    (void)cudaGetLastError();  // do not leave the error for the caller
    g_last_cuda_error = (int)e;
    return e == cudaErrorLaunchOutOfResources ? MT_ERR_OUT_OF_RESOURCES
                                              : MT_ERR_CUDA;
}

// Kernels that have been allowed clusters beyond the portable size, per
// device: the attribute is set once per (device, kernel), not per launch.
namespace {
std::mutex g_nonportable_mu;
std::unordered_set<uint64_t> g_nonportable;
}  // namespace

std::mutex g_stage_smem_mu;
std::unordered_set<uint64_t> g_stage_smem;

cudaError_t allow_stage_smem(const void *kernel) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t key = (reinterpret_cast<uintptr_t>(kernel) << 8) ^
                         (uint64_t)(dev & 0xff);
    std::lock_guard<std::mutex> lk(g_stage_smem_mu);
    if (g_stage_smem.count(key)) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kStageMaxRunBytes);
    if (e == cudaSuccess) g_stage_smem.insert(key);
    return e;
}

cudaError_t allow_nonportable_cluster(const void *kernel) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t key = (reinterpret_cast<uintptr_t>(kernel) << 8) ^
                         (uint64_t)(dev & 0xff);
    std::lock_guard<std::mutex> lk(g_nonportable_mu);
    if (g_nonportable.count(key)) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel,
                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess) g_nonportable.insert(key);
    return e;
}

namespace {

mt_status cuda_status(cudaError_t e) { return status_from_cuda(e); }

bool misaligned(const void *p, int bytes) {
    return (reinterpret_cast<uintptr_t>(p) & (uintptr_t)(bytes - 1)) != 0;
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

typedef cudaError_t (*LaunchFn)(const mt_plan_t &, const KArgs &, int,
                                cudaStream_t);
typedef cudaError_t (*OccFn)(const mt_plan_t &, int, int64_t, int *);

#define MT_ROW(op)                                                           \
    {launch_##op##_f32, launch_##op##_f16, launch_##op##_bf16}
#define MT_OCC_ROW(op)                                                       \
    {launch_##op##_f32_occupancy, launch_##op##_f16_occupancy,               \
     launch_##op##_bf16_occupancy}
const LaunchFn kLaunch[OP_COUNT][DT_COUNT] = {
    MT_ROW(rmsnorm),       MT_ROW(layernorm),
    MT_ROW(residual_layernorm), MT_ROW(softmax),
    MT_ROW(row_sum),       MT_ROW(cross_entropy),
    MT_ROW(residual_rmsnorm), MT_ROW(log_softmax)};
const OccFn kOcc[OP_COUNT][DT_COUNT] = {
    MT_OCC_ROW(rmsnorm),       MT_OCC_ROW(layernorm),
    MT_OCC_ROW(residual_layernorm), MT_OCC_ROW(softmax),
    MT_OCC_ROW(row_sum),       MT_OCC_ROW(cross_entropy),
    MT_OCC_ROW(residual_rmsnorm), MT_OCC_ROW(log_softmax)};
typedef cudaError_t (*TimeoutFn)(unsigned long long *);
#define MT_TO_ROW(op)                                                        \
    {launch_##op##_f32_timeouts, launch_##op##_f16_timeouts,                 \
     launch_##op##_bf16_timeouts}
const TimeoutFn kTimeouts[OP_COUNT][DT_COUNT] = {
    MT_TO_ROW(rmsnorm),       MT_TO_ROW(layernorm),
    MT_TO_ROW(residual_layernorm), MT_TO_ROW(softmax),
    MT_TO_ROW(row_sum),       MT_TO_ROW(cross_entropy),
    MT_TO_ROW(residual_rmsnorm), MT_TO_ROW(log_softmax)};
#undef MT_ROW
#undef MT_OCC_ROW
#undef MT_TO_ROW

// Resident CTAs per SM for a (device, op, dtype, kernel variant, block).
std::mutex g_occ_mu;
std::unordered_map<uint64_t, int> g_occ;

cudaError_t blocks_per_sm(int dev, int op, int dtype, const mt_plan_t &p,
                          int mode, int64_t cols, int *out) {
    // Staged plans: the shared memory of a run (whole KiB) and the cluster
    // size join the key.
    uint64_t stage = 0;
    if (p.path == MT_PATH_STAGE)
        stage = ((uint64_t)(stage_run_bytes(cols, dtype_size(dtype),
                                            p.cluster > 1 ? p.cluster : 1) /
                            1024) << 11) |
                (uint64_t)(p.cluster & 31) << 19;
    const uint64_t key =
        ((uint64_t)(dev & 0xff) << 56) | ((uint64_t)op << 50) |
        ((uint64_t)dtype << 46) | ((uint64_t)p.path << 44) |
        ((uint64_t)p.values_per_thread << 40) |
        ((uint64_t)(p.chunks & 0xff) << 32) | ((uint64_t)mode << 30) |
        (uint64_t)(p.threads_per_row * p.rows_per_block) | stage;
    {
        std::lock_guard<std::mutex> lk(g_occ_mu);
        auto it = g_occ.find(key);
        if (it != g_occ.end()) {
            *out = it->second;
            return cudaSuccess;
        }
    }
    int n = 0;
    cudaError_t e = kOcc[op][dtype](p, mode, cols, &n);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_occ_mu);
    g_occ[key] = n;
    *out = n;
    return cudaSuccess;
}

// Arguments of one call.
struct Call {
    int op = 0, dtype = 0;
    const void *x = nullptr, *res = nullptr, *w = nullptr, *b = nullptr;
    const int32_t *labels = nullptr;
    void *y = nullptr, *h = nullptr;
    float *out = nullptr, *mean = nullptr;
    int64_t rows = 0, cols = 0;
    float eps = 0.f;
    int32_t ignore_index = MT_NO_IGNORE_INDEX;
};

// Which pointers each operator takes (the others must be NULL), and which
// of them must be non-NULL when rows > 0.
enum : unsigned {
    U_RES = 1, U_W = 2, U_B = 4, U_LABELS = 8, U_Y = 16, U_H = 32,
    U_OUT = 64, U_MEAN = 128
};
unsigned uses(int op) {
    switch (op) {
        case OP_RMSNORM: return U_W | U_Y;
        case OP_LAYERNORM: return U_W | U_B | U_Y;
        case OP_RESIDUAL_LAYERNORM: return U_RES | U_W | U_B | U_Y | U_H;
        case OP_SOFTMAX: return U_Y;
        case OP_ROW_SUM: return U_OUT;
        case OP_CROSS_ENTROPY: return U_LABELS | U_OUT | U_MEAN;
        case OP_RESIDUAL_RMSNORM: return U_RES | U_W | U_Y | U_H;
        case OP_LOG_SOFTMAX: return U_Y;
    }
    return 0;
}
unsigned required(int op) {
    switch (op) {
        case OP_RMSNORM:
        case OP_LAYERNORM:
        case OP_SOFTMAX:
        case OP_LOG_SOFTMAX: return U_Y;
        case OP_RESIDUAL_LAYERNORM:
        case OP_RESIDUAL_RMSNORM: return U_RES | U_Y;
        case OP_ROW_SUM: return U_OUT;
        case OP_CROSS_ENTROPY: return U_LABELS | U_OUT;
    }
    return 0;
}

mt_status validate(const Call &c) {
    if (c.op < 0 || c.op >= OP_COUNT || c.dtype < 0 || c.dtype >= DT_COUNT)
        return MT_ERR_INVALID_ARGUMENT;
    if (c.rows < 0 || c.cols < 1 || c.cols > 0x7fffffff)
        return MT_ERR_INVALID_ARGUMENT;
    if (c.rows > 0 && c.rows > INT64_MAX / c.cols)
        return MT_ERR_INVALID_ARGUMENT;
    const unsigned present = (c.res ? U_RES : 0) | (c.w ? U_W : 0) |
                             (c.b ? U_B : 0) | (c.labels ? U_LABELS : 0) |
                             (c.y ? U_Y : 0) | (c.h ? U_H : 0) |
                             (c.out ? U_OUT : 0) | (c.mean ? U_MEAN : 0);
    if (present & ~uses(c.op)) return MT_ERR_INVALID_ARGUMENT;
    const unsigned req = required(c.op);
    if (c.rows > 0 && (!c.x || (present & req) != req))
        return MT_ERR_INVALID_ARGUMENT;
    const int es = dtype_size(c.dtype);
    if (misaligned(c.x, es) || misaligned(c.res, es) || misaligned(c.w, es) ||
        misaligned(c.b, es) || misaligned(c.y, es) || misaligned(c.h, es) ||
        misaligned(c.labels, 4) || misaligned(c.out, 4) ||
        misaligned(c.mean, 4))
        return MT_ERR_INVALID_ARGUMENT;
    return MT_OK;
}

mt_status run(const Call &c, const mt_plan_t *forced, cudaStream_t stream) {
    if (mt_status st = validate(c)) return st;
    mt_plan_t p;
    if (forced != nullptr) {
        p = *forced;
        if (mt_status st = plan_check(c.op, c.dtype, c.cols, p)) return st;
    } else {
        if (mt_status st = plan_lookup(c.op, c.dtype, c.rows, c.cols, &p))
            return st;
    }
    if (c.rows == 0) return MT_OK;

    KArgs a = {};
    a.x = c.x;
    a.res = c.res;
    a.w = c.w;
    a.b = c.b;
    a.y = c.y;
    a.h = c.h;
    a.out = c.out;
    a.labels = c.labels;
    a.rows = c.rows;
    a.cols = (int32_t)c.cols;
    a.eps = c.eps;
    a.ignore_index = c.ignore_index;
    a.has_ignore = c.ignore_index != MT_NO_IGNORE_INDEX;

    // Alignment mode: the "aligned" kernels need every row of every
    // vector-accessed pointer to start on a V*element-size boundary.  A
    // pack of one FP32 value is always aligned.
    const int V = p.values_per_thread;
    const int es = dtype_size(c.dtype);
    const uintptr_t mask = (uintptr_t)(V * es - 1);
    auto al = [&](const void *q) {
        return q == nullptr || (reinterpret_cast<uintptr_t>(q) & mask) == 0;
    };
    const bool aligned = (V == 1 && es == 4) ||
                         (c.cols % V == 0 && al(c.x) && al(c.y) &&
                          al(c.res) && al(c.h) && al(c.w) && al(c.b));
    // The staged path copies rows with 16-byte bulk copies, so it needs
    // aligned rows.  A forced staged plan on other rows is refused; the
    // table's staged plan gives way to the loop path with the same threads
    // (at most the loop path's limit), cluster and flags.
    if (p.path == MT_PATH_STAGE && !aligned) {
        if (forced != nullptr) return MT_ERR_INVALID_ARGUMENT;
        p.path = MT_PATH_LOOP;
        p.chunks = 0;
        if (p.threads_per_row > kLoopMaxThreads)
            p.threads_per_row = kLoopMaxThreads;
    }
    // Unaligned kernels: a pointer keeps x's phase when its distance from x
    // is a multiple of V elements; then its row bodies are aligned too.
    auto phase = [&](const void *q) -> int32_t {
        if (q == nullptr) return 0;
        return ((reinterpret_cast<uintptr_t>(q) -
                 reinterpret_cast<uintptr_t>(c.x)) & mask) == 0;
    };
    a.y_vec = phase(c.y);
    a.h_vec = phase(c.h);
    a.r_vec = phase(c.res);
    // Whole tiles: every pack of every row exists and every parameter
    // vector the operator reads is present, so the kernel needs no guard.
    const bool params =
        (c.op == OP_RMSNORM || c.op == OP_RESIDUAL_RMSNORM)
            ? c.w != nullptr
            : (c.op == OP_LAYERNORM || c.op == OP_RESIDUAL_LAYERNORM)
                  ? (c.w != nullptr && c.b != nullptr)
                  : true;
    const bool full = (p.flags & MT_PLAN_WHOLE_TILES) && aligned && params &&
                      p.path == MT_PATH_REGISTERS && p.cluster <= 1 &&
                      (int64_t)p.threads_per_row * V * p.chunks == c.cols &&
                      c.rows % p.rows_per_block == 0;
    const int mode = full ? KM_FULL : (aligned ? KM_ALIGNED : KM_UNALIGNED);
    a.W = p.threads_per_row;
    int l = 0;
    while ((1 << l) < a.W) ++l;
    a.log2W = l;
    a.B = p.rows_per_block;
    a.pdl = (p.flags & MT_PLAN_PDL) ? 1 : 0;
    a.prefetch_next = (p.flags & MT_PLAN_PREFETCH_NEXT) ? 1 : 0;
    a.csize = p.cluster > 1 ? p.cluster : 1;
    a.pieces = p.path == MT_PATH_STAGE ? p.chunks : 0;
    const int64_t C = a.csize;

    // Row groups are processed by CTAs, or by clusters of C CTAs.
    const int64_t ngroups = (a.rows + a.B - 1) / a.B;
    int64_t grid = p.grid / C;  // in units of row-group workers
    if (grid == 0) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return cuda_status(e);
        int sms = 0, bps = 0;
        e = sm_count(dev, &sms);
        if (e != cudaSuccess) return cuda_status(e);
        e = blocks_per_sm(dev, c.op, c.dtype, p, mode, c.cols, &bps);
        if (e != cudaSuccess) return cuda_status(e);
        if (bps < 1) return MT_ERR_OUT_OF_RESOURCES;
        grid = (int64_t)sms * bps / C;
        if (grid < 1) grid = 1;
    }
    if (grid > ngroups) grid = ngroups;
    if (grid * C > 0x7fffffff) grid = 0x7fffffff / C;
    p.grid = (int32_t)(grid * C);

    if (mt_status st =
            cuda_status(kLaunch[c.op][c.dtype](p, a, mode, stream)))
        return st;
    if (c.op == OP_CROSS_ENTROPY && c.mean != nullptr)
        return cuda_status(launch_mean(c.out, c.mean, c.rows, c.labels,
                                       a.ignore_index, a.has_ignore, stream));
    return MT_OK;
}

Call make_call(int op, int dtype, const void *x, int64_t rows, int64_t cols) {
    Call c;
    c.op = op;
    c.dtype = dtype;
    c.x = x;
    c.rows = rows;
    c.cols = cols;
    return c;
}

mt_status rmsnorm_call(int dt, const void *x, const void *w, void *y,
                       int64_t rows, int64_t cols, float eps, mt_stream_t s,
                       const mt_plan_t *plan) {
    Call c = make_call(OP_RMSNORM, dt, x, rows, cols);
    c.w = w;
    c.y = y;
    c.eps = eps;
    return run(c, plan, (cudaStream_t)s);
}

mt_status layernorm_call(int dt, const void *x, const void *g,
                         const void *b, void *y, int64_t rows, int64_t cols,
                         float eps, mt_stream_t s, const mt_plan_t *plan) {
    Call c = make_call(OP_LAYERNORM, dt, x, rows, cols);
    c.w = g;
    c.b = b;
    c.y = y;
    c.eps = eps;
    return run(c, plan, (cudaStream_t)s);
}

mt_status resln_call(int dt, const void *x, const void *r, const void *g,
                     const void *b, void *y, void *h, int64_t rows,
                     int64_t cols, float eps, mt_stream_t s,
                     const mt_plan_t *plan) {
    Call c = make_call(OP_RESIDUAL_LAYERNORM, dt, x, rows, cols);
    c.res = r;
    c.w = g;
    c.b = b;
    c.y = y;
    c.h = h;
    c.eps = eps;
    return run(c, plan, (cudaStream_t)s);
}

mt_status softmax_call(int dt, const void *x, void *y, int64_t rows,
                       int64_t cols, mt_stream_t s, const mt_plan_t *plan) {
    Call c = make_call(OP_SOFTMAX, dt, x, rows, cols);
    c.y = y;
    return run(c, plan, (cudaStream_t)s);
}

mt_status row_sum_call(int dt, const void *x, float *out, int64_t rows,
                       int64_t cols, mt_stream_t s, const mt_plan_t *plan) {
    Call c = make_call(OP_ROW_SUM, dt, x, rows, cols);
    c.out = out;
    return run(c, plan, (cudaStream_t)s);
}

mt_status ce_call(int dt, const void *x, const int32_t *labels, float *loss,
                  float *mean, int64_t rows, int64_t cols, mt_stream_t s,
                  const mt_plan_t *plan,
                  int32_t ignore_index = MT_NO_IGNORE_INDEX) {
    Call c = make_call(OP_CROSS_ENTROPY, dt, x, rows, cols);
    c.labels = labels;
    c.out = loss;
    c.mean = mean;
    c.ignore_index = ignore_index;
    return run(c, plan, (cudaStream_t)s);
}

mt_status res_rms_call(int dt, const void *x, const void *r, const void *w,
                       void *y, void *h, int64_t rows, int64_t cols,
                       float eps, mt_stream_t s, const mt_plan_t *plan) {
    Call c = make_call(OP_RESIDUAL_RMSNORM, dt, x, rows, cols);
    c.res = r;
    c.w = w;
    c.y = y;
    c.h = h;
    c.eps = eps;
    return run(c, plan, (cudaStream_t)s);
}

mt_status log_softmax_call(int dt, const void *x, void *y, int64_t rows,
                           int64_t cols, mt_stream_t s,
                           const mt_plan_t *plan) {
    Call c = make_call(OP_LOG_SOFTMAX, dt, x, rows, cols);
    c.y = y;
    return run(c, plan, (cudaStream_t)s);
}

}  // namespace
}  // namespace mt

using namespace mt;

extern "C" {

// ---- FP32 -------------------------------------------------------------------
mt_status mt_rmsnorm_f32_with_plan(const float *x, const float *weight,
                                   float *y, int64_t rows, int64_t cols,
                                   float eps, mt_stream_t stream,
                                   const mt_plan_t *plan) {
    return rmsnorm_call(MT_DTYPE_F32, x, weight, y, rows, cols, eps, stream,
                        plan);
}
mt_status mt_rmsnorm_f32(const float *x, const float *weight, float *y,
                         int64_t rows, int64_t cols, float eps,
                         mt_stream_t stream) {
    return rmsnorm_call(MT_DTYPE_F32, x, weight, y, rows, cols, eps, stream,
                        nullptr);
}
mt_status mt_layernorm_f32_with_plan(const float *x, const float *gamma,
                                     const float *beta, float *y,
                                     int64_t rows, int64_t cols, float eps,
                                     mt_stream_t stream,
                                     const mt_plan_t *plan) {
    return layernorm_call(MT_DTYPE_F32, x, gamma, beta, y, rows, cols, eps,
                          stream, plan);
}
mt_status mt_layernorm_f32(const float *x, const float *gamma,
                           const float *beta, float *y, int64_t rows,
                           int64_t cols, float eps, mt_stream_t stream) {
    return layernorm_call(MT_DTYPE_F32, x, gamma, beta, y, rows, cols, eps,
                          stream, nullptr);
}
mt_status mt_residual_layernorm_f32_with_plan(
    const float *x, const float *residual, const float *gamma,
    const float *beta, float *y, float *h_out, int64_t rows, int64_t cols,
    float eps, mt_stream_t stream, const mt_plan_t *plan) {
    return resln_call(MT_DTYPE_F32, x, residual, gamma, beta, y, h_out, rows,
                      cols, eps, stream, plan);
}
mt_status mt_residual_layernorm_f32(const float *x, const float *residual,
                                    const float *gamma, const float *beta,
                                    float *y, float *h_out, int64_t rows,
                                    int64_t cols, float eps,
                                    mt_stream_t stream) {
    return resln_call(MT_DTYPE_F32, x, residual, gamma, beta, y, h_out, rows,
                      cols, eps, stream, nullptr);
}
mt_status mt_softmax_f32_with_plan(const float *x, float *y, int64_t rows,
                                   int64_t cols, mt_stream_t stream,
                                   const mt_plan_t *plan) {
    return softmax_call(MT_DTYPE_F32, x, y, rows, cols, stream, plan);
}
mt_status mt_softmax_f32(const float *x, float *y, int64_t rows,
                         int64_t cols, mt_stream_t stream) {
    return softmax_call(MT_DTYPE_F32, x, y, rows, cols, stream, nullptr);
}
mt_status mt_row_sum_f32_with_plan(const float *x, float *out, int64_t rows,
                                   int64_t cols, mt_stream_t stream,
                                   const mt_plan_t *plan) {
    return row_sum_call(MT_DTYPE_F32, x, out, rows, cols, stream, plan);
}
mt_status mt_row_sum_f32(const float *x, float *out, int64_t rows,
                         int64_t cols, mt_stream_t stream) {
    return row_sum_call(MT_DTYPE_F32, x, out, rows, cols, stream, nullptr);
}
mt_status mt_cross_entropy_f32_with_plan(const float *logits,
                                         const int32_t *labels, float *loss,
                                         float *mean_loss, int64_t rows,
                                         int64_t cols, mt_stream_t stream,
                                         const mt_plan_t *plan) {
    return ce_call(MT_DTYPE_F32, logits, labels, loss, mean_loss, rows, cols,
                   stream, plan);
}
mt_status mt_cross_entropy_f32(const float *logits, const int32_t *labels,
                               float *loss, float *mean_loss, int64_t rows,
                               int64_t cols, mt_stream_t stream) {
    return ce_call(MT_DTYPE_F32, logits, labels, loss, mean_loss, rows, cols,
                   stream, nullptr);
}

mt_status mt_residual_rmsnorm_f32_with_plan(const float *x,
                                            const float *residual,
                                            const float *weight, float *y,
                                            float *h_out, int64_t rows,
                                            int64_t cols, float eps,
                                            mt_stream_t stream,
                                            const mt_plan_t *plan) {
    return res_rms_call(MT_DTYPE_F32, x, residual, weight, y, h_out, rows,
                        cols, eps, stream, plan);
}
mt_status mt_residual_rmsnorm_f32(const float *x, const float *residual,
                                  const float *weight, float *y, float *h_out,
                                  int64_t rows, int64_t cols, float eps,
                                  mt_stream_t stream) {
    return res_rms_call(MT_DTYPE_F32, x, residual, weight, y, h_out, rows,
                        cols, eps, stream, nullptr);
}
mt_status mt_log_softmax_f32_with_plan(const float *x, float *y,
                                       int64_t rows, int64_t cols,
                                       mt_stream_t stream,
                                       const mt_plan_t *plan) {
    return log_softmax_call(MT_DTYPE_F32, x, y, rows, cols, stream, plan);
}
mt_status mt_log_softmax_f32(const float *x, float *y, int64_t rows,
                             int64_t cols, mt_stream_t stream) {
    return log_softmax_call(MT_DTYPE_F32, x, y, rows, cols, stream, nullptr);
}
mt_status mt_cross_entropy_ignore_f32(const float *logits,
                                      const int32_t *labels,
                                      int32_t ignore_index, float *loss,
                                      float *mean_loss, int64_t rows,
                                      int64_t cols, mt_stream_t stream) {
    return ce_call(MT_DTYPE_F32, logits, labels, loss, mean_loss, rows, cols,
                   stream, nullptr, ignore_index);
}

// ---- FP16 / BF16 ------------------------------------------------------------
#define MT_HALF_ENTRY_POINTS(suffix, DT, TY)                                  \
    mt_status mt_rmsnorm_##suffix(const TY *x, const TY *weight, TY *y,      \
                                  int64_t rows, int64_t cols, float eps,     \
                                  mt_stream_t stream) {                      \
        return rmsnorm_call(DT, x, weight, y, rows, cols, eps, stream,       \
                            nullptr);                                        \
    }                                                                        \
    mt_status mt_layernorm_##suffix(const TY *x, const TY *gamma,            \
                                    const TY *beta, TY *y, int64_t rows,     \
                                    int64_t cols, float eps,                 \
                                    mt_stream_t stream) {                    \
        return layernorm_call(DT, x, gamma, beta, y, rows, cols, eps,        \
                              stream, nullptr);                              \
    }                                                                        \
    mt_status mt_residual_layernorm_##suffix(                                \
        const TY *x, const TY *residual, const TY *gamma, const TY *beta,    \
        TY *y, TY *h_out, int64_t rows, int64_t cols, float eps,             \
        mt_stream_t stream) {                                                \
        return resln_call(DT, x, residual, gamma, beta, y, h_out, rows,      \
                          cols, eps, stream, nullptr);                       \
    }                                                                        \
    mt_status mt_softmax_##suffix(const TY *x, TY *y, int64_t rows,          \
                                  int64_t cols, mt_stream_t stream) {        \
        return softmax_call(DT, x, y, rows, cols, stream, nullptr);          \
    }                                                                        \
    mt_status mt_row_sum_##suffix(const TY *x, float *out, int64_t rows,     \
                                  int64_t cols, mt_stream_t stream) {        \
        return row_sum_call(DT, x, out, rows, cols, stream, nullptr);        \
    }                                                                        \
    mt_status mt_cross_entropy_##suffix(                                     \
        const TY *logits, const int32_t *labels, float *loss,                \
        float *mean_loss, int64_t rows, int64_t cols, mt_stream_t stream) {  \
        return ce_call(DT, logits, labels, loss, mean_loss, rows, cols,      \
                       stream, nullptr);                                     \
    }                                                                        \
    mt_status mt_cross_entropy_ignore_##suffix(                              \
        const TY *logits, const int32_t *labels, int32_t ignore_index,       \
        float *loss, float *mean_loss, int64_t rows, int64_t cols,           \
        mt_stream_t stream) {                                                \
        return ce_call(DT, logits, labels, loss, mean_loss, rows, cols,      \
                       stream, nullptr, ignore_index);                       \
    }                                                                        \
    mt_status mt_residual_rmsnorm_##suffix(                                  \
        const TY *x, const TY *residual, const TY *weight, TY *y, TY *h_out, \
        int64_t rows, int64_t cols, float eps, mt_stream_t stream) {         \
        return res_rms_call(DT, x, residual, weight, y, h_out, rows, cols,   \
                            eps, stream, nullptr);                           \
    }                                                                        \
    mt_status mt_log_softmax_##suffix(const TY *x, TY *y, int64_t rows,      \
                                      int64_t cols, mt_stream_t stream) {    \
        return log_softmax_call(DT, x, y, rows, cols, stream, nullptr);      \
    }
MT_HALF_ENTRY_POINTS(f16, MT_DTYPE_F16, mt_f16_t)
MT_HALF_ENTRY_POINTS(bf16, MT_DTYPE_BF16, mt_bf16_t)
#undef MT_HALF_ENTRY_POINTS

mt_status mt_row_reduce_with_plan(int op, int dtype, const void *x,
                                  const void *residual, const void *weight,
                                  const void *beta, const int32_t *labels,
                                  int32_t ignore_index, void *y, void *h_out,
                                  float *out, float *mean_loss, int64_t rows,
                                  int64_t cols, float eps, mt_stream_t stream,
                                  const mt_plan_t *plan) {
    Call c = make_call(op, dtype, x, rows, cols);
    c.res = residual;
    c.w = weight;
    c.b = beta;
    c.labels = labels;
    c.ignore_index = ignore_index;
    c.y = y;
    c.h = h_out;
    c.out = out;
    c.mean = mean_loss;
    c.eps = eps;
    return run(c, plan, (cudaStream_t)stream);
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

int mt_last_cuda_error(void) { return g_last_cuda_error; }

mt_status mt_stage_wait_timeouts(uint64_t *count) {
    if (count == nullptr) return MT_ERR_INVALID_ARGUMENT;
    uint64_t total = 0;
    for (int op = 0; op < OP_COUNT; ++op)
        for (int dt = 0; dt < DT_COUNT; ++dt) {
            unsigned long long n = 0;
            if (mt_status st = cuda_status(kTimeouts[op][dt](&n))) return st;
            total += n;
        }
    *count = total;
    return MT_OK;
}

}  // extern "C"
