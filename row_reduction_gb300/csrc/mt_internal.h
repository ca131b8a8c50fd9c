// mt_internal.h -- types shared by the C-ABI layer, the planner and the
// kernel translation units.  Not part of the public interface.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mt_rowreduce.h"

namespace mt {

enum : int {
    OP_RMSNORM = MT_OP_RMSNORM,
    OP_LAYERNORM = MT_OP_LAYERNORM,
    OP_RESIDUAL_LAYERNORM = MT_OP_RESIDUAL_LAYERNORM,
    OP_SOFTMAX = MT_OP_SOFTMAX,
    OP_ROW_SUM = MT_OP_ROW_SUM,
    OP_CROSS_ENTROPY = MT_OP_CROSS_ENTROPY,
    OP_RESIDUAL_RMSNORM = MT_OP_RESIDUAL_RMSNORM,
    OP_LOG_SOFTMAX = MT_OP_LOG_SOFTMAX,
    OP_COUNT = 8
};

enum : int {
    DT_F32 = MT_DTYPE_F32,
    DT_F16 = MT_DTYPE_F16,
    DT_BF16 = MT_DTYPE_BF16,
    DT_COUNT = 3
};

inline int dtype_size(int dt) { return dt == DT_F32 ? 4 : 2; }

// Kernel arguments; one struct for all operators (unused fields are NULL).
// Matrices and parameter vectors hold the storage type of the launch
// (FP32, FP16 or BF16); per-row outputs are always FP32.
struct KArgs {
    const void *x;         // input matrix (logits for cross-entropy)
    const void *res;       // residual (residual LayerNorm)
    const void *w;         // RMSNorm weight / LayerNorm gamma (NULL = 1)
    const void *b;         // LayerNorm beta (NULL = 0)
    void *y;               // output matrix
    void *h;               // residual LayerNorm h_out (NULL = not written)
    float *out;            // per-row output (row sum, cross-entropy loss)
    const int32_t *labels; // cross-entropy labels
    int64_t rows;
    int32_t cols;
    int32_t W;             // threads per row (power of two)
    int32_t log2W;
    int32_t B;             // rows per CTA
    float eps;
    // Cross-entropy: rows whose label equals ignore_index (when has_ignore)
    // get loss 0 and leave the mean.
    int32_t ignore_index;
    int32_t has_ignore;
    // Unaligned mode only: 1 when the pointer keeps x's 16-byte phase, so
    // its row body can use vector accesses too.
    int32_t y_vec, h_vec, r_vec;
    // Launched as a programmatic dependent: prefetch the first row group
    // into L2 before waiting on the previous grid.
    int32_t pdl;
    // Persistent CTAs prefetch their next row group into L2.
    int32_t prefetch_next;
    // CTAs per row (thread-block cluster size; 1 = no cluster).
    int32_t csize;
    // Staged path: bulk copies (and barriers) per CTA's run of the row.
    int32_t pieces;
};

// Instantiated register-path chunk counts.
constexpr int kChunkSet[] = {1, 2, 4, 8, 16};
constexpr int kNumChunkSet = 5;

// Largest CTA the register-path kernel with V*K values per thread is
// compiled for (its __launch_bounds__): 64 registers per thread at 1024
// threads leaves room for 16 values; 128 at 512 for 32; 255 at 256 for 64.
constexpr int reg_max_threads(int vk) {
    return vk <= 16 ? 1024 : (vk <= 32 ? 512 : 256);
}
// Whole-tile kernels issue every load unguarded, so the compiler hoists
// more of them at once than in the guarded kernels.  For 32 values in
// packs of 16 bytes a cap of kFullCapRegs registers lets seven 128-thread
// CTAs share an SM (one wave for 1024 rows of one CTA each); it applies to
// the operators that fit it without spilling (not the two-parameter
// LayerNorms, nor residual RMSNorm).
constexpr int kFullCapRegs = 72;
constexpr bool reg_full_capped(int op, int vk, int pack_bytes,
                               int elem_bytes) {
    return vk == 32 && pack_bytes == 16 &&
           (elem_bytes == 2 || (op != MT_OP_LAYERNORM &&
                                op != MT_OP_RESIDUAL_LAYERNORM &&
                                op != MT_OP_RESIDUAL_RMSNORM));
}
constexpr int kLoopMaxThreads = 512;
// Staged path: largest run of a row one CTA stages in shared memory (bytes)
// and the most bulk-copy pieces per run.
constexpr int64_t kStageMaxRunBytes = 200 * 1024;
constexpr int kStagePiecesMax = 8;
// Bytes of shared memory a staged CTA needs for one run of a row of `cols`
// elements of `elem` bytes split over `csize` CTAs.
inline int64_t stage_run_bytes(int64_t cols, int elem, int64_t csize) {
    const int64_t units = cols * elem / 16;
    return (units + csize - 1) / csize * 16;
}
inline bool stage_op(int op) {
    return op == MT_OP_RMSNORM || op == MT_OP_LAYERNORM ||
           op == MT_OP_SOFTMAX || op == MT_OP_LOG_SOFTMAX ||
           op == MT_OP_CROSS_ENTROPY || op == MT_OP_ROW_SUM;
}

// Kernel variants of one plan.  KM_ALIGNED: every access of the row body is
// a V-wide vector access without a head.  KM_FULL (register path, no
// cluster): aligned, and every pack of every row exists (cols = W*V*K,
// rows a multiple of B, every parameter vector present), so the kernel
// carries no bounds guard at all.
enum KMode : int { KM_UNALIGNED = 0, KM_ALIGNED = 1, KM_FULL = 2 };

// Launchers, one translation unit per (operator, storage type).  `mode`
// is a KMode; `plan.grid` is already resolved (> 0).
#define MT_DECLARE_LAUNCHER(name)                                            \
    cudaError_t name(const mt_plan_t &plan, const KArgs &a, int mode,        \
                     cudaStream_t stream);                                   \
    cudaError_t name##_occupancy(const mt_plan_t &plan, int mode,            \
                                 int64_t cols, int *blocks_per_sm);          \
    cudaError_t name##_timeouts(unsigned long long *n);
#define MT_DECLARE_OP(op)                                                    \
    MT_DECLARE_LAUNCHER(launch_##op##_f32)                                   \
    MT_DECLARE_LAUNCHER(launch_##op##_f16)                                   \
    MT_DECLARE_LAUNCHER(launch_##op##_bf16)
MT_DECLARE_OP(rmsnorm)
MT_DECLARE_OP(layernorm)
MT_DECLARE_OP(residual_layernorm)
MT_DECLARE_OP(softmax)
MT_DECLARE_OP(row_sum)
MT_DECLARE_OP(cross_entropy)
MT_DECLARE_OP(residual_rmsnorm)
MT_DECLARE_OP(log_softmax)
#undef MT_DECLARE_OP
#undef MT_DECLARE_LAUNCHER

// One-CTA fixed-order mean of `rows` per-row losses; with has_ignore, rows
// whose label is ignore_index are left out of the count (their loss is 0).
cudaError_t launch_mean(const float *loss, float *mean, int64_t rows,
                        const int32_t *labels, int32_t ignore_index,
                        int32_t has_ignore, cudaStream_t stream);

// MT_OK for cudaSuccess; otherwise records e as the calling thread's last
// CUDA error (mt_last_cuda_error), clears it and returns MT_ERR_CUDA (or
// MT_ERR_OUT_OF_RESOURCES for a launch out of resources).
mt_status status_from_cuda(cudaError_t e);

// Lets `kernel` launch with clusters beyond the portable size (16 CTAs) on
// the current device.  The attribute is set on the first call for each
// (device, kernel) and remembered, so later launches make no driver call.
cudaError_t allow_nonportable_cluster(const void *kernel);
// Lets a staged-path `kernel` take kStageMaxRunBytes of dynamic shared
// memory on the current device (set once per device and kernel, likewise).
cudaError_t allow_stage_smem(const void *kernel);

// Planner (planner.cpp).
mt_status plan_lookup(int op, int dtype, int64_t rows, int64_t cols,
                      mt_plan_t *out);
mt_status plan_check(int op, int dtype, int64_t cols, const mt_plan_t &p);

}  // namespace mt
