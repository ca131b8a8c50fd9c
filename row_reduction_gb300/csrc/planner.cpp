// planner.cpp -- launch-plan choice and legality (host only, no CUDA call).
//
// A plan fixes W (threads per row), V (consecutive values per thread per
// chunk), the register chunk count K, the rows per CTA B, the path and the
// grid.  The operators take the plan from a table of winners measured on the
// GPU (plan_table.inc, written by the package's tuner), keyed by operator and
// a (cols, rows) range; shapes outside the table fall back to a heuristic.
//
// The legality rules follow the fail-closed contract of the pages: a plan is
// checked before dispatch and an illegal one is rejected, never remapped
// ("Thread Ownership and Software Staging", §Compiler-selected communication,
// the maxTotalThreadsPerThreadgroup check; "Consecutive-worker reduction
// layout checkpoint", §Verification checkpoint: invalid widths and resource
// overflow fail closed), and the private-slot bound is enforced before a plan
// is used ("Consecutive-worker reduction layout checkpoint", §Implementation
// and semantics).
#include <stdio.h>
#include <string.h>

#include "mt_internal.h"

namespace mt {
namespace {

struct PlanEntry {
    int op;
    int dtype;
    int64_t cols_min, cols_max;  // inclusive
    int64_t rows_min, rows_max;  // inclusive
    mt_plan_t plan;
};

#include "plan_table.inc"

bool is_pow2(int64_t v) { return v > 0 && (v & (v - 1)) == 0; }

int64_t pow2_ceil(int64_t v) {
    int64_t p = 1;
    while (p < v) p <<= 1;
    return p;
}

bool chunk_instantiated(int k) {
    for (int i = 0; i < kNumChunkSet; ++i)
        if (kChunkSet[i] == k) return true;
    return false;
}

// Values per thread per chunk instantiated for a storage type: FP32 packs of
// 1, 2, 4 values; FP16/BF16 packs of 2, 4, 8 values (4, 8, 16 bytes).
bool v_instantiated(int dtype, int64_t V) {
    if (dtype == DT_F32) return V == 1 || V == 2 || V == 4;
    return V == 2 || V == 4 || V == 8;
}

// Heuristic plan for shapes the measured table does not cover: 16-byte
// packs (V = 16 / element size), about `per_thread` values per thread,
// blocks of about 256 threads; register path while one of the instantiated
// chunk counts holds the row, else the loop path.
mt_plan_t heuristic_plan(int op, int dtype, int64_t rows, int64_t cols) {
    (void)op;
    mt_plan_t p;
    memset(&p, 0, sizeof(p));
    const int vmax = 16 / dtype_size(dtype);
    const int vmin = dtype == DT_F32 ? 1 : 2;
    p.values_per_thread = cols >= 16 ? vmax : vmin;
    const int V = p.values_per_thread;
    const int64_t per_thread = rows >= 2048 ? 16 : 8;
    int64_t W = pow2_ceil((cols + per_thread - 1) / per_thread);
    if (W < V) W = V;
    if (W > 1024) W = 1024;
    p.threads_per_row = (int)W;
    int64_t K = pow2_ceil((cols + W * V - 1) / (W * V));
    if (K <= 16 && W <= reg_max_threads((int)(V * K))) {
        p.path = MT_PATH_REGISTERS;
        p.chunks = (int)K;
    } else {
        p.path = MT_PATH_LOOP;
        p.chunks = 0;
        if (W > kLoopMaxThreads) p.threads_per_row = (int)(W = kLoopMaxThreads);
    }
    p.rows_per_block = W >= 256 ? 1 : (int)(256 / W);
    p.grid = 0;
    p.flags = MT_PLAN_PDL;
    return p;
}

}  // namespace

mt_status plan_check(int op, int dtype, int64_t cols, const mt_plan_t &p) {
    if (op < 0 || op >= OP_COUNT || cols < 1) return MT_ERR_INVALID_ARGUMENT;
    if (dtype < 0 || dtype >= DT_COUNT) return MT_ERR_INVALID_ARGUMENT;
    const int64_t W = p.threads_per_row, V = p.values_per_thread;
    const int64_t B = p.rows_per_block;
    if (!is_pow2(W) || W > 1024) return MT_ERR_INVALID_ARGUMENT;
    if (!v_instantiated(dtype, V)) return MT_ERR_INVALID_ARGUMENT;
    // The alignment head (< V elements) is owned one element per worker.
    if (V > 1 && W < V) return MT_ERR_INVALID_ARGUMENT;
    if (B < 1 || B > 1024) return MT_ERR_INVALID_ARGUMENT;
    if (p.grid < 0) return MT_ERR_INVALID_ARGUMENT;
    if (p.flags & ~(MT_PLAN_PDL | MT_PLAN_PREFETCH_NEXT))
        return MT_ERR_INVALID_ARGUMENT;
    const int64_t C = p.cluster <= 1 ? 1 : p.cluster;
    if (p.cluster < 0 || (C != 1 && C != 2 && C != 4 && C != 8))
        return MT_ERR_INVALID_ARGUMENT;
    // Split rows (clusters) are built for 16-byte packs only.
    if (C > 1 && (B != 1 || W < 32 || p.grid % C != 0 ||
                  V * dtype_size(dtype) != 16))
        return MT_ERR_INVALID_ARGUMENT;
    const int64_t threads = W * B;
    if (threads % 32 != 0) return MT_ERR_INVALID_ARGUMENT;
    if (p.path == MT_PATH_REGISTERS) {
        if (!chunk_instantiated(p.chunks)) return MT_ERR_INVALID_ARGUMENT;
        if (threads > reg_max_threads((int)(V * p.chunks)))
            return MT_ERR_OUT_OF_RESOURCES;
        // Every worker's private slots must hold its share of the row; a
        // cluster's CTAs together provide C*W workers.
        if (mt_private_slot_bound(cols, (int32_t)(W * C), (int32_t)V) >
            V * p.chunks)
            return MT_ERR_OUT_OF_RESOURCES;
    } else if (p.path == MT_PATH_LOOP) {
        if (threads > kLoopMaxThreads) return MT_ERR_OUT_OF_RESOURCES;
    } else {
        return MT_ERR_INVALID_ARGUMENT;
    }
    return MT_OK;
}

mt_status plan_lookup(int op, int dtype, int64_t rows, int64_t cols,
                      mt_plan_t *out) {
    if (op < 0 || op >= OP_COUNT || dtype < 0 || dtype >= DT_COUNT ||
        rows < 0 || cols < 1 || out == nullptr)
        return MT_ERR_INVALID_ARGUMENT;
    for (const PlanEntry &e : kPlanTable) {
        if (e.op != op || e.dtype != dtype || cols < e.cols_min ||
            cols > e.cols_max || rows < e.rows_min || rows > e.rows_max)
            continue;
        if (plan_check(op, dtype, cols, e.plan) == MT_OK) {
            *out = e.plan;
            return MT_OK;
        }
    }
    *out = heuristic_plan(op, dtype, rows, cols);
    return MT_OK;
}

}  // namespace mt

extern "C" {

int64_t mt_private_slot_bound(int64_t n, int32_t W, int32_t V) {
    if (n < 0 || W < 1 || V < 1) return -1;
    const int64_t span = (int64_t)W * V;
    const int64_t rem = n % span;
    return (n / span) * V + (rem < V ? rem : V);
}

mt_status mt_plan_query(int op, int64_t rows, int64_t cols, mt_plan_t *out) {
    return mt::plan_lookup(op, MT_DTYPE_F32, rows, cols, out);
}

mt_status mt_plan_check(int op, int64_t cols, const mt_plan_t *plan) {
    if (plan == nullptr) return MT_ERR_INVALID_ARGUMENT;
    return mt::plan_check(op, MT_DTYPE_F32, cols, *plan);
}

mt_status mt_plan_query_dtype(int op, int dtype, int64_t rows, int64_t cols,
                              mt_plan_t *out) {
    return mt::plan_lookup(op, dtype, rows, cols, out);
}

mt_status mt_plan_check_dtype(int op, int dtype, int64_t cols,
                              const mt_plan_t *plan) {
    if (plan == nullptr) return MT_ERR_INVALID_ARGUMENT;
    return mt::plan_check(op, dtype, cols, *plan);
}

size_t mt_describe_plan(const mt_plan_t *p, char *buf, size_t n) {
    char tmp[256];
    int len;
    if (p == nullptr) {
        len = snprintf(tmp, sizeof(tmp), "(null plan)");
    } else {
        char grid[32];
        if (p->grid == 0)
            snprintf(grid, sizeof(grid), "auto");
        else
            snprintf(grid, sizeof(grid), "%d", p->grid);
        const char *path = p->path == MT_PATH_REGISTERS ? "registers"
                           : p->path == MT_PATH_LOOP    ? "loop"
                                                        : "invalid";
        char cl[32] = "";
        if (p->cluster > 1) snprintf(cl, sizeof(cl), " cluster=%d", p->cluster);
        len = snprintf(tmp, sizeof(tmp),
                       "path=%s W=%d V=%d chunks=%d rows_per_block=%d "
                       "threads=%d grid=%s%s%s%s",
                       path, p->threads_per_row, p->values_per_thread,
                       p->chunks, p->rows_per_block,
                       p->threads_per_row * p->rows_per_block, grid, cl,
                       (p->flags & MT_PLAN_PDL) ? " pdl" : "",
                       (p->flags & MT_PLAN_PREFETCH_NEXT) ? " prefetch_next"
                                                          : "");
    }
    if (len < 0) len = 0;
    if (buf != nullptr && n > 0) {
        size_t c = (size_t)len < n - 1 ? (size_t)len : n - 1;
        memcpy(buf, tmp, c);
        buf[c] = '\0';
    }
    return (size_t)len;
}

}  // extern "C"
