// planner.cpp -- launch-plan choice and legality (host only, no CUDA call).
//
// A plan fixes W (threads per row), V (consecutive values per thread per
// chunk), the register chunk count K, the rows per CTA B, the path, the
// grid, launch flags and the cluster size.  The operators take the plan from
// a table of winners measured on the GPU (plan_table.inc, written by the
// package's tuner), keyed by operator, storage type and a (cols, rows)
// range.  A shape outside the table takes the measured winner of the
// nearest tuned shape -- nearest in log2(cols), then log2(rows) -- with its
// chunk count (and if need be its width, or its path) re-fitted to the new
// row length; the heuristic below is the last resort.
//
// The legality rules follow the fail-closed contract of the pages: a plan is
// checked before dispatch and an illegal one is rejected, never remapped
// ("Thread Ownership and Software Staging", §Compiler-selected communication,
// the maxTotalThreadsPerThreadgroup check; "Consecutive-worker reduction
// layout checkpoint", §Verification checkpoint: invalid widths and resource
// overflow fail closed), and the private-slot bound is enforced before a plan
// is used ("Consecutive-worker reduction layout checkpoint", §Implementation
// and semantics).
#include <math.h>
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
    int64_t rows_tuned;          // the row count the plan was measured at
    mt_plan_t plan;
};

#include "plan_table.inc"

bool is_pow2(int64_t v) { return v > 0 && (v & (v - 1)) == 0; }

int64_t pow2_ceil(int64_t v) {
    int64_t p = 1;
    while (p < v) p <<= 1;
    return p;
}

// CTAs per row for a row count: rows are split across a cluster only while
// there are too few rows to give each SM work (152 SMs: 16 CTAs per row up
// to 9 rows, 8 up to 19, 4 up to 38, 2 up to 76).
int64_t cluster_for(int64_t rows) {
    return rows <= 9    ? 16
           : rows <= 19 ? 8
           : rows <= 38 ? 4
           : rows <= 76 ? 2
                        : 1;
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

// Values one CTA's registers hold with V-value packs: 256 threads x 16
// chunks, the largest register-path team at the 256-thread limit.
int64_t cta_register_values(int64_t V) { return 256 * 16 * V; }

// Rows wider than one CTA's registers stay on the register path, on a
// cluster of two CTAs, when there are enough rows to keep every SM busy
// with such CTAs: measured on 4096 and 8192 rows of 32000 values.  With
// fewer rows the loop path's wider teams keep more bytes in flight.
int64_t wide_row_cluster(int64_t rows, int64_t cols, int64_t V) {
    if (rows < 512) return 0;
    for (int64_t C = 1; C <= 2; C *= 2)
        if (C * cta_register_values(V) >= cols) return C;
    return 0;
}

// Staged rows: the smallest cluster (1..16 CTAs) whose runs take at most
// 128 KiB of shared memory each, so at least one CTA fits an SM beside
// another's run (the measured staged winners: 32000 FP32 values on one CTA
// or two, 131072 BF16 values on two); 0 when even 16 CTAs do not suffice.
int64_t stage_cluster(int64_t cols, int es) {
    for (int64_t C = 1; C <= 16; C *= 2)
        if (stage_run_bytes(cols, es, C) <= 128 * 1024) return C;
    return 0;
}

// Heuristic plan for shapes far from every measured one.  It follows what
// the measured winners have in common:
//  * 16-byte packs (V = 16 / element size) unless the row is tiny;
//  * short rows (<= 32 packs): a warp or less per row, several rows per CTA;
//  * rows that fit in registers at about 16 values per thread (up to 64 KiB
//    of FP32 data): one row per CTA of W = row/16 threads (at most 1024),
//    two rows per CTA when that leaves fewer than 256 threads;
//  * wider rows, fewer rows than SMs: a cluster of 8 CTAs per row;
//  * wider rows of the staged operators (cols a multiple of the 16-byte
//    unit): the staged path, 512 threads, two bulk copies per run, on the
//    smallest cluster whose runs take at most 128 KiB (stage_cluster) --
//    the row read once, as the measured wide-row winners do;
//  * other wider rows, at least 512 of them, that one or two CTAs of 256
//    threads x 16 chunks hold: the register path on that cluster -- one
//    read of the row instead of the loop path's two (wide_row_cluster);
//  * the other wide rows: the loop path with 256 threads per row and two
//    rows per CTA, so several rows stream through each SM at once.
// All launches use the programmatic-dependent prologue.  Register-path CTAs
// prefetch their next row group; loop-path CTAs do not (the measured loop
// winners mostly do without it: their own second pass re-reads the row from
// L2, and the prefetch competes with it).
mt_plan_t heuristic_plan(int op, int dtype, int64_t rows, int64_t cols) {
    mt_plan_t p;
    memset(&p, 0, sizeof(p));
    const int es = dtype_size(dtype);
    const int vmax = 16 / es;
    const int vmin = dtype == DT_F32 ? 1 : 2;
    const int V = cols >= 4 * vmax ? vmax : vmin;
    p.values_per_thread = V;
    p.flags = MT_PLAN_PDL | MT_PLAN_PREFETCH_NEXT;
    const int64_t packs = (cols + V - 1) / V;
    if (packs <= 32) {
        int64_t W = pow2_ceil(packs);
        if (W < V) W = V;
        if (W < 1) W = 1;
        p.threads_per_row = (int)W;
        p.chunks = 1;
        p.rows_per_block = (int)(256 / W);
        p.path = MT_PATH_REGISTERS;
        return p;
    }
    const int64_t reg_cap = 16384;  // FP32 values a row may keep in registers
    if (cols <= reg_cap) {
        int64_t W = pow2_ceil((packs + 3) / 4);  // about 4 packs per thread
        if (W > 1024) W = 1024;
        if (W < 32) W = 32;
        int64_t K = pow2_ceil((cols + W * V - 1) / (W * V));
        while (K > 16 || W > reg_max_threads((int)(V * K))) {
            if (W >= 1024) break;
            W *= 2;
            K = pow2_ceil((cols + W * V - 1) / (W * V));
        }
        if (K <= 16 && W <= reg_max_threads((int)(V * K))) {
            p.threads_per_row = (int)W;
            p.chunks = (int)K;
            p.rows_per_block = W >= 256 ? 1 : (int)(256 / W);
            p.path = MT_PATH_REGISTERS;
            return p;
        }
    }
    const int64_t C = cluster_for(rows);
    if (C > 1 && V * es == 16) {
        // A cluster of C CTAs per row: registers while the row fits.
        p.cluster = (int)C;
        p.rows_per_block = 1;
        for (int64_t W = 32; W <= 1024; W *= 2) {
            for (int i = 0; i < kNumChunkSet; ++i) {
                const int64_t K = kChunkSet[i];
                if (K > 4 || C * W * V * K < cols ||
                    W > reg_max_threads((int)(V * K)))
                    continue;
                p.threads_per_row = (int)W;
                p.chunks = (int)K;
                p.path = MT_PATH_REGISTERS;
                return p;
            }
        }
        p.path = MT_PATH_LOOP;
        p.chunks = 0;
        p.flags = MT_PLAN_PDL;
        p.threads_per_row = 512;
        return p;
    }
    if (V * es == 16 && stage_op(op) && cols % V == 0) {
        const int64_t Cs = stage_cluster(cols, es);
        if (Cs > 0) {
            p.path = MT_PATH_STAGE;
            p.cluster = Cs > 1 ? (int)Cs : 0;
            p.threads_per_row = 512;
            p.chunks = 2;
            p.rows_per_block = 1;
            return p;
        }
    }
    if (V * es == 16) {
        const int64_t Cw = wide_row_cluster(rows, cols, V);
        if (Cw > 0) {
            int64_t K = 16;
            for (int i = 0; i < kNumChunkSet; ++i)
                if (Cw * 256 * V * kChunkSet[i] >= cols) {
                    K = kChunkSet[i];
                    break;
                }
            p.cluster = Cw > 1 ? (int)Cw : 0;
            p.threads_per_row = 256;
            p.chunks = (int)K;
            p.rows_per_block = 1;
            p.path = MT_PATH_REGISTERS;
            return p;
        }
    }
    p.path = MT_PATH_LOOP;
    p.chunks = 0;
    p.flags = MT_PLAN_PDL;
    // Two rows per CTA once there are enough rows for two CTAs per SM.
    p.threads_per_row = rows >= 304 ? 256 : 512;
    p.rows_per_block = rows >= 304 ? 2 : 1;
    return p;
}

}  // namespace

namespace {
double log2d(double v) { return log2(v < 1.0 ? 1.0 : v); }

mt_status plan_check_impl(int op, int dtype, int64_t cols, const mt_plan_t &p);

// Re-fits the measured plan of shape (rows_src, cols_src) to (rows, cols).
// The source plan says how many threads the device wanted in flight
// (rows_src * W * cluster) and how they were grouped (threads per CTA,
// flags, V); the re-fit keeps those and recomputes the rest:
//  * cluster: cluster_for(rows) for wide rows (>= 8192) of 16-byte packs;
//    on the register path, rows wider than those CTAs' registers take
//    wide_row_cluster's cluster, or the loop path when it has none;
//  * W = the source's threads in flight / rows / cluster (a power of two),
//    raised until the row fits in at most 8 chunks, capped at 1024, then
//    lowered while that breaks the kernel's thread limit for the chunk
//    count the row needs;
//  * chunks: the smallest instantiated count that holds the row, the loop
//    path when none does;
//  * rows per CTA: what keeps the source's CTA size.
// Returns false when nothing legal is left.
bool refit(int op, int dtype, int64_t rows_src, int64_t rows, int64_t cols,
           mt_plan_t *p) {
    const int64_t V = p->values_per_thread;
    if (p->path == MT_PATH_STAGE) {
        // A staged winner stays staged where the row can be: same threads,
        // copies and flags, the cluster that keeps runs within 128 KiB (or
        // spreads few rows as cluster_for does), a resident grid.
        const int64_t Cs = stage_cluster(cols, dtype_size(dtype));
        int64_t C = cluster_for(rows);
        if (Cs > C) C = Cs;
        if (Cs > 0 && cols % V == 0 && C <= 16) {
            mt_plan_t q = *p;
            q.cluster = C > 1 ? (int32_t)C : 0;
            q.grid = 0;
            if (plan_check_impl(op, dtype, cols, q) == MT_OK) {
                *p = q;
                return true;
            }
        }
        // Otherwise the loop path with the same team.
        p->path = MT_PATH_LOOP;
        p->chunks = 0;
        p->cluster = 0;
    }
    const int64_t cta = (int64_t)p->threads_per_row * p->rows_per_block;
    const int64_t c_src = p->cluster > 1 ? p->cluster : 1;
    // Split rows when there are few of them and they are wide, and on the
    // register path whenever one CTA's registers cannot hold the row.
    const bool packs16 = V * dtype_size(dtype) == 16;
    const int64_t c_loop = (packs16 && cols >= 8192) ? cluster_for(rows) : 1;
    int64_t C = c_loop;
    if (packs16 && p->path == MT_PATH_REGISTERS &&
        C * cta_register_values(V) < cols) {
        const int64_t cw = wide_row_cluster(rows, cols, V);
        if (cw == 0)
            p->path = MT_PATH_LOOP;
        else if (cw > C)
            C = cw;
    }
    p->cluster = C > 1 ? (int32_t)C : 0;
    p->grid = 0;
    const double inflight = (double)(rows_src < 1 ? 1 : rows_src) *
                            p->threads_per_row * c_src;
    int64_t W = pow2_ceil((int64_t)(inflight / (double)(rows < 1 ? 1 : rows) /
                                    (double)C / 1.414));
    const int64_t wmin = C > 1 ? 32 : (V > 1 ? V : 1);
    if (W < wmin) W = wmin;
    while (W < 1024 && C * W * V * 8 < cols) W *= 2;
    if (W > 1024) W = 1024;
    if (p->path == MT_PATH_REGISTERS) {
        // From W down: narrower teams hold more chunks each, and the
        // kernel's thread limit falls as the chunks per thread rise.
        for (int64_t w = W; w >= wmin; w /= 2) {
            int64_t K = 0;
            for (int i = 0; i < kNumChunkSet; ++i)
                if (C * w * V * kChunkSet[i] >= cols) {
                    K = kChunkSet[i];
                    break;
                }
            if (K == 0) break;
            int64_t B = C > 1 ? 1 : (cta / w < 1 ? 1 : cta / w);
            while (B > 1 && w * B > reg_max_threads((int)(V * K))) B /= 2;
            if ((w * B) % 32 == 0 && w * B <= reg_max_threads((int)(V * K))) {
                p->threads_per_row = (int32_t)w;
                p->chunks = (int32_t)K;
                p->rows_per_block = (int32_t)B;
                // ptxas holds the FP32 4-value, 2-chunk instance to 32
                // registers (it spills); the same row in 2-value packs and
                // 4 chunks does not.
                if (dtype == DT_F32 && V == 4 && K == 2 && C == 1 &&
                    w >= 2) {
                    p->values_per_thread = 2;
                    p->chunks = 4;
                    if (plan_check_impl(op, dtype, cols, *p) == MT_OK)
                        return true;
                    p->values_per_thread = 4;
                    p->chunks = 2;
                }
                if (plan_check_impl(op, dtype, cols, *p) == MT_OK)
                    return true;
            }
        }
        p->path = MT_PATH_LOOP;
        // The loop path splits rows only when they are few.
        C = c_loop;
        p->cluster = C > 1 ? (int32_t)C : 0;
        if (W < 32 && C > 1) W = 32;
    }
    p->chunks = 0;
    if (W > kLoopMaxThreads) W = kLoopMaxThreads;
    int64_t B = C > 1 ? 1 : (cta / W < 1 ? 1 : cta / W);
    while (W * B > kLoopMaxThreads) B /= 2;
    while ((W * B) % 32 != 0) B *= 2;
    p->threads_per_row = (int32_t)W;
    p->rows_per_block = (int32_t)(B < 1 ? 1 : B);
    return plan_check_impl(op, dtype, cols, *p) == MT_OK;
}

}  // namespace

mt_status plan_check(int op, int dtype, int64_t cols, const mt_plan_t &p) {
    return plan_check_impl(op, dtype, cols, p);
}

namespace {
mt_status plan_check_impl(int op, int dtype, int64_t cols, const mt_plan_t &p) {
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
    if (p.flags & ~(MT_PLAN_PDL | MT_PLAN_PREFETCH_NEXT | MT_PLAN_WHOLE_TILES))
        return MT_ERR_INVALID_ARGUMENT;
    const int64_t C = p.cluster <= 1 ? 1 : p.cluster;
    if (p.cluster < 0 || (C != 1 && C != 2 && C != 4 && C != 8 && C != 16))
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
    } else if (p.path == MT_PATH_STAGE) {
        // One row per CTA (or cluster), 16-byte units, W >= 32, 1..8 bulk
        // copies per run, a run that fits the shared-memory budget.
        if (!stage_op(op) || B != 1 || W < 32 ||
            V * dtype_size(dtype) != 16 || p.chunks < 1 ||
            p.chunks > kStagePiecesMax || !is_pow2(p.chunks) ||
            cols % V != 0)
            return MT_ERR_INVALID_ARGUMENT;
        if (stage_run_bytes(cols, dtype_size(dtype), C) > kStageMaxRunBytes)
            return MT_ERR_OUT_OF_RESOURCES;
    } else {
        return MT_ERR_INVALID_ARGUMENT;
    }
    return MT_OK;
}
}  // namespace

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
    // Nearest measured shape of the same operator and storage type.
    const PlanEntry *best = nullptr;
    double best_d = 0.0;
    for (const PlanEntry &e : kPlanTable) {
        if (e.op != op || e.dtype != dtype) continue;
        const double d =
            fabs(log2d((double)cols) - log2d((double)e.cols_min)) +
            0.5 * fabs(log2d((double)rows) - log2d((double)e.rows_tuned));
        if (best == nullptr || d < best_d) {
            best = &e;
            best_d = d;
        }
    }
    // A measured plan transfers to rows within a factor 4 in length and 16
    // in count; farther shapes take the heuristic.
    if (best != nullptr &&
        fabs(log2d((double)cols) - log2d((double)best->cols_min)) <= 2.0 &&
        fabs(log2d((double)rows) - log2d((double)best->rows_tuned)) <= 4.0) {
        mt_plan_t p = best->plan;
        if (refit(op, dtype, best->rows_tuned, rows, cols, &p)) {
            *out = p;
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
                           : p->path == MT_PATH_STAGE   ? "staged"
                                                        : "invalid";
        char cl[32] = "";
        if (p->cluster > 1) snprintf(cl, sizeof(cl), " cluster=%d", p->cluster);
        len = snprintf(tmp, sizeof(tmp),
                       "path=%s W=%d V=%d chunks=%d rows_per_block=%d "
                       "threads=%d grid=%s%s%s%s%s",
                       path, p->threads_per_row, p->values_per_thread,
                       p->chunks, p->rows_per_block,
                       p->threads_per_row * p->rows_per_block, grid, cl,
                       (p->flags & MT_PLAN_PDL) ? " pdl" : "",
                       (p->flags & MT_PLAN_PREFETCH_NEXT) ? " prefetch_next"
                                                          : "",
                       (p->flags & MT_PLAN_WHOLE_TILES) ? " whole_tiles"
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
