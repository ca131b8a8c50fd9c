// planner.cpp -- launch-plan choice and legality (host only, no CUDA call).
//
// A plan fixes W (threads per row), V (consecutive values per thread per
// chunk), the register chunk count K, the rows per CTA B, the path, the
// grid, launch flags and the cluster size.  The operators take the plan from
// a table of winners measured on the GPU (plan_table.inc, written by the
// package's tuner), keyed by operator, storage type and a (cols, rows)
// range.  A shape outside the table takes a plan derived from the shape
// (shape_plan: values per thread from the work per SM, active groups per
// SM, live lanes, the staged path for wide rows); the heuristic below is the
// last resort.
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

// ---- shape-derived plans --------------------------------------------------
// The fallback for shapes outside the table prices the two features the
// pages name for this choice ("Consecutive-worker reduction layout
// checkpoint", §Evidence and what remains: the loss of active groups from
// short-row packing, live lanes, shape-derived collaborating widths), with
// constants read off the measured winners (the tuned table and the
// held-out regret set):
//  * values per thread vt = R*cols / (SMs * 512) rounded down to a power of
//    two and clamped to [8, 32] (the residual operators, which hold two
//    inputs, to 32 bytes of row per thread for LayerNorm and 64 for
//    RMSNorm): the device's share of the work sets how long each thread
//    stays busy, so that about a quarter of the SM's thread slots carry it;
//  * the one-pass operators (row sum, cross-entropy) on rows of up to 16
//    packs per lane: one warp per row, so no shared-memory combine;
//  * the collaborating width W = the row's packs / (vt / V), a power of two,
//    and the chunk count K the smallest that covers the row (the live lanes
//    W*V*K >= cols); FP32 rows at 8 values per thread take 2-value packs
//    (the 4-value, 2-chunk instance spills);
//  * rows per CTA B: CTAs of about 256 threads (128 for the residual
//    operators), halved while that leaves fewer than three active groups
//    per SM (ceil(R / B) < 3 * SMs);
//  * rows of more than 16384 values (more than 32 register values per
//    thread at 512 threads): the staged path for its operators (the
//    one-pass ones from ten rows, the others from 39; FP32 one-pass rows
//    on 304 rows or more keep the loop path), on the smallest cluster whose
//    runs take at most 160 KiB (doubled once when there are fewer runs
//    than 1.5 per SM), 512 threads for runs of 96 KiB and more, else 256;
//  * other few wide rows (at most 38, at least 8192 values): the register
//    path on a cluster of 4, 8 or 16 CTAs per row (cluster_for);
//  * one-pass rows on the loop path: 64-thread teams on many rows, a
//    cluster of 512-thread CTAs for fewer rows than 1.5 per SM.
// Plans that tile the rows exactly also take the whole-tile variant.
constexpr int64_t kPlanSMs = 152;  // GB300

mt_status plan_check_impl(int op, int dtype, int64_t cols, const mt_plan_t &p);

bool has_residual_op(int op) {
    return op == OP_RESIDUAL_LAYERNORM || op == OP_RESIDUAL_RMSNORM;
}

int64_t pow2_floor(int64_t v) {
    int64_t p = 1;
    while (p * 2 <= v) p <<= 1;
    return p;
}

// Staged rows: the smallest cluster whose runs take at most `cap` bytes.
int64_t stage_cluster_cap(int64_t cols, int es, int64_t cap) {
    for (int64_t C = 1; C <= 16; C *= 2)
        if (stage_run_bytes(cols, es, C) <= cap) return C;
    return 0;
}

// One pass, one value out per row: row sum and cross-entropy.
bool one_pass_op(int op) { return op == OP_ROW_SUM || op == OP_CROSS_ENTROPY; }

// Smallest cluster (a power of two, at most 16) that gives `rows` rows at
// least 1.5 CTAs per SM.
int64_t cluster_for_rows(int64_t rows) {
    int64_t C = 1;
    while (C < 16 && rows * C * 2 < 3 * kPlanSMs) C *= 2;
    return C;
}

bool shape_plan(int op, int dtype, int64_t rows, int64_t cols,
                mt_plan_t *out) {
    mt_plan_t p;
    memset(&p, 0, sizeof(p));
    const int es = dtype_size(dtype);
    const int64_t vmax = 16 / es;
    const int64_t R = rows < 1 ? 1 : rows;
    p.flags = MT_PLAN_PDL | MT_PLAN_PREFETCH_NEXT;
    // Wide rows of the staged operators: read once through shared memory.
    // Rows that need more than 32 register values per thread at 512
    // threads (16384 values) count as wide; the cluster is the smallest
    // whose runs take at most 160 KiB, doubled once when that leaves fewer
    // runs than 1.5 per SM.  The one-pass operators stage from ten rows on,
    // the others from 39 (fewer rows keep the register path on a
    // cluster).
    // FP32 one-pass rows on many rows stay on the loop path, which reads
    // them once too (measured: cross-entropy FP32 512x32768 and
    // 4096x32000); their 16-bit rows, with twice the arithmetic per byte,
    // are staged.
    const bool fp32_one_pass_loop =
        one_pass_op(op) && dtype == DT_F32 && R >= 2 * kPlanSMs;
    if (cols > 16384 && (one_pass_op(op) ? R > 9 : cluster_for(R) <= 2) &&
        !fp32_one_pass_loop && stage_op(op) && cols % vmax == 0) {
        int64_t C = stage_cluster_cap(cols, es, 160 * 1024);
        // Fewer runs than 1.5 per SM: split each row once more.
        if (C > 0 && C < 16 && R * C * 2 < 3 * kPlanSMs) C *= 2;
        if (C > 0) {
            p.path = MT_PATH_STAGE;
            p.values_per_thread = (int32_t)vmax;
            p.cluster = C > 1 ? (int32_t)C : 0;
            p.threads_per_row =
                stage_run_bytes(cols, es, C) >= 96 * 1024 ? 512 : 256;
            p.chunks = 2;
            p.rows_per_block = 1;
            if (plan_check_impl(op, dtype, cols, p) == MT_OK) {
                *out = p;
                return true;
            }
        }
    }
    // Few wide rows (at most 38) split across a cluster; wider rows than a
    // cluster's registers hold go to the caller's other rules.
    const int64_t C = (cols >= 8192 && cluster_for(R) > 2) ? cluster_for(R) : 1;
    if (cols > C * cta_register_values(vmax)) return false;
    int64_t V, W;
    if (one_pass_op(op) && C == 1 && cols <= 32 * vmax * 16) {
        // One warp per row: no shared-memory combine at all (the measured
        // one-pass winners on 300..4000 values); 16-bit rows in 16-byte
        // packs, FP32 rows in 8-byte packs.
        V = dtype == DT_F32 ? 2 : vmax;
        // Short 16-bit rows (two 16-byte packs per thread or fewer): 8-byte
        // packs, twice as many.
        if (dtype != DT_F32 && cols <= 32 * vmax * 2) V = vmax / 2;
        if (cols < 4 * V) V = dtype == DT_F32 ? 1 : 2;
        W = 32;
    } else {
        // Values per thread from the work per SM.
        // The residual operators hold two inputs: at most 32 bytes of row
        // per thread for residual LayerNorm, 64 for residual RMSNorm.
        int64_t vt = pow2_floor(R * cols / (kPlanSMs * 512));
        const int64_t vt_max = op == OP_RESIDUAL_LAYERNORM ? 32 / es
                               : op == OP_RESIDUAL_RMSNORM ? 64 / es
                                                           : 32;
        if (vt < 8) vt = 8;
        if (vt > vt_max) vt = vt_max;
        V = cols >= 4 * vmax ? vmax : (dtype == DT_F32 ? 1 : 2);
        if (V > vt) V = vt;
        if (dtype == DT_F32 && vt == 8 && V == 4 && !has_residual_op(op))
            V = 2;
        if (C > 1) V = vmax;  // clusters take 16-byte packs
        const int64_t kt = vt / V < 1 ? 1 : vt / V;
        const int64_t packs = (cols + V - 1) / V;
        W = pow2_ceil((packs + C * kt - 1) / (C * kt));
    }
    const int64_t wmin = C > 1 ? 32 : (V > 1 ? V : 1);
    if (W < wmin) W = wmin;
    if (W > 1024) W = 1024;
    // The chunk count that covers the row (the live lanes W*V*K >= cols); a
    // wider team while the kernel's thread limit allows, if the row needs
    // more than 16 chunks.
    for (;; W *= 2) {
        int64_t K = 0;
        for (int i = 0; i < kNumChunkSet; ++i)
            if (C * W * V * kChunkSet[i] >= cols) {
                K = kChunkSet[i];
                break;
            }
        if (K != 0 && W <= reg_max_threads((int)(V * K))) {
            p.chunks = (int32_t)K;
            break;
        }
        if (W >= 1024) return false;
    }
    // Rows per CTA: about 256 threads, halved while that leaves fewer than
    // three active groups per SM (short rows: many rows per CTA when there
    // are rows to spare, one row per CTA when there are not)
    int64_t B = 1;
    if (C == 1) {
        const int64_t bmin = W >= 32 ? 1 : 32 / W;
        // (the residual operators, heavier in registers: 128 threads)
        const int64_t T = has_residual_op(op) ? 128 : 256;
        B = W >= T ? 1 : T / W;
        while (B > bmin && (R + B - 1) / B < 3 * kPlanSMs) B /= 2;
        while (B > bmin && W * B > reg_max_threads((int)(V * p.chunks)))
            B /= 2;
    }
    p.path = MT_PATH_REGISTERS;
    p.values_per_thread = (int32_t)V;
    p.threads_per_row = (int32_t)W;
    p.rows_per_block = (int32_t)B;
    p.cluster = C > 1 ? (int32_t)C : 0;
    // Exact tilings take the whole-tile variant, except for the residual
    // operators, whose guarded kernels hold fewer registers.
    if (C == 1 && W * V * p.chunks == cols && R % B == 0 &&
        !has_residual_op(op))
        p.flags |= MT_PLAN_WHOLE_TILES;
    if (plan_check_impl(op, dtype, cols, p) != MT_OK) return false;
    *out = p;
    return true;
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
    if (V * es == 16 && stage_op(op) && cols % V == 0 &&
        !(one_pass_op(op) && dtype == DT_F32 && rows >= 2 * kPlanSMs)) {
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
    if (one_pass_op(op) && dtype == DT_F32 && rows >= 2 * kPlanSMs) {
        // FP32 one-pass rows on many rows: the loop path (below).
    } else if (V * es == 16) {
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
    if (one_pass_op(op)) {
        // One-pass loops: no dependent-launch prologue, 64-thread teams on
        // unaligned rows (2048x50257), 256 threads on aligned ones
        // (512x32768); fewer rows than 1.5 per SM split across a cluster
        // of 512-thread CTAs.
        const int64_t Cr = V * es == 16 ? cluster_for_rows(rows) : 1;
        if (Cr > 1) {
            p.cluster = (int32_t)Cr;
            p.threads_per_row = 512;
            p.rows_per_block = 1;
            return p;
        }
        p.flags = 0;
        p.threads_per_row = cols % V == 0 ? 256 : 64;
        p.rows_per_block = 1;
        return p;
    }
    // Two rows per CTA once there are enough rows for two CTAs per SM.
    p.threads_per_row = rows >= 304 ? 256 : 512;
    p.rows_per_block = rows >= 304 ? 2 : 1;
    return p;
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
    // Shapes outside the table: the shape-derived plan, else the heuristic.
    mt_plan_t p;
    if (shape_plan(op, dtype, rows, cols, &p)) {
        *out = p;
        return MT_OK;
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
