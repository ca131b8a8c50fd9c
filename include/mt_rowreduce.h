/*
 * mt_rowreduce.h -- C ABI of a GB300 (sm_103a) library of per-row
 * reductions with FP32 arithmetic: RMSNorm, LayerNorm, residual LayerNorm,
 * softmax, row sum and cross-entropy, plus the fused residual RMSNorm,
 * log-softmax and cross-entropy with an ignore index; FP32, FP16 or BF16
 * storage.
 *
 * Operator family: "Consecutive-worker reduction layout checkpoint",
 * §Evidence and what remains (generic V=4 operator coverage: sum, softmax,
 * RMSNorm, LayerNorm, residual LayerNorm and cross-entropy).  RMSNorm
 * semantics: "Thread Ownership and Software Staging", §Register-tiled
 * reductions (the rmsnorm_register kernel: FP32 reduction and epilogue, one
 * rounding at the output store).  Work mapping: "Consecutive-worker reduction
 * layout checkpoint", §Implementation and semantics (W workers per row, V
 * consecutive values per worker, full/tail split, private-slot bound).
 *
 * Conventions shared by every call below
 * -------------------------------------
 * Layout     every matrix is rows x cols in the call's storage type (FP32
 *            for the *_f32 calls, FP16 for *_f16, BF16 for *_bf16),
 *            contiguous row-major (row r starts at element r*cols); vectors
 *            (weight, gamma, beta) hold cols values of the same type;
 *            per-row outputs (row sums, losses, the mean) hold FP32 values;
 *            labels hold rows int32 values.
 * Memory     every data pointer is a DEVICE pointer owned by the caller and
 *            must be aligned to its element size (4 bytes for FP32, labels
 *            and per-row outputs; 2 bytes for FP16/BF16).  Calls allocate
 *            no device memory and never synchronise the host; work is
 *            enqueued on `stream` (NULL = the legacy default stream) on the
 *            current device, and device-side faults surface at the
 *            caller's next synchronisation.  16-byte aligned pointers and
 *            cols a multiple of V get the fully vectorised path; other
 *            alignments are handled by a per-row scalar head before the
 *            vector body.
 * Aliasing   y == x (in place) is allowed; so are h_out == x and
 *            h_out == residual.  Any other (partial) overlap between an
 *            output and an input is undefined.
 * Errors     arguments are checked before anything is enqueued: a NULL
 *            required pointer (rows > 0), a pointer not aligned to its
 *            element size, a pointer the operator does not take, rows < 0,
 *            cols < 1, cols > INT32_MAX or rows*cols overflowing int64 give
 *            MT_ERR_INVALID_ARGUMENT and enqueue nothing.
 *            rows == 0 returns MT_OK without a launch (outputs untouched).
 *            A failed launch gives MT_ERR_CUDA (mt_last_cuda_error() has the
 *            cudaError_t value).  A forced plan that is malformed gives
 *            MT_ERR_INVALID_ARGUMENT; one that cannot hold the row or
 *            exceeds the kernel's thread limit gives MT_ERR_OUT_OF_RESOURCES.
 *            Plans are never silently remapped.
 * Numerics   all arithmetic is FP32 with one rounding at each output store;
 *            the addition order depends on the plan (W, V, chunks), and the
 *            same inputs with the same plan give bit-identical outputs.  No
 *            float atomics are used.
 */
#ifndef MT_ROWREDUCE_H
#define MT_ROWREDUCE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MT_API __attribute__((visibility("default")))
#else
#define MT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *mt_stream_t;

typedef enum mt_status {
    MT_OK = 0,
    MT_ERR_INVALID_ARGUMENT = 1,
    MT_ERR_UNSUPPORTED = 2,
    MT_ERR_OUT_OF_RESOURCES = 3,
    MT_ERR_CUDA = 4
} mt_status;

typedef enum mt_op {
    MT_OP_RMSNORM = 0,
    MT_OP_LAYERNORM = 1,
    MT_OP_RESIDUAL_LAYERNORM = 2,
    MT_OP_SOFTMAX = 3,
    MT_OP_ROW_SUM = 4,
    MT_OP_CROSS_ENTROPY = 5,
    MT_OP_RESIDUAL_RMSNORM = 6,
    MT_OP_LOG_SOFTMAX = 7
} mt_op;

/* ignore_index value meaning "no label is ignored". */
#define MT_NO_IGNORE_INDEX INT32_MIN

/* Storage type of the matrices and parameter vectors of a call.  All
 * arithmetic is FP32 whatever the storage type; per-row outputs (row sums,
 * losses, the mean) are FP32 for every type. */
typedef enum mt_dtype {
    MT_DTYPE_F32 = 0,
    MT_DTYPE_F16 = 1,  /* IEEE binary16 */
    MT_DTYPE_BF16 = 2  /* bfloat16: the upper 16 bits of an FP32 */
} mt_dtype;

/* 16-bit storage, passed by bit pattern. */
typedef uint16_t mt_f16_t;
typedef uint16_t mt_bf16_t;

typedef enum mt_path {
    /* The whole row is read once into registers (V*chunks values per
     * thread) and written from them. */
    MT_PATH_REGISTERS = 0,
    /* Rows too wide for registers: a strided loop computes the statistics
     * and a second loop re-reads x to write y.  Row sum and cross-entropy
     * need only the first loop. */
    MT_PATH_LOOP = 1,
    /* Rows staged in shared memory: each CTA (of a cluster of
     * `cluster` CTAs per row) copies its contiguous run of the row, at most
     * 200 KiB, into shared memory with `chunks` bulk asynchronous copies
     * (1, 2, 4 or 8 pieces), computes the statistics from shared memory and
     * writes y from it, so x is read from global memory once.  Inside the
     * run, 16-byte units go round robin to the W threads.  For RMSNorm,
     * LayerNorm, softmax, log-softmax, cross-entropy and row sum; 16-byte
     * units (V*element size = 16), rows_per_block = 1, W >= 32, and rows
     * that start on 16-byte boundaries (cols a multiple of V, 16-byte
     * aligned pointers): a forced staged plan on other rows returns
     * MT_ERR_INVALID_ARGUMENT, and a staged plan from the table gives way
     * to the loop path there. */
    MT_PATH_STAGE = 2
} mt_path;

/* One launch configuration ("plan").  In the pages' notation W =
 * threads_per_row cooperating workers per row, V = values_per_thread
 * consecutive values each worker owns per chunk; element i of a row (after
 * its alignment head) belongs to worker (i / V) % W, chunk i / (W*V), slot
 * (chunk*V + i % V).  ("Consecutive-worker reduction layout checkpoint",
 * §Implementation and semantics.) */
typedef struct mt_plan {
    int32_t threads_per_row;   /* W: power of two, 1..1024 */
    int32_t values_per_thread; /* V: FP32 1, 2 or 4; FP16/BF16 2, 4 or 8
                                  (V*element size = 16 is one 16-byte
                                  access) */
    int32_t chunks;            /* register path: chunks held per thread, one
                                  of 1, 2, 4, 8, 16; W*V*chunks >= cols.
                                  Staged path: bulk copies per CTA run (1,
                                  2, 4 or 8).  Loop path: ignored (set
                                  0). */
    int32_t rows_per_block;    /* B >= 1 rows per CTA; W*B threads per CTA,
                                  a multiple of 32 and <= 1024 */
    int32_t path;              /* mt_path */
    int32_t grid;              /* CTAs to launch; 0 = min(row groups, CTAs
                                  resident on the device), the CTAs then loop
                                  over row groups (grid-stride) */
    int32_t flags;             /* MT_PLAN_* bits */
    int32_t cluster;           /* CTAs sharing one row: 0 or 1 = none; 2, 4,
                                  8 or 16 (16: beyond the portable cluster
                                  size; the launch fails with MT_ERR_CUDA
                                  where the device cannot place it) = a
                                  thread-block cluster of that many
                                  CTAs splits every row (then
                                  rows_per_block = 1, W >= 32, 16-byte packs
                                  (V*element size = 16), the ownership map
                                  spans cluster*W workers, and an explicit
                                  grid counts CTAs, a multiple of the
                                  cluster size) */
} mt_plan_t;

/* Plan flag: launch as a programmatic dependent of the previous kernel on
 * the stream.  The kernel may start while that kernel finishes; it only
 * prefetches its first rows into L2 and then waits for the previous
 * kernel's completion (and memory visibility) before it reads or writes any
 * operand, so results are the same as with an ordinary launch. */
#define MT_PLAN_PDL 1
/* Plan flag: when the grid is smaller than the number of row groups (CTAs
 * loop over row groups), each CTA asks L2 to prefetch its next row group
 * while it processes the current one. */
#define MT_PLAN_PREFETCH_NEXT 2
/* Plan flag (register path, no cluster): where the plan tiles every row
 * exactly (cols = W*V*chunks), rows is a multiple of rows_per_block, the
 * rows are aligned and every parameter vector the operator reads is
 * present, run the variant of the kernel without bounds guards.  Elsewhere
 * the flag has no effect.  The results are the same bits either way; the
 * two variants differ in instructions and registers, so the tuner measures
 * both. */
#define MT_PLAN_WHOLE_TILES 4

/* ---- operators ---------------------------------------------------------
 * Each takes its plan from the built-in, measured plan table
 * (mt_plan_query).  The *_with_plan forms take an explicit plan; plan ==
 * NULL means the table's plan. */

/* RMSNorm per row: y = x / sqrt(mean(x^2) + eps) * weight.
 * weight may be NULL (all ones).  ("Thread Ownership and Software Staging",
 * §Register-tiled reductions, rmsnorm_register.) */
MT_API mt_status mt_rmsnorm_f32(const float *x, const float *weight, float *y,
                         int64_t rows, int64_t cols, float eps,
                         mt_stream_t stream);
MT_API mt_status mt_rmsnorm_f32_with_plan(const float *x, const float *weight,
                                   float *y, int64_t rows, int64_t cols,
                                   float eps, mt_stream_t stream,
                                   const mt_plan_t *plan);

/* LayerNorm per row: mu = mean(x), var = mean((x-mu)^2) (biased),
 * y = (x - mu) / sqrt(var + eps) * gamma + beta.  gamma may be NULL (ones),
 * beta may be NULL (zeros).  ("Consecutive-worker reduction layout checkpoint", §Evidence and
 * what remains, names the operator; the textbook definition is used.) */
MT_API mt_status mt_layernorm_f32(const float *x, const float *gamma,
                           const float *beta, float *y, int64_t rows,
                           int64_t cols, float eps, mt_stream_t stream);
MT_API mt_status mt_layernorm_f32_with_plan(const float *x, const float *gamma,
                                     const float *beta, float *y,
                                     int64_t rows, int64_t cols, float eps,
                                     mt_stream_t stream,
                                     const mt_plan_t *plan);

/* Residual LayerNorm per row: h = x + residual (FP32 add);
 * y = LayerNorm(h) as above; if h_out != NULL it receives h.
 * ("Consecutive-worker reduction layout checkpoint", §Evidence and
 * what remains, names the operator; the textbook definition is used.) */
MT_API mt_status mt_residual_layernorm_f32(const float *x, const float *residual,
                                    const float *gamma, const float *beta,
                                    float *y, float *h_out, int64_t rows,
                                    int64_t cols, float eps,
                                    mt_stream_t stream);
MT_API mt_status mt_residual_layernorm_f32_with_plan(
    const float *x, const float *residual, const float *gamma,
    const float *beta, float *y, float *h_out, int64_t rows, int64_t cols,
    float eps, mt_stream_t stream, const mt_plan_t *plan);

/* Softmax per row: y = exp(x - max(x)) / sum(exp(x - max(x))).  A row that
 * holds a NaN gives an all-NaN output row.  ("Consecutive-worker reduction layout checkpoint", §Evidence and
 * what remains, names the operator; the textbook definition is used.) */
MT_API mt_status mt_softmax_f32(const float *x, float *y, int64_t rows,
                         int64_t cols, mt_stream_t stream);
MT_API mt_status mt_softmax_f32_with_plan(const float *x, float *y, int64_t rows,
                                   int64_t cols, mt_stream_t stream,
                                   const mt_plan_t *plan);

/* Row sum: out[r] = sum of row r (rows outputs).  Accumulated with
 * compensated (two-sum) FP32 arithmetic, so sums of small integers are
 * exact and near-zero sums keep their relative accuracy.
 * ("Consecutive-worker reduction layout checkpoint", §Evidence and
 * what remains, names the operator; the textbook definition is used.) */
MT_API mt_status mt_row_sum_f32(const float *x, float *out, int64_t rows,
                         int64_t cols, mt_stream_t stream);
MT_API mt_status mt_row_sum_f32_with_plan(const float *x, float *out, int64_t rows,
                                   int64_t cols, mt_stream_t stream,
                                   const mt_plan_t *plan);

/* Cross-entropy per row: loss[r] = log(sum(exp(x_r))) - x_r[labels[r]]
 * (computed with the row max subtracted).  labels holds rows int32 class
 * indices; a label outside [0, cols) gives loss NaN for that row.  If
 * mean_loss != NULL it receives sum(loss) / rows, summed in a fixed order by
 * a second one-CTA kernel on the same stream (deterministic).
 * ("Consecutive-worker reduction layout checkpoint", §Evidence and
 * what remains, names the operator; the textbook definition is used.) */
MT_API mt_status mt_cross_entropy_f32(const float *logits, const int32_t *labels,
                               float *loss, float *mean_loss, int64_t rows,
                               int64_t cols, mt_stream_t stream);
MT_API mt_status mt_cross_entropy_f32_with_plan(const float *logits,
                                         const int32_t *labels, float *loss,
                                         float *mean_loss, int64_t rows,
                                         int64_t cols, mt_stream_t stream,
                                         const mt_plan_t *plan);

/* ---- fused variants (same engine, same conventions) ---------------------
 * The pages do not name these; each is the plain composition of the
 * definitions above. */

/* Residual RMSNorm (pre-norm add-and-norm) per row: h = x + residual (FP32
 * add); y = h / sqrt(mean(h^2) + eps) * weight; if h_out != NULL it
 * receives h.  weight may be NULL (all ones). */
MT_API mt_status mt_residual_rmsnorm_f32(const float *x, const float *residual,
                                         const float *weight, float *y,
                                         float *h_out, int64_t rows,
                                         int64_t cols, float eps,
                                         mt_stream_t stream);
MT_API mt_status mt_residual_rmsnorm_f32_with_plan(
    const float *x, const float *residual, const float *weight, float *y,
    float *h_out, int64_t rows, int64_t cols, float eps, mt_stream_t stream,
    const mt_plan_t *plan);

/* Log-softmax per row: y = (x - max(x)) - log(sum(exp(x - max(x)))).  A row
 * that holds a NaN gives an all-NaN output row. */
MT_API mt_status mt_log_softmax_f32(const float *x, float *y, int64_t rows,
                                    int64_t cols, mt_stream_t stream);
MT_API mt_status mt_log_softmax_f32_with_plan(const float *x, float *y,
                                              int64_t rows, int64_t cols,
                                              mt_stream_t stream,
                                              const mt_plan_t *plan);

/* Cross-entropy with an ignore index: rows whose label equals ignore_index
 * get loss 0 and are left out of the mean, which divides by the number of
 * other rows (NaN when every row is ignored).  Any other label outside
 * [0, cols) still gives loss NaN.  MT_NO_IGNORE_INDEX ignores nothing (same
 * as mt_cross_entropy_f32). */
MT_API mt_status mt_cross_entropy_ignore_f32(const float *logits,
                                             const int32_t *labels,
                                             int32_t ignore_index, float *loss,
                                             float *mean_loss, int64_t rows,
                                             int64_t cols, mt_stream_t stream);

/* ---- FP16 / BF16 storage ------------------------------------------------
 * Same operators with 16-bit matrices and parameter vectors: every value is
 * widened to FP32 on load, all statistics and the epilogue (including the
 * weight / gamma / beta multiply-add) are FP32, and the result is rounded to
 * the storage type once, at the store (round to nearest even).  Residual
 * LayerNorm normalises the FP32 sum x + r and stores h_out = round(x + r).
 * Row sums, losses and the mean stay FP32.  Pointers must be 2-byte
 * aligned; everything else is as for the FP32 calls. */
MT_API mt_status mt_rmsnorm_f16(const mt_f16_t *x, const mt_f16_t *weight,
                                mt_f16_t *y, int64_t rows, int64_t cols,
                                float eps, mt_stream_t stream);
MT_API mt_status mt_rmsnorm_bf16(const mt_bf16_t *x, const mt_bf16_t *weight,
                                 mt_bf16_t *y, int64_t rows, int64_t cols,
                                 float eps, mt_stream_t stream);
MT_API mt_status mt_layernorm_f16(const mt_f16_t *x, const mt_f16_t *gamma,
                                  const mt_f16_t *beta, mt_f16_t *y,
                                  int64_t rows, int64_t cols, float eps,
                                  mt_stream_t stream);
MT_API mt_status mt_layernorm_bf16(const mt_bf16_t *x, const mt_bf16_t *gamma,
                                   const mt_bf16_t *beta, mt_bf16_t *y,
                                   int64_t rows, int64_t cols, float eps,
                                   mt_stream_t stream);
MT_API mt_status mt_residual_layernorm_f16(
    const mt_f16_t *x, const mt_f16_t *residual, const mt_f16_t *gamma,
    const mt_f16_t *beta, mt_f16_t *y, mt_f16_t *h_out, int64_t rows,
    int64_t cols, float eps, mt_stream_t stream);
MT_API mt_status mt_residual_layernorm_bf16(
    const mt_bf16_t *x, const mt_bf16_t *residual, const mt_bf16_t *gamma,
    const mt_bf16_t *beta, mt_bf16_t *y, mt_bf16_t *h_out, int64_t rows,
    int64_t cols, float eps, mt_stream_t stream);
MT_API mt_status mt_softmax_f16(const mt_f16_t *x, mt_f16_t *y, int64_t rows,
                                int64_t cols, mt_stream_t stream);
MT_API mt_status mt_softmax_bf16(const mt_bf16_t *x, mt_bf16_t *y,
                                 int64_t rows, int64_t cols,
                                 mt_stream_t stream);
MT_API mt_status mt_row_sum_f16(const mt_f16_t *x, float *out, int64_t rows,
                                int64_t cols, mt_stream_t stream);
MT_API mt_status mt_row_sum_bf16(const mt_bf16_t *x, float *out, int64_t rows,
                                 int64_t cols, mt_stream_t stream);
MT_API mt_status mt_cross_entropy_f16(const mt_f16_t *logits,
                                      const int32_t *labels, float *loss,
                                      float *mean_loss, int64_t rows,
                                      int64_t cols, mt_stream_t stream);
MT_API mt_status mt_cross_entropy_bf16(const mt_bf16_t *logits,
                                       const int32_t *labels, float *loss,
                                       float *mean_loss, int64_t rows,
                                       int64_t cols, mt_stream_t stream);
MT_API mt_status mt_cross_entropy_ignore_f16(
    const mt_f16_t *logits, const int32_t *labels, int32_t ignore_index,
    float *loss, float *mean_loss, int64_t rows, int64_t cols,
    mt_stream_t stream);
MT_API mt_status mt_cross_entropy_ignore_bf16(
    const mt_bf16_t *logits, const int32_t *labels, int32_t ignore_index,
    float *loss, float *mean_loss, int64_t rows, int64_t cols,
    mt_stream_t stream);
MT_API mt_status mt_residual_rmsnorm_f16(const mt_f16_t *x,
                                         const mt_f16_t *residual,
                                         const mt_f16_t *weight, mt_f16_t *y,
                                         mt_f16_t *h_out, int64_t rows,
                                         int64_t cols, float eps,
                                         mt_stream_t stream);
MT_API mt_status mt_residual_rmsnorm_bf16(const mt_bf16_t *x,
                                          const mt_bf16_t *residual,
                                          const mt_bf16_t *weight,
                                          mt_bf16_t *y, mt_bf16_t *h_out,
                                          int64_t rows, int64_t cols,
                                          float eps, mt_stream_t stream);
MT_API mt_status mt_log_softmax_f16(const mt_f16_t *x, mt_f16_t *y,
                                    int64_t rows, int64_t cols,
                                    mt_stream_t stream);
MT_API mt_status mt_log_softmax_bf16(const mt_bf16_t *x, mt_bf16_t *y,
                                     int64_t rows, int64_t cols,
                                     mt_stream_t stream);

/* Any operator (mt_op) and storage type with an explicit plan (NULL = the
 * table's plan).  Pointer arguments follow the typed calls above; pointers
 * an operator does not take must be NULL: x, weight (gamma), beta,
 * residual, y, h_out are of `dtype`; out (row sums / losses) and mean_loss
 * are FP32; labels are int32.  ignore_index applies to cross-entropy only
 * (MT_NO_IGNORE_INDEX for none); eps is ignored by the operators that have
 * none. */
MT_API mt_status mt_row_reduce_with_plan(
    int op, int dtype, const void *x, const void *residual,
    const void *weight, const void *beta, const int32_t *labels,
    int32_t ignore_index, void *y, void *h_out, float *out, float *mean_loss,
    int64_t rows, int64_t cols, float eps, mt_stream_t stream,
    const mt_plan_t *plan);

/* ---- planning and introspection (host only; no CUDA call) ------------- */

/* The plan the operators use for (op, rows, cols): a lookup in the table of
 * measured winners, else the nearest measured shape re-fitted, else the
 * built-in heuristic.  grid is 0 (resolved at launch from the device's SM
 * count and occupancy) unless the measured winner had an explicit
 * persistent grid (a multiple of the SM count it was measured on).
 * Returns MT_ERR_INVALID_ARGUMENT for an unknown op, rows < 0 or
 * cols < 1. */
MT_API mt_status mt_plan_query(int op, int64_t rows, int64_t cols, mt_plan_t *out);

/* Legality of a plan for (op, cols) without launching anything: MT_OK, or
 * the error the *_with_plan call would return. */
MT_API mt_status mt_plan_check(int op, int64_t cols, const mt_plan_t *plan);

/* The same two calls for any storage type (mt_dtype); the plain forms above
 * are MT_DTYPE_F32.  An unknown dtype gives MT_ERR_INVALID_ARGUMENT. */
MT_API mt_status mt_plan_query_dtype(int op, int dtype, int64_t rows,
                                     int64_t cols, mt_plan_t *out);
MT_API mt_status mt_plan_check_dtype(int op, int dtype, int64_t cols,
                                     const mt_plan_t *plan);

/* Private-slot bound of the consecutive-worker map: the most values any one
 * of W workers owns in a row of n elements with V consecutive values per
 * worker, floor(n/(W*V))*V + min(n % (W*V), V).  ("Consecutive-worker
 * reduction layout checkpoint", §Implementation and semantics.)  Returns
 * -1 for n < 0, W < 1 or V < 1. */
MT_API int64_t mt_private_slot_bound(int64_t n, int32_t W, int32_t V);

/* Writes a one-line description of `plan` into buf (at most n bytes,
 * NUL-terminated when n > 0).  Returns the length the full text needs,
 * excluding the NUL (snprintf convention). */
MT_API size_t mt_describe_plan(const mt_plan_t *plan, char *buf, size_t n);

/* ---- measurement aids ----------------------------------------------------
 * Not operators, and the pages have no counterpart: they give the floor a
 * row-reduction launch is measured against.  Both launch like the
 * operators, as programmatic dependents of the previous kernel on the stream
 * (MT_PLAN_PDL), so a chain of them is timed the way a chain of operator
 * calls is.  threads: CTA size, a multiple of 32 in [32, 1024]; grid: CTAs
 * to launch, 0 = one wave (SMs x CTAs resident per SM).  They allocate
 * nothing and never synchronise. */

/* Copies `bytes` bytes from src to dst (device pointers, both 16-byte
 * aligned, bytes a multiple of 16, the two ranges disjoint) with 16-byte
 * loads and stores.  Each CTA copies one contiguous slice of the buffer (as
 * an operator's CTA owns its rows); its threads stride over the slice, each
 * keeping `unroll` (1, 2, 4 or 8) loads in flight.  flags: 0, or
 * MT_PLAN_PDL to have each CTA prefetch its slice into L2 before it waits
 * for the previous kernel, as the operators do under that flag.
 * bytes == 0 is a no-op.  Bad arguments give MT_ERR_INVALID_ARGUMENT and
 * enqueue nothing. */
MT_API mt_status mt_probe_copy(const void *src, void *dst, int64_t bytes,
                               int32_t threads, int32_t unroll, int32_t grid,
                               int32_t flags, mt_stream_t stream);

/* Reads `bytes` bytes at src (16-byte aligned, bytes a multiple of 16)
 * with the CTA slices, threads and loads in flight of mt_probe_copy, and
 * writes one 32-bit word per CTA to dst[cta]: the XOR of the words of its
 * slice.  dst holds dst_words words; the grid (given, or one wave when
 * grid == 0) must not exceed it.  The floor of an operator that reads a
 * matrix and writes one value per row.  flags as for mt_probe_copy. */
MT_API mt_status mt_probe_read(const void *src, int64_t bytes, uint32_t *dst,
                               int64_t dst_words, int32_t threads,
                               int32_t unroll, int32_t grid, int32_t flags,
                               mt_stream_t stream);

/* A kernel that does no work: the fixed cost of one dependent launch. */
MT_API mt_status mt_probe_empty(int32_t threads, int32_t grid,
                                mt_stream_t stream);

/* Static string naming a status. */
MT_API const char *mt_status_string(mt_status status);

/* The cudaError_t behind the calling thread's last MT_ERR_CUDA (0 if
 * none). */
MT_API int mt_last_cuda_error(void);

/* Diagnostic of the staged path (no counterpart on the pages): *count =
 * the number of waits for a bulk copy into shared memory that gave up
 * (after about two seconds) on the current device since the library was
 * loaded; 0 unless something else has gone wrong on the device.  A kernel
 * that gives up leaves its outputs undefined but returns.  Synchronous (a
 * device-to-host copy per kernel family); not for hot paths. */
MT_API mt_status mt_stage_wait_timeouts(uint64_t *count);

#ifdef __cplusplus
}
#endif

#endif /* MT_ROWREDUCE_H */
