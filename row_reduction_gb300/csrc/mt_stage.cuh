// mt_stage.cuh -- the staged path: rows wider than the register budget,
// copied once into shared memory by bulk asynchronous copies (sm_90+
// cp.async.bulk completing on an mbarrier), reduced from shared memory and
// written from it, so that x is read from HBM exactly once and the bytes in
// flight do not depend on registers.  Included by mt_kernels.cuh.
//
// Mapping.  One row per CTA, or per thread-block cluster of C CTAs.  The
// row is cut into 16-byte units (V = 16 / sizeof(T) values each); CTA rank
// q of the cluster owns the contiguous run of units [q*per, (q+1)*per),
// per = ceil(units / C), staged whole in its shared memory.  Inside a CTA
// the W threads take the units of the run round robin (unit u to thread
// u mod W), the pages' consecutive-worker map with V-value packs applied to
// the staged run ("Consecutive-worker reduction layout checkpoint",
// §Implementation and semantics).  The run is copied as up to `pieces`
// bulk copies, each completing on its own mbarrier, so the first pass
// starts on the first piece while the later ones are in flight.
//
// Statistics and epilogues are those of the register path: FP32 arithmetic
// from the staged values, the cross-warp and cross-CTA combines of
// team_allreduce*, one rounding at the store ("Thread Ownership and
// Software Staging", §Register-tiled reductions).  Passes over the staged
// run: RMSNorm 2, LayerNorm 2 (shifted moments, then the output; 16-bit
// rows on a lone CTA 3: the mean, the deviations, the output), softmax and
// log-softmax 2 (a running max/sum, then the output), cross-entropy and row
// sum 1.
//
// The path needs every row to start on a 16-byte boundary (aligned mode:
// cols a multiple of V and 16-byte aligned pointers).
//
// Waits.  Every mbarrier wait gives up after kStageWaitCycles clock cycles
// (about two seconds at 2 GHz): the thread counts the event in
// g_stage_timeouts; from the end of that row on the CTA issues no copies
// and waits for none, still takes part in every barrier of its cluster (so
// no peer waits forever) and, before it exits, waits once more (with the
// same limit) for that row's copies.  A copy of valid memory always
// completes; the limit only bounds a fault elsewhere.
#pragma once

namespace mt {

constexpr int kStageMaxThreads = 1024;
constexpr long long kStageWaitCycles = 1ll << 32;

// Waits that gave up (a diagnostic; one counter per translation unit, all
// of them summed by mt_stage_wait_timeouts).
static __device__ unsigned long long g_stage_timeouts;

__device__ __forceinline__ unsigned smem_addr(const void *p) {
    return (unsigned)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(
                     smem_addr(bar)),
                 "r"(count)
                 : "memory");
}

// Makes the initialised barriers visible to the async proxy and the cluster.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier shared-memory accesses (generic proxy) before
// its later bulk copies into shared memory (async proxy).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar,
                                               unsigned bytes) {
    asm volatile(
        "mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
            smem_addr(bar)),
        "r"(bytes)
        : "memory");
}

// Copies `bytes` (a multiple of 16; both addresses 16-byte aligned) from
// global memory into this CTA's shared memory; completion is counted on
// `bar` in bytes.
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src,
                                              unsigned bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1], %2, [%3];" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar,
                                              unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for phase `parity` of `bar` to complete; false if it did not within
// kStageWaitCycles.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar,
                                                  unsigned parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > kStageWaitCycles) return false;
    }
    return true;
}

// 16-byte unit of staged values, widened to FP32.
template <typename T>
__device__ __forceinline__ void unit_to_f(const uint4 &u, float *d) {
    constexpr int PW = Pack<T>::kPerWord;
    Pack<T>::unpack(u.x, d);
    Pack<T>::unpack(u.y, d + PW);
    Pack<T>::unpack(u.z, d + 2 * PW);
    Pack<T>::unpack(u.w, d + 3 * PW);
}

// Applies f(values, unit) to every staged unit this thread owns, U units'
// shared-memory reads in flight at a time.
template <typename T, int U, class F>
__device__ __forceinline__ void for_units(const uint4 *buf, int lo, int hi,
                                          int W, F f) {
    constexpr int V = 16 / (int)sizeof(T);
    int u = lo + (int)threadIdx.x;
    for (; u + (U - 1) * W < hi; u += U * W) {
        uint4 raw[U];
#pragma unroll
        for (int i = 0; i < U; ++i) raw[i] = buf[u + i * W];
#pragma unroll
        for (int i = 0; i < U; ++i) {
            float t[V];
            unit_to_f<T>(raw[i], t);
            f(t, u + i * W);
        }
    }
    for (; u < hi; u += W) {
        float t[V];
        unit_to_f<T>(buf[u], t);
        f(t, u);
    }
}

template <int OP>
__host__ __device__ constexpr bool stage_supported() {
    return OP == OP_RMSNORM || OP == OP_LAYERNORM || OP == OP_SOFTMAX ||
           OP == OP_LOG_SOFTMAX || OP == OP_CROSS_ENTROPY || OP == OP_ROW_SUM;
}

template <int OP, typename T, bool CL>
__global__ void __launch_bounds__(kStageMaxThreads)
    stage_kernel(const KArgs a) {
    static_assert(stage_supported<OP>(), "operator has no staged path");
    constexpr int V = 16 / (int)sizeof(T);
    constexpr int U = 4;
    extern __shared__ __align__(128) uint4 sbuf[];
    __shared__ __align__(8) uint64_t bars[kStagePiecesMax];
    __shared__ RedScratch red;
    int parity = 0, cpar = 0;
    const T *X = static_cast<const T *>(a.x);
    const T *Wt = static_cast<const T *>(a.w);
    const T *Bt = static_cast<const T *>(a.b);
    T *Y = static_cast<T *>(a.y);
    const int W = (int)blockDim.x;
    const int tid = (int)threadIdx.x;
    const int csize = CL ? a.csize : 1;
    const int rank = csize > 1 ? (int)cluster_ctarank() : 0;
    const int64_t g0 = csize > 1 ? (int64_t)cluster_id_x() : blockIdx.x;
    const int64_t gstride =
        csize > 1 ? (int64_t)num_clusters_x() : (int64_t)gridDim.x;
    const int cols = a.cols;
    // This CTA's run of 16-byte units and its pieces.
    const int units = cols / V;
    const int per = (units + csize - 1) / csize;
    const int u0 = rank * per < units ? rank * per : units;
    const int ucnt = (units - u0 < per ? units - u0 : per);
    const int npieces = a.pieces;
    const int upiece = (ucnt + npieces - 1) / npieces;
    auto piece_lo = [&](int j) { return j * upiece < ucnt ? j * upiece : ucnt; };
    auto piece_hi = [&](int j) {
        return (j + 1) * upiece < ucnt ? (j + 1) * upiece : ucnt;
    };

    if (tid == 0) {
        for (int j = 0; j < npieces; ++j) mbar_init(&bars[j], 1);
        mbar_init_fence();
    }
    if (a.pdl && tid == 0 && g0 < a.rows && ucnt > 0)
        prefetch_l2(X + g0 * (int64_t)cols + (int64_t)u0 * V,
                    (int64_t)ucnt * 16);
    __syncthreads();
    grid_launch_dependents();
    grid_wait_prerequisites();

    // A wait gave up: from the end of that row on, the CTA (every thread
    // agrees at the row's closing barrier) issues no copies and waits for
    // none; fail_ph is the parity of that row's barrier phases.
    bool failed = false;
    unsigned fail_ph = 0;
    unsigned ph = 0;           // phase parity of this row's barriers
    for (int64_t row = g0; row < a.rows; row += gstride, ph ^= 1u) {
        const T *xrow = X + row * (int64_t)cols;
        const T *xs = xrow + (int64_t)u0 * V;  // this CTA's run
        if (tid == 0 && !failed) {
            fence_proxy_async_smem();
            for (int j = 0; j < npieces; ++j) {
                const int lo = piece_lo(j), hi = piece_hi(j);
                if (hi <= lo) continue;
                const unsigned bytes = (unsigned)(hi - lo) * 16u;
                mbar_expect_tx(&bars[j], bytes);
                bulk_copy_g2s(sbuf + lo, xs + (int64_t)lo * V, bytes,
                              &bars[j]);
            }
            if (a.prefetch_next && row + gstride < a.rows && ucnt > 0)
                prefetch_l2(xs + gstride * (int64_t)cols, (int64_t)ucnt * 16);
        }
        // Waits for piece j of this row (every thread; bounded).  A thread
        // whose wait gives up reads whatever the run holds from then on.
        bool gave_up = failed;
        auto wait_piece = [&](int j) {
            if (piece_hi(j) <= piece_lo(j) || gave_up) return;
            if (!mbar_wait_bounded(&bars[j], ph)) {
                gave_up = true;
                atomicAdd(&g_stage_timeouts, 1ull);
            }
        };
        const int64_t ybase = row * (int64_t)cols + (int64_t)u0 * V;

        if constexpr (OP == OP_RMSNORM) {
            float ss = 0.f;
            for (int j = 0; j < npieces; ++j) {
                wait_piece(j);
                for_units<T, U>(sbuf, piece_lo(j), piece_hi(j), W,
                                [&](const float *t, int) {
#pragma unroll
                                    for (int e = 0; e < V; ++e)
                                        ss = fmaf(t[e], t[e], ss);
                                });
            }
            ss = team_allreduce<SumOp>(ss, W, csize, red, parity, cpar);
            const float r = rsqrtf(ss / (float)cols + a.eps);
            for_units<T, U>(sbuf, 0, ucnt, W, [&](const float *t, int u) {
                const int col = (u0 + u) * V;
                float wv[V], o[V];
                param_pack<T, V>(Wt, col, V, true, 1.f, wv);
#pragma unroll
                for (int e = 0; e < V; ++e) o[e] = t[e] * r * wv[e];
                st_vec<T, V>(Y + ybase + (int64_t)u * V, o);
            });
        } else if constexpr (OP == OP_LAYERNORM) {
            float mean, rstd;
            if constexpr (sizeof(T) == 2 && !CL) {
                // 16-bit rows on a lone CTA: the mean, then the squared
                // deviations about it, both from the staged run (measured
                // faster here than the one-pass form below).
                float s = 0.f;
                for (int j = 0; j < npieces; ++j) {
                    wait_piece(j);
                    for_units<T, U>(sbuf, piece_lo(j), piece_hi(j), W,
                                    [&](const float *t, int) {
#pragma unroll
                                        for (int e = 0; e < V; ++e) s += t[e];
                                    });
                }
                s = team_allreduce<SumOp>(s, W, csize, red, parity, cpar);
                mean = s / (float)cols;
                float q = 0.f;
                for_units<T, U>(sbuf, 0, ucnt, W, [&](const float *t, int) {
#pragma unroll
                    for (int e = 0; e < V; ++e) {
                        const float d = t[e] - mean;
                        q = fmaf(d, d, q);
                    }
                });
                q = team_allreduce<SumOp>(q, W, csize, red, parity, cpar);
                rstd = rsqrtf(q / (float)cols + a.eps);
            } else {
                // Shifted moments about the row's first value x0 (every CTA
                // of a cluster reads it from global memory; only rank 0
                // stages column 0): one pass and one reduction.  One
                // accumulator pair per value of a unit keeps the addition
                // chains short.
                const float x0 = to_f(xrow[0]);
                float s1v[V], s2v[V];
#pragma unroll
                for (int e = 0; e < V; ++e) s1v[e] = s2v[e] = 0.f;
                for (int j = 0; j < npieces; ++j) {
                    wait_piece(j);
                    for_units<T, U>(sbuf, piece_lo(j), piece_hi(j), W,
                                    [&](const float *t, int) {
#pragma unroll
                                        for (int e = 0; e < V; ++e) {
                                            const float d = t[e] - x0;
                                            s1v[e] += d;
                                            s2v[e] = fmaf(d, d, s2v[e]);
                                        }
                                    });
                }
                float s1 = 0.f, s2 = 0.f;
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    s1 += s1v[e];
                    s2 += s2v[e];
                }
                team_allreduce_sum2(s1, s2, W, csize, red, parity, cpar);
                const float md = s1 / (float)cols;
                mean = x0 + md;
                rstd = rsqrtf(fmaxf(fmaf(-md, md, s2 / (float)cols), 0.f) +
                              a.eps);
            }
            for_units<T, U>(sbuf, 0, ucnt, W, [&](const float *t, int u) {
                const int col = (u0 + u) * V;
                float gv[V], bv[V], o[V];
                param_pack<T, V>(Wt, col, V, true, 1.f, gv);
                param_pack<T, V>(Bt, col, V, true, 0.f, bv);
#pragma unroll
                for (int e = 0; e < V; ++e)
                    o[e] = fmaf((t[e] - mean) * rstd, gv[e], bv[e]);
                st_vec<T, V>(Y + ybase + (int64_t)u * V, o);
            });
        } else if constexpr (OP == OP_SOFTMAX || OP == OP_LOG_SOFTMAX ||
                             OP == OP_CROSS_ENTROPY) {
            // Running (max, sum of exp(x - max)) over the thread's units, as
            // on the loop path: the sum is rescaled only when a unit raises
            // the max.
            float m = -INFINITY, sm = 0.f;
            for (int j = 0; j < npieces; ++j) {
                wait_piece(j);
                for_units<T, U>(sbuf, piece_lo(j), piece_hi(j), W,
                                [&](const float *t, int) {
                                    float pm = -INFINITY;
#pragma unroll
                                    for (int e = 0; e < V; ++e)
                                        pm = nanmax(pm, t[e]);
                                    const float mm = nanmax(m, pm);
                                    if (mm != m) {
                                        sm *= exp_shifted(m - mm);
                                        m = mm;
                                    }
                                    if (m != -INFINITY) {
                                        float ps = 0.f;
#pragma unroll
                                        for (int e = 0; e < V; ++e)
                                            ps += exp_shifted(t[e] - m);
                                        sm += ps;
                                    }
                                });
            }
            team_allreduce_lse(m, sm, W, csize, red, parity, cpar);
            if constexpr (OP == OP_SOFTMAX) {
                const float inv = 1.f / sm;
                for_units<T, U>(sbuf, 0, ucnt, W,
                                [&](const float *t, int u) {
                                    float o[V];
#pragma unroll
                                    for (int e = 0; e < V; ++e)
                                        o[e] = exp_shifted(t[e] - m) * inv;
                                    st_vec<T, V>(Y + ybase + (int64_t)u * V,
                                                 o);
                                });
            } else if constexpr (OP == OP_LOG_SOFTMAX) {
                const float ls = logf(sm);
                for_units<T, U>(sbuf, 0, ucnt, W,
                                [&](const float *t, int u) {
                                    float o[V];
#pragma unroll
                                    for (int e = 0; e < V; ++e)
                                        o[e] = (t[e] - m) - ls;
                                    st_vec<T, V>(Y + ybase + (int64_t)u * V,
                                                 o);
                                });
            } else {
                if (rank == 0 && tid == 0) {
                    const int32_t lab = __ldg(a.labels + row);
                    const LabelInfo li = label_info(a, lab, cols);
                    const float xl = li.valid ? to_f(xrow[lab]) : NAN;
                    a.out[row] = li.ignored ? 0.f : (m + logf(sm)) - xl;
                }
            }
        } else if constexpr (OP == OP_ROW_SUM) {
            float s = 0.f, c = 0.f;
            for (int j = 0; j < npieces; ++j) {
                wait_piece(j);
                for_units<T, U>(sbuf, piece_lo(j), piece_hi(j), W,
                                [&](const float *t, int) {
#pragma unroll
                                    for (int e = 0; e < V; ++e) {
                                        float v, err;
                                        two_sum(s, t[e], v, err);
                                        s = v;
                                        c += err;
                                    }
                                });
            }
            team_allreduce_compensated(s, c, W, csize, red, parity, cpar);
            if (rank == 0 && tid == 0) a.out[row] = s + c;
        }
        // Every thread is done with the staged run before the next row's
        // copies overwrite it; the same barrier makes a give-up CTA-wide.
        const bool any = __syncthreads_or(gave_up) != 0;
        if (any && !failed) fail_ph = ph;
        failed = any;
    }
    // Copies of the row a wait gave up on may still land: wait for them
    // (bounded) before the shared memory goes away.
    if (tid == 0 && failed)
        for (int j = 0; j < npieces; ++j)
            if (piece_hi(j) > piece_lo(j))
                (void)mbar_wait_bounded(&bars[j], fail_ph);
    __syncthreads();
    // Peers may still read this CTA's cluster slots.
    if (csize > 1) cluster_sync();
}

}  // namespace mt
