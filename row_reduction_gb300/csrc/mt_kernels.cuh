// mt_kernels.cuh -- the per-row reduction kernels (sm_103a).
//
// Work mapping ("Consecutive-worker reduction layout checkpoint",
// §Implementation and semantics): a row is served by W consecutive threads
// ("workers"); worker w owns, in chunk k, the V consecutive elements
//     i = (k*W + w)*V + e,   0 <= e < V,
// of the row body, so with 16-byte packs (V=4 FP32, V=8 FP16/BF16) a warp's
// accesses of one chunk cover 512 contiguous bytes.  Complete packs take
// unguarded vector accesses; only the last, partial pack is guarded element
// by element.
//
// Storage types.  T is the element type of the matrices and parameter
// vectors (float, __half or __nv_bfloat16).  Every value is widened to FP32
// on load and every statistic and epilogue is computed in FP32; the only
// rounding to T is the final store ("FP32 reduction and epilogue arithmetic,
// rounding only on the output store", Thread Ownership and Software
// Staging, §Register-tiled reductions).  Per-row outputs (row sums, losses,
// the mean) are FP32 for every T.
//
// Alignment.  CUDA vector accesses must be naturally aligned.  When every
// row starts on a V*sizeof(T)-byte boundary (the "aligned" kernels:
// cols % V == 0 and aligned base pointers) the body is the whole row.
// Otherwise each row first peels a head of hd = (-row_address/sizeof(T))
// mod V scalar elements, owned one each by workers 0..hd-1, and the map
// above applies to the rest.
//
// Reduction ("Thread Ownership and Software Staging", §Register-tiled
// reductions): each thread combines its own slots, then the W lanes of a row
// combine with xor shuffles; for W > 32 each warp's lane 0 publishes one
// partial to shared memory, one __syncthreads() publishes them, and every
// warp reads all of its row's partials and finishes the reduction itself --
// no second barrier and no broadcast.  Consecutive reductions alternate
// between two scratch buffers, so the next reduction's barrier is what keeps
// a buffer from being overwritten before every warp has read it.
//
// Register path: the whole row (V*K values per thread) is loaded once,
// before any arithmetic, and the output is written from registers (the
// rmsnorm_register idea: "retains its input values across the reduction").
// Loop path: rows wider than the register budget are streamed in a strided
// loop; the normalising operators re-read x (from L2) to write y.
//
// Blocks hold B = blockDim / W row groups and loop over row groups with a
// grid stride, so a grid of "resident CTAs" is persistent.  All threads of
// a block run the same number of loop iterations (rows past the end are
// inactive but still take part in every shuffle and barrier).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>
#include <stdint.h>

#include "mt_internal.h"

namespace mt {

constexpr unsigned kFull = 0xffffffffu;

// NaN-propagating max: PTX max with the .NaN modifier returns NaN when
// either operand is NaN (fmaxf would drop it).  One instruction.
__device__ __forceinline__ float nanmax(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// NaN-propagating max over the 32 lanes of a warp, returned to every lane:
// one warp-wide reduction instruction (redux.sync on FP32, sm_100 family).
__device__ __forceinline__ float warp_nanmax(float v) {
    float r;
    asm volatile("redux.sync.max.NaN.f32 %0, %1, %2;"
                 : "=f"(r)
                 : "f"(v), "r"(kFull));
    return r;
}

// Error-free transformation of a + b (Knuth's two-sum): s + err == a + b
// exactly.  Used for the compensated row sum.
__device__ __forceinline__ void two_sum(float a, float b, float &s,
                                        float &err) {
    s = __fadd_rn(a, b);
    const float bp = __fsub_rn(s, a);
    const float ap = __fsub_rn(s, bp);
    err = __fadd_rn(__fsub_rn(a, ap), __fsub_rn(b, bp));
}

// e^d for d = x - max(row) <= 0, as 2^(d * log2(e)) with the PTX base-2
// exponential instruction ex2.approx.ftz.f32 (one MUFU operation; results
// below 2^-126 flush to zero, 2^-inf = 0, NaN stays NaN).  The difference d
// is formed first (exact when x is near the max), so the product adds a
// relative error of at most |d| * 2^-24, whose absolute effect on a term of
// weight e^d is at most 2^-24 / e; the instruction itself is an
// approximation within a few units in the last place.  Both are far below
// the FP32 tolerance of every output that sums or normalises these terms.
__device__ __forceinline__ float exp_shifted(float d) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(d * 1.4426950408889634f));
    return r;
}

// Operators that add a residual to x before normalising.
template <int OP>
__host__ __device__ constexpr bool has_residual() {
    return OP == OP_RESIDUAL_LAYERNORM || OP == OP_RESIDUAL_RMSNORM;
}

// Cross-entropy label handling: the logit of the label, 0-loss rows for the
// ignore index, NaN for any other label outside [0, cols).
struct LabelInfo {
    bool ignored;
    bool valid;
};
__device__ __forceinline__ LabelInfo label_info(const KArgs &a, int32_t lab,
                                                int cols) {
    LabelInfo li;
    li.ignored = a.has_ignore && lab == a.ignore_index;
    li.valid = lab >= 0 && lab < cols;
    return li;
}

// ---- storage types ---------------------------------------------------------
// Conversions between 32-bit words holding T values and FP32.
template <typename T>
struct Pack;

template <>
struct Pack<float> {
    static constexpr int kPerWord = 1;
    static __device__ __forceinline__ void unpack(unsigned w, float *d) {
        d[0] = __uint_as_float(w);
    }
    static __device__ __forceinline__ unsigned pack(const float *d) {
        return __float_as_uint(d[0]);
    }
    static __device__ __forceinline__ float scalar(float v) { return v; }
    static __device__ __forceinline__ float from(float v) { return v; }
};

template <>
struct Pack<__nv_bfloat16> {
    static constexpr int kPerWord = 2;
    // A bfloat16 is the high half of the FP32 with the same value.
    static __device__ __forceinline__ void unpack(unsigned w, float *d) {
        d[0] = __uint_as_float(w << 16);
        d[1] = __uint_as_float(w & 0xffff0000u);
    }
    static __device__ __forceinline__ unsigned pack(const float *d) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(d[0], d[1]);
        return *reinterpret_cast<const unsigned *>(&h);
    }
    static __device__ __forceinline__ float scalar(__nv_bfloat16 v) {
        return __bfloat162float(v);
    }
    static __device__ __forceinline__ __nv_bfloat16 from(float v) {
        return __float2bfloat16_rn(v);
    }
};

template <>
struct Pack<__half> {
    static constexpr int kPerWord = 2;
    static __device__ __forceinline__ void unpack(unsigned w, float *d) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w));
        d[0] = f.x;
        d[1] = f.y;
    }
    static __device__ __forceinline__ unsigned pack(const float *d) {
        const __half2 h = __floats2half2_rn(d[0], d[1]);
        return *reinterpret_cast<const unsigned *>(&h);
    }
    static __device__ __forceinline__ float scalar(__half v) {
        return __half2float(v);
    }
    static __device__ __forceinline__ __half from(float v) {
        return __float2half_rn(v);
    }
};

template <typename T>
__device__ __forceinline__ float to_f(T v) {
    return Pack<T>::scalar(v);
}
template <typename T>
__device__ __forceinline__ T from_f(float v) {
    return Pack<T>::from(v);
}

// ---- vector access ---------------------------------------------------------
// V values of type T at p (aligned to V*sizeof(T) bytes), widened to FP32.
// RO selects the read-only data path, used only for the parameter vectors,
// which no kernel writes.
template <typename T, int V, bool RO = false>
__device__ __forceinline__ void ld_vec(const T *p, float *d) {
    constexpr int kBytes = V * (int)sizeof(T);
    if constexpr (kBytes >= 4) {
        constexpr int NW = kBytes / 4;
        unsigned w[NW];
        if constexpr (NW == 4) {
            const uint4 u = RO ? __ldg(reinterpret_cast<const uint4 *>(p))
                               : *reinterpret_cast<const uint4 *>(p);
            w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
        } else if constexpr (NW == 2) {
            const uint2 u = RO ? __ldg(reinterpret_cast<const uint2 *>(p))
                               : *reinterpret_cast<const uint2 *>(p);
            w[0] = u.x; w[1] = u.y;
        } else {
            w[0] = RO ? __ldg(reinterpret_cast<const unsigned *>(p))
                      : *reinterpret_cast<const unsigned *>(p);
        }
#pragma unroll
        for (int i = 0; i < NW; ++i)
            Pack<T>::unpack(w[i], d + i * Pack<T>::kPerWord);
    } else {
        d[0] = to_f(RO ? __ldg(p) : *p);
    }
}

// V FP32 values rounded to T and stored at p (aligned to V*sizeof(T)).
template <typename T, int V>
__device__ __forceinline__ void st_vec(T *p, const float *d) {
    constexpr int kBytes = V * (int)sizeof(T);
    if constexpr (kBytes >= 4) {
        constexpr int NW = kBytes / 4;
        constexpr int PW = Pack<T>::kPerWord;
        unsigned w[NW];
#pragma unroll
        for (int i = 0; i < NW; ++i) w[i] = Pack<T>::pack(d + i * PW);
        if constexpr (NW == 4) {
            *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
        } else if constexpr (NW == 2) {
            *reinterpret_cast<uint2 *>(p) = make_uint2(w[0], w[1]);
        } else {
            *reinterpret_cast<unsigned *>(p) = w[0];
        }
    } else {
        *p = from_f<T>(d[0]);
    }
}

// Up to V values of a parameter vector starting at column `col`; only the
// first `nv` exist (the rest, and every value of a NULL vector, read as
// `dflt`).  `vec` says the address is V*sizeof(T)-byte aligned.
template <typename T, int V>
__device__ __forceinline__ void param_pack(const T *p, int col, int nv,
                                           bool vec, float dflt, float *d) {
    if (p == nullptr || nv <= 0) {
#pragma unroll
        for (int e = 0; e < V; ++e) d[e] = dflt;
    } else if (vec && nv == V) {
        ld_vec<T, V, true>(p + col, d);
    } else {
#pragma unroll
        for (int e = 0; e < V; ++e)
            d[e] = e < nv ? to_f(__ldg(p + col + e)) : dflt;
    }
}

template <typename T>
__device__ __forceinline__ float param_at(const T *p, int col, float dflt) {
    return p ? to_f(__ldg(p + col)) : dflt;
}

// ---- cooperative reductions ---------------------------------------------
struct SumOp {
    static constexpr bool kWarpRedux = false;
    __device__ __forceinline__ float operator()(float a, float b) const {
        return a + b;
    }
    static __device__ __forceinline__ float ident() { return 0.f; }
};
struct MaxOp {
    // A full warp reduces with one redux.sync instead of a butterfly.
    static constexpr bool kWarpRedux = true;
    __device__ __forceinline__ float operator()(float a, float b) const {
        return nanmax(a, b);
    }
    static __device__ __forceinline__ float ident() { return -INFINITY; }
};

struct RedScratch {
    float buf[2][2][32];  // [alternating buffer][component][warp]
    float cl[2][2];       // cluster exchange: [alternating buffer][component]
};

// All-reduce of one value over the W threads of each row; every thread of
// the row returns the same bits.
template <class Op>
__device__ __forceinline__ float row_allreduce(float v, int W,
                                               RedScratch &red,
                                               int &parity) {
    Op op;
    if (W < 32 || (W == 32 && !Op::kWarpRedux)) {
        for (int off = W >> 1; off > 0; off >>= 1)
            v = op(v, __shfl_xor_sync(kFull, v, off));
        return v;
    }
    if constexpr (Op::kWarpRedux) {
        v = warp_nanmax(v);
    } else {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            v = op(v, __shfl_xor_sync(kFull, v, off));
    }
    if (W == 32) return v;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nw = W >> 5;
    float *buf = red.buf[parity][0];
    parity ^= 1;
    if (lane == 0) buf[warp] = v;
    __syncthreads();
    const int first = warp & ~(nw - 1);
    float t = lane < nw ? buf[first + lane] : Op::ident();
    if constexpr (Op::kWarpRedux) return warp_nanmax(t);
    for (int off = nw >> 1; off > 0; off >>= 1)
        t = op(t, __shfl_xor_sync(kFull, t, off));
    return __shfl_sync(kFull, t, 0);
}

// Compensated (sum, error) pairs: (s1,c1)+(s2,c2) = two_sum(s1,s2) with the
// rounding error folded into the compensation term.
__device__ __forceinline__ void pair_add(float &s, float &c, float s2,
                                         float c2) {
    float t, e;
    two_sum(s, s2, t, e);
    s = t;
    c = c + c2 + e;
}

__device__ __forceinline__ void row_allreduce_compensated(float &s, float &c,
                                                          int W,
                                                          RedScratch &red,
                                                          int &parity) {
    if (W <= 32) {
        for (int off = W >> 1; off > 0; off >>= 1) {
            const float s2 = __shfl_xor_sync(kFull, s, off);
            const float c2 = __shfl_xor_sync(kFull, c, off);
            pair_add(s, c, s2, c2);
        }
        return;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float s2 = __shfl_xor_sync(kFull, s, off);
        const float c2 = __shfl_xor_sync(kFull, c, off);
        pair_add(s, c, s2, c2);
    }
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nw = W >> 5;
    float(*buf)[32] = red.buf[parity];
    parity ^= 1;
    if (lane == 0) {
        buf[0][warp] = s;
        buf[1][warp] = c;
    }
    __syncthreads();
    const int first = warp & ~(nw - 1);
    float ts = lane < nw ? buf[0][first + lane] : 0.f;
    float tc = lane < nw ? buf[1][first + lane] : 0.f;
    for (int off = nw >> 1; off > 0; off >>= 1) {
        const float s2 = __shfl_xor_sync(kFull, ts, off);
        const float c2 = __shfl_xor_sync(kFull, tc, off);
        pair_add(ts, tc, s2, c2);
    }
    s = __shfl_sync(kFull, ts, 0);
    c = __shfl_sync(kFull, tc, 0);
}

// Online (max, sum of exp(x - max)) pairs for softmax / cross-entropy on the
// loop path: (m1,s1) + (m2,s2) = (m, s1*e^(m1-m) + s2*e^(m2-m)).
// `self_first` fixes the operand order of the final fused multiply-add, so
// the two lanes of a shuffle pair compute the same bits.
__device__ __forceinline__ void lse_merge(float &m, float &s, float m2,
                                          float s2, bool self_first = true) {
    const float mm = nanmax(m, m2);
    const float f1 = (m == mm) ? 1.f : exp_shifted(m - mm);
    const float f2 = (m2 == mm) ? 1.f : exp_shifted(m2 - mm);
    s = self_first ? fmaf(s, f1, s2 * f2) : fmaf(s2, f2, s * f1);
    m = mm;
}

__device__ __forceinline__ void row_allreduce_lse(float &m, float &s, int W,
                                                  RedScratch &red,
                                                  int &parity) {
    const int lane = threadIdx.x & 31;
    if (W <= 32) {
        for (int off = W >> 1; off > 0; off >>= 1) {
            const float m2 = __shfl_xor_sync(kFull, m, off);
            const float s2 = __shfl_xor_sync(kFull, s, off);
            lse_merge(m, s, m2, s2, (lane & off) == 0);
        }
        return;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float m2 = __shfl_xor_sync(kFull, m, off);
        const float s2 = __shfl_xor_sync(kFull, s, off);
        lse_merge(m, s, m2, s2, (lane & off) == 0);
    }
    const int warp = threadIdx.x >> 5;
    const int nw = W >> 5;
    float(*buf)[32] = red.buf[parity];
    parity ^= 1;
    if (lane == 0) {
        buf[0][warp] = m;
        buf[1][warp] = s;
    }
    __syncthreads();
    const int first = warp & ~(nw - 1);
    float tm = lane < nw ? buf[0][first + lane] : -INFINITY;
    float ts = lane < nw ? buf[1][first + lane] : 0.f;
    for (int off = nw >> 1; off > 0; off >>= 1) {
        const float m2 = __shfl_xor_sync(kFull, tm, off);
        const float s2 = __shfl_xor_sync(kFull, ts, off);
        lse_merge(tm, ts, m2, s2, (lane & off) == 0);
    }
    m = __shfl_sync(kFull, tm, 0);
    s = __shfl_sync(kFull, ts, 0);
}

// ---- split rows: thread-block clusters -------------------------------------
// With a cluster of `csize` CTAs per row, each CTA reduces its slice of the
// row as above, thread 0 publishes the CTA total in its own shared memory,
// one cluster barrier (release/acquire) makes the totals visible, and every
// CTA reads all csize totals through distributed shared memory and combines
// them in rank order -- the same single-barrier, private-scratch scheme as
// the cross-warp stage, one level up.  Consecutive cluster reductions
// alternate between two slots, so the next cluster barrier keeps a slot from
// being rewritten before every peer has read it; a last cluster barrier
// before exit keeps each CTA's shared memory alive until its peers are done.
// Every CTA of a cluster runs the same number of loop iterations and hence
// the same number of cluster barriers.
__device__ __forceinline__ unsigned cluster_ctarank() {
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ unsigned cluster_id_x() {
    unsigned r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ unsigned num_clusters_x() {
    unsigned r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n\t"
        "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Reads a float at the same shared-memory offset in the CTA of cluster rank
// `rank`.
__device__ __forceinline__ float ld_cluster(const float *p, unsigned rank) {
    const unsigned la = (unsigned)__cvta_generic_to_shared(p);
    unsigned ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(ra)
                 : "r"(la), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];"
                 : "=f"(v)
                 : "r"(ra)
                 : "memory");
    return v;
}

// Row all-reduces over a team: the W threads of this CTA, then (csize > 1)
// the csize CTAs of the cluster.  `cpar` alternates the cluster slots.
template <class Op>
__device__ __forceinline__ float team_allreduce(float v, int W, int csize,
                                                RedScratch &red, int &parity,
                                                int &cpar) {
    v = row_allreduce<Op>(v, W, red, parity);
    if (csize > 1) {
        Op op;
        if (threadIdx.x == 0) red.cl[cpar][0] = v;
        cluster_sync();
        const int lane = threadIdx.x & 31;
        float t = lane < csize ? ld_cluster(&red.cl[cpar][0], lane)
                               : Op::ident();
        for (int off = csize >> 1; off > 0; off >>= 1)
            t = op(t, __shfl_xor_sync(kFull, t, off));
        v = __shfl_sync(kFull, t, 0);
        cpar ^= 1;
    }
    return v;
}

// Row all-reduce of two sums at once (one shared-memory publication, one
// barrier, one cluster barrier), in the same fixed order as team_allreduce.
__device__ __forceinline__ void team_allreduce_sum2(float &a, float &b, int W,
                                                    int csize,
                                                    RedScratch &red,
                                                    int &parity, int &cpar) {
    if (W <= 32) {
        for (int off = W >> 1; off > 0; off >>= 1) {
            a += __shfl_xor_sync(kFull, a, off);
            b += __shfl_xor_sync(kFull, b, off);
        }
    } else {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            a += __shfl_xor_sync(kFull, a, off);
            b += __shfl_xor_sync(kFull, b, off);
        }
        const int lane = threadIdx.x & 31;
        const int warp = threadIdx.x >> 5;
        const int nw = W >> 5;
        float(*buf)[32] = red.buf[parity];
        parity ^= 1;
        if (lane == 0) {
            buf[0][warp] = a;
            buf[1][warp] = b;
        }
        __syncthreads();
        const int first = warp & ~(nw - 1);
        float ta = lane < nw ? buf[0][first + lane] : 0.f;
        float tb = lane < nw ? buf[1][first + lane] : 0.f;
        for (int off = nw >> 1; off > 0; off >>= 1) {
            ta += __shfl_xor_sync(kFull, ta, off);
            tb += __shfl_xor_sync(kFull, tb, off);
        }
        a = __shfl_sync(kFull, ta, 0);
        b = __shfl_sync(kFull, tb, 0);
    }
    if (csize > 1) {
        if (threadIdx.x == 0) {
            red.cl[cpar][0] = a;
            red.cl[cpar][1] = b;
        }
        cluster_sync();
        const int lane = threadIdx.x & 31;
        float ta = lane < csize ? ld_cluster(&red.cl[cpar][0], lane) : 0.f;
        float tb = lane < csize ? ld_cluster(&red.cl[cpar][1], lane) : 0.f;
        for (int off = csize >> 1; off > 0; off >>= 1) {
            ta += __shfl_xor_sync(kFull, ta, off);
            tb += __shfl_xor_sync(kFull, tb, off);
        }
        a = __shfl_sync(kFull, ta, 0);
        b = __shfl_sync(kFull, tb, 0);
        cpar ^= 1;
    }
}

__device__ __forceinline__ void team_allreduce_compensated(
    float &s, float &c, int W, int csize, RedScratch &red, int &parity,
    int &cpar) {
    row_allreduce_compensated(s, c, W, red, parity);
    if (csize > 1) {
        if (threadIdx.x == 0) {
            red.cl[cpar][0] = s;
            red.cl[cpar][1] = c;
        }
        cluster_sync();
        const int lane = threadIdx.x & 31;
        float ts = lane < csize ? ld_cluster(&red.cl[cpar][0], lane) : 0.f;
        float tc = lane < csize ? ld_cluster(&red.cl[cpar][1], lane) : 0.f;
        for (int off = csize >> 1; off > 0; off >>= 1) {
            const float s2 = __shfl_xor_sync(kFull, ts, off);
            const float c2 = __shfl_xor_sync(kFull, tc, off);
            pair_add(ts, tc, s2, c2);
        }
        s = __shfl_sync(kFull, ts, 0);
        c = __shfl_sync(kFull, tc, 0);
        cpar ^= 1;
    }
}

__device__ __forceinline__ void team_allreduce_lse(float &m, float &s, int W,
                                                   int csize, RedScratch &red,
                                                   int &parity, int &cpar) {
    row_allreduce_lse(m, s, W, red, parity);
    if (csize > 1) {
        if (threadIdx.x == 0) {
            red.cl[cpar][0] = m;
            red.cl[cpar][1] = s;
        }
        cluster_sync();
        const int lane = threadIdx.x & 31;
        float tm = lane < csize ? ld_cluster(&red.cl[cpar][0], lane)
                                : -INFINITY;
        float ts = lane < csize ? ld_cluster(&red.cl[cpar][1], lane) : 0.f;
        for (int off = csize >> 1; off > 0; off >>= 1) {
            const float m2 = __shfl_xor_sync(kFull, tm, off);
            const float s2 = __shfl_xor_sync(kFull, ts, off);
            lse_merge(tm, ts, m2, s2, (lane & off) == 0);
        }
        m = __shfl_sync(kFull, tm, 0);
        s = __shfl_sync(kFull, ts, 0);
        cpar ^= 1;
    }
}

// ---- launch overlap ---------------------------------------------------------
// Programmatic dependent launch: the next kernel on the stream may start as
// soon as every CTA of this one has started; griddepcontrol.wait then holds
// it until this grid has completed and its writes are visible.  Without the
// launch attribute both instructions have no effect.
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_wait_prerequisites() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Asks L2 to fetch the 16-byte-aligned interior of [p, p + bytes) with bulk
// prefetches of at most 64 KiB each.  A prefetch changes no value, so it may
// run before the wait on the previous grid.
__device__ __forceinline__ void prefetch_l2(const void *p, int64_t bytes) {
    uintptr_t s = (reinterpret_cast<uintptr_t>(p) + 15) & ~(uintptr_t)15;
    const uintptr_t e =
        (reinterpret_cast<uintptr_t>(p) + (uintptr_t)bytes) & ~(uintptr_t)15;
    while (s < e) {
        const uintptr_t n = e - s < 65536 ? e - s : 65536;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(s),
                     "r"((unsigned)n)
                     : "memory");
        s += n;
    }
}

// L2 prefetch of row group g (x and, for residual LayerNorm, the residual).
template <int OP, typename T>
__device__ __forceinline__ void prefetch_group(const KArgs &a, int64_t g) {
    const int64_t r0 = g * a.B;
    if (r0 >= a.rows) return;
    const int64_t nr = a.rows - r0 < a.B ? a.rows - r0 : a.B;
    const int64_t bytes = nr * (int64_t)a.cols * (int64_t)sizeof(T);
    prefetch_l2(static_cast<const T *>(a.x) + r0 * a.cols, bytes);
    if constexpr (has_residual<OP>())
        prefetch_l2(static_cast<const T *>(a.res) + r0 * a.cols, bytes);
}

// Persistent CTAs: with `prefetch_next`, thread 0 (of cluster rank 0) asks
// L2 for the row group processed after `g`, so its DRAM reads overlap this
// one.
template <int OP, typename T>
__device__ __forceinline__ void prefetch_next_group(const KArgs &a,
                                                    int64_t g,
                                                    int64_t ngroups,
                                                    int64_t gstride,
                                                    int rank) {
    const int64_t gn = g + gstride;
    if (!a.prefetch_next || threadIdx.x != 0 || rank != 0 || gn >= ngroups)
        return;
    prefetch_group<OP, T>(a, gn);
}

// Kernel prologue: with `pdl`, thread 0 (of cluster rank 0) prefetches the
// first row group into L2; then every thread lets dependents launch and
// waits for the previous grid.
template <int OP, typename T, bool CL>
__device__ __forceinline__ void kernel_prologue(const KArgs &a) {
    if (a.pdl && threadIdx.x == 0) {
        if (CL && a.csize > 1) {
            if (cluster_ctarank() == 0) prefetch_group<OP, T>(a, cluster_id_x());
        } else {
            prefetch_group<OP, T>(a, blockIdx.x);
        }
    }
    grid_launch_dependents();
    grid_wait_prerequisites();
}

// ---- per-row geometry ------------------------------------------------------
template <typename T, int V, bool AL>
struct RowGeom {
    int64_t base;  // element offset of the row
    int hd;        // head length (unaligned kernels only)
    int nb;        // body length
    __device__ __forceinline__ RowGeom(const T *x, int64_t row, int cols) {
        base = row * (int64_t)cols;
        hd = 0;
        if constexpr (!AL && V > 1) {
            const unsigned elems = (unsigned)(
                reinterpret_cast<uintptr_t>(x + base) / sizeof(T));
            hd = (int)((0u - elems) & (unsigned)(V - 1));
            hd = hd < cols ? hd : cols;
        }
        nb = cols - hd;
    }
};

// Loads V consecutive values at body offset `off` of a row (`p` = row
// start + head): a vector access for a complete pack when `vec`, otherwise
// guarded scalars; missing values read as `fill`.  In aligned kernels
// (AL) cols % V == 0, so a pack is either complete or wholly past the end.
template <typename T, int V, bool AL, bool FU = false>
__device__ __forceinline__ void load_pack(const T *p, int off, int nb,
                                          bool active, bool vec, float fill,
                                          float *d) {
    if constexpr (FU) {
        ld_vec<T, V>(p + off, d);
    } else if constexpr (AL) {
        if (active && off < nb) {
            ld_vec<T, V>(p + off, d);
        } else {
#pragma unroll
            for (int e = 0; e < V; ++e) d[e] = fill;
        }
    } else if (active && off + V <= nb) {
        if (vec) {
            ld_vec<T, V>(p + off, d);
        } else {
#pragma unroll
            for (int e = 0; e < V; ++e) d[e] = to_f(p[off + e]);
        }
    } else {
#pragma unroll
        for (int e = 0; e < V; ++e)
            d[e] = (active && off + e < nb) ? to_f(p[off + e]) : fill;
    }
}

template <typename T, int V, bool AL, bool FU = false>
__device__ __forceinline__ void store_pack(T *p, int off, int nb,
                                           bool active, bool vec,
                                           const float *d) {
    if constexpr (FU) {
        st_vec<T, V>(p + off, d);
        return;
    }
    if (!active) return;
    if constexpr (AL) {
        if (off < nb) st_vec<T, V>(p + off, d);
    } else if (off + V <= nb) {
        if (vec) {
            st_vec<T, V>(p + off, d);
        } else {
#pragma unroll
            for (int e = 0; e < V; ++e) p[off + e] = from_f<T>(d[e]);
        }
    } else {
#pragma unroll
        for (int e = 0; e < V; ++e)
            if (off + e < nb) p[off + e] = from_f<T>(d[e]);
    }
}

// Parameter pack for the register path: aligned kernels read complete
// vectors (or nothing past the end), the others guard each element; whole-
// tile kernels (FU) read every pack of a vector that is known to exist.
template <typename T, int V, bool AL, bool FU = false>
__device__ __forceinline__ void param_row_pack(const T *p, int col,
                                               int off, int nb, bool active,
                                               float dflt, float *d) {
    if constexpr (FU) {
        ld_vec<T, V, true>(p + col, d);
    } else if constexpr (AL) {
        if (p != nullptr && active && off < nb) {
            ld_vec<T, V, true>(p + col, d);
        } else {
#pragma unroll
            for (int e = 0; e < V; ++e) d[e] = dflt;
        }
    } else {
        const int nv = active ? min(max(nb - off, 0), V) : 0;
        param_pack<T, V>(p, col, nv, false, dflt, d);
    }
}

// =========================================================================
// Register path
// =========================================================================
template <int OP, typename T, int V, int K, bool AL, bool CL, bool FU>
__device__ __forceinline__ void reg_body(const KArgs &a) {
    static_assert(!FU || (AL && !CL), "whole-tile kernels are aligned, "
                                      "one CTA per row group");
    kernel_prologue<OP, T, CL>(a);
    __shared__ RedScratch red;
    int parity = 0;
    const T *X = static_cast<const T *>(a.x);
    const T *Wt = static_cast<const T *>(a.w);
    const T *Bt = static_cast<const T *>(a.b);
    T *Y = static_cast<T *>(a.y);
    const int W = a.W;             // threads of this CTA per row
    // CTAs per row (thread-block cluster); the CL=false kernels fold every
    // cluster step away.
    const int csize = CL ? a.csize : 1;
    const int rank = csize > 1 ? (int)cluster_ctarank() : 0;
    const int WT = W * csize;      // workers per row
    const int worker = rank * W + (int)(threadIdx.x & (W - 1));
    const int slot = threadIdx.x >> a.log2W;
    const int64_t g0 = csize > 1 ? (int64_t)cluster_id_x() : blockIdx.x;
    const int64_t gstride =
        csize > 1 ? (int64_t)num_clusters_x() : (int64_t)gridDim.x;
    int cpar = 0;
    const int cols = a.cols;
    const int64_t ngroups = (a.rows + a.B - 1) / a.B;
    constexpr bool kMaxFill = (OP == OP_SOFTMAX || OP == OP_CROSS_ENTROPY ||
                               OP == OP_LOG_SOFTMAX);
    const float fill = kMaxFill ? -INFINITY : 0.f;
    constexpr bool kHead = !AL && V > 1;
    const bool yvec = AL || a.y_vec;

    for (int64_t g = g0; g < ngroups; g += gstride) {
        prefetch_next_group<OP, T>(a, g, ngroups, gstride, rank);
        const int64_t row = g * a.B + slot;
        const bool active = FU || row < a.rows;
        const RowGeom<T, V, AL> geo(X, active ? row : 0, cols);
        const T *xb = X + geo.base + geo.hd;  // body start
        const int nb = geo.nb;
        const bool head = kHead && active && worker < geo.hd;

        // LayerNorm's pivot, the row's first value: loaded ahead of the
        // row so that its latency hides under the row's own.
        float piv = 0.f;
        if constexpr (OP == OP_LAYERNORM || OP == OP_RESIDUAL_LAYERNORM) {
            piv = to_f(X[geo.base]);
            if constexpr (has_residual<OP>())
                piv = __fadd_rn(piv,
                                to_f(static_cast<const T *>(a.res)[geo.base]));
        }

        // ---- single read of the row into registers --------------------
        float v[K][V];
        float hv = fill;
#pragma unroll
        for (int k = 0; k < K; ++k)
            load_pack<T, V, AL, FU>(xb, (k * WT + worker) * V, nb, active, true,
                                fill, v[k]);
        if (head) hv = to_f(X[geo.base + worker]);

        if constexpr (has_residual<OP>()) {
            const T *R = static_cast<const T *>(a.res);
            const T *rb = R + geo.base + geo.hd;
            const bool rvec = AL || a.r_vec;
#pragma unroll
            for (int k = 0; k < K; ++k) {
                float t[V];
                load_pack<T, V, AL, FU>(rb, (k * WT + worker) * V, nb, active,
                                    rvec, 0.f, t);
#pragma unroll
                for (int e = 0; e < V; ++e) v[k][e] = __fadd_rn(v[k][e], t[e]);
            }
            if (head) hv = __fadd_rn(hv, to_f(R[geo.base + worker]));
            if (a.h != nullptr) {
                T *H = static_cast<T *>(a.h);
                T *hb = H + geo.base + geo.hd;
                const bool hvec = AL || a.h_vec;
#pragma unroll
                for (int k = 0; k < K; ++k)
                    store_pack<T, V, AL, FU>(hb, (k * WT + worker) * V, nb, active,
                                         hvec, v[k]);
                if (head) H[geo.base + worker] = from_f<T>(hv);
            }
        }

        // Cross-entropy: fetch the label and its logit while the row loads
        // are in flight.
        float xl = 0.f;
        bool ignored = false;
        if constexpr (OP == OP_CROSS_ENTROPY) {
            if (active && worker == 0) {
                const int32_t lab = __ldg(a.labels + row);
                const LabelInfo li = label_info(a, lab, cols);
                ignored = li.ignored;
                xl = li.valid ? to_f(X[geo.base + lab]) : NAN;
            }
        }

        // ---- per-operator reduction and epilogue ----------------------
        if constexpr (OP == OP_RMSNORM || OP == OP_RESIDUAL_RMSNORM) {
            float acc[V];
#pragma unroll
            for (int e = 0; e < V; ++e) acc[e] = 0.f;
#pragma unroll
            for (int k = 0; k < K; ++k)
#pragma unroll
                for (int e = 0; e < V; ++e)
                    acc[e] = fmaf(v[k][e], v[k][e], acc[e]);
            float ss = hv * hv;
#pragma unroll
            for (int e = 0; e < V; ++e) ss += acc[e];
            ss = team_allreduce<SumOp>(ss, W, csize, red, parity, cpar);
            const float r = rsqrtf(ss / (float)cols + a.eps);
            T *yb = Y + geo.base + geo.hd;
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int off = (k * WT + worker) * V;
                float wv[V], o[V];
                param_row_pack<T, V, AL, FU>(Wt, geo.hd + off, off, nb, active,
                                         1.f, wv);
#pragma unroll
                for (int e = 0; e < V; ++e) o[e] = v[k][e] * r * wv[e];
                store_pack<T, V, AL, FU>(yb, off, nb, active, yvec, o);
            }
            if (head)
                Y[geo.base + worker] =
                    from_f<T>(hv * r * param_at(Wt, worker, 1.f));
        } else if constexpr (OP == OP_LAYERNORM ||
                             OP == OP_RESIDUAL_LAYERNORM) {
            // Shifted moments: the sums of d = x - x0 and d^2 about the
            // row's first value x0 (every thread reads it: a cache hit)
            // in one reduction of two values, then mean = x0 + mean(d) and
            // var = mean(d^2) - mean(d)^2.  x0 lies in the row's spread, so
            // the subtraction loses no more than a few units of the
            // spread's own rounding.
            const float x0 = piv;
            float s1v[V], s2v[V];
#pragma unroll
            for (int e = 0; e < V; ++e) s1v[e] = s2v[e] = 0.f;
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int off = (k * WT + worker) * V;
                // Aligned rows hold whole packs, so one test per pack.
                const bool pack_in = active && off < nb;
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    const float d = v[k][e] - x0;
                    if (FU || (AL ? pack_in : (active && off + e < nb))) {
                        s1v[e] += d;
                        s2v[e] = fmaf(d, d, s2v[e]);
                    }
                }
            }
            float s1 = 0.f, s2 = 0.f;
            if (head) {
                const float d = hv - x0;
                s1 = d;
                s2 = d * d;
            }
#pragma unroll
            for (int e = 0; e < V; ++e) {
                s1 += s1v[e];
                s2 += s2v[e];
            }
            team_allreduce_sum2(s1, s2, W, csize, red, parity, cpar);
            const float md = s1 / (float)cols;
            const float var = fmaxf(fmaf(-md, md, s2 / (float)cols), 0.f);
            const float mean = x0 + md;
            const float rstd = rsqrtf(var + a.eps);
            T *yb = Y + geo.base + geo.hd;
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int off = (k * WT + worker) * V;
                float gv[V], bv[V], o[V];
                param_row_pack<T, V, AL, FU>(Wt, geo.hd + off, off, nb, active,
                                         1.f, gv);
                param_row_pack<T, V, AL, FU>(Bt, geo.hd + off, off, nb, active,
                                         0.f, bv);
#pragma unroll
                for (int e = 0; e < V; ++e)
                    o[e] = fmaf((v[k][e] - mean) * rstd, gv[e], bv[e]);
                store_pack<T, V, AL, FU>(yb, off, nb, active, yvec, o);
            }
            if (head)
                Y[geo.base + worker] = from_f<T>(
                    fmaf((hv - mean) * rstd, param_at(Wt, worker, 1.f),
                         param_at(Bt, worker, 0.f)));
        } else if constexpr (OP == OP_SOFTMAX) {
            float mx[V];
#pragma unroll
            for (int e = 0; e < V; ++e) mx[e] = hv;
#pragma unroll
            for (int k = 0; k < K; ++k)
#pragma unroll
                for (int e = 0; e < V; ++e) mx[e] = nanmax(mx[e], v[k][e]);
            float m = mx[0];
#pragma unroll
            for (int e = 1; e < V; ++e) m = nanmax(m, mx[e]);
            m = team_allreduce<MaxOp>(m, W, csize, red, parity, cpar);
            float acc[V];
#pragma unroll
            for (int e = 0; e < V; ++e) acc[e] = 0.f;
#pragma unroll
            for (int k = 0; k < K; ++k)
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    v[k][e] = exp_shifted(v[k][e] - m);
                    acc[e] += v[k][e];
                }
            float s = 0.f;
            if (head) {
                hv = exp_shifted(hv - m);
                s = hv;
            }
#pragma unroll
            for (int e = 0; e < V; ++e) s += acc[e];
            s = team_allreduce<SumOp>(s, W, csize, red, parity, cpar);
            const float inv = 1.f / s;
            T *yb = Y + geo.base + geo.hd;
#pragma unroll
            for (int k = 0; k < K; ++k) {
                float o[V];
#pragma unroll
                for (int e = 0; e < V; ++e) o[e] = v[k][e] * inv;
                store_pack<T, V, AL, FU>(yb, (k * WT + worker) * V, nb, active,
                                     yvec, o);
            }
            if (head) Y[geo.base + worker] = from_f<T>(hv * inv);
        } else if constexpr (OP == OP_ROW_SUM) {
            // Pairwise tree of error-free additions over the thread's V*K
            // values (independent at every level, so every load is in
            // flight before the first addition); the rounding errors of
            // the tree are summed separately and carried as the
            // compensation term.
            float c = 0.f;
#pragma unroll
            for (int step = 1; step < K * V; step <<= 1)
#pragma unroll
                for (int i = 0; i + step < K * V; i += 2 * step) {
                    float t, err;
                    two_sum(v[i / V][i % V], v[(i + step) / V][(i + step) % V],
                            t, err);
                    v[i / V][i % V] = t;
                    c += err;
                }
            float s, err;
            two_sum(v[0][0], hv, s, err);
            c += err;
            team_allreduce_compensated(s, c, W, csize, red, parity, cpar);
            if (active && worker == 0) a.out[row] = s + c;
        } else if constexpr (OP == OP_CROSS_ENTROPY) {
            float mx[V];
#pragma unroll
            for (int e = 0; e < V; ++e) mx[e] = hv;
#pragma unroll
            for (int k = 0; k < K; ++k)
#pragma unroll
                for (int e = 0; e < V; ++e) mx[e] = nanmax(mx[e], v[k][e]);
            float m = mx[0];
#pragma unroll
            for (int e = 1; e < V; ++e) m = nanmax(m, mx[e]);
            m = team_allreduce<MaxOp>(m, W, csize, red, parity, cpar);
            float acc[V];
#pragma unroll
            for (int e = 0; e < V; ++e) acc[e] = 0.f;
#pragma unroll
            for (int k = 0; k < K; ++k)
#pragma unroll
                for (int e = 0; e < V; ++e) acc[e] += exp_shifted(v[k][e] - m);
            float s = head ? exp_shifted(hv - m) : 0.f;
#pragma unroll
            for (int e = 0; e < V; ++e) s += acc[e];
            s = team_allreduce<SumOp>(s, W, csize, red, parity, cpar);
            if (active && worker == 0)
                a.out[row] = ignored ? 0.f : (m + logf(s)) - xl;
        } else if constexpr (OP == OP_LOG_SOFTMAX) {
            float mx[V];
#pragma unroll
            for (int e = 0; e < V; ++e) mx[e] = hv;
#pragma unroll
            for (int k = 0; k < K; ++k)
#pragma unroll
                for (int e = 0; e < V; ++e) mx[e] = nanmax(mx[e], v[k][e]);
            float m = mx[0];
#pragma unroll
            for (int e = 1; e < V; ++e) m = nanmax(m, mx[e]);
            m = team_allreduce<MaxOp>(m, W, csize, red, parity, cpar);
            float acc[V];
#pragma unroll
            for (int e = 0; e < V; ++e) acc[e] = 0.f;
#pragma unroll
            for (int k = 0; k < K; ++k)
#pragma unroll
                for (int e = 0; e < V; ++e) acc[e] += exp_shifted(v[k][e] - m);
            float s = head ? exp_shifted(hv - m) : 0.f;
#pragma unroll
            for (int e = 0; e < V; ++e) s += acc[e];
            s = team_allreduce<SumOp>(s, W, csize, red, parity, cpar);
            const float ls = logf(s);
            T *yb = Y + geo.base + geo.hd;
#pragma unroll
            for (int k = 0; k < K; ++k) {
                float o[V];
#pragma unroll
                for (int e = 0; e < V; ++e) o[e] = (v[k][e] - m) - ls;
                store_pack<T, V, AL, FU>(yb, (k * WT + worker) * V, nb, active,
                                     yvec, o);
            }
            if (head) Y[geo.base + worker] = from_f<T>((hv - m) - ls);
        }
    }
    // Peers may still read this CTA's cluster slots.
    if (csize > 1) cluster_sync();
}

template <int OP, typename T, int V, int K, bool AL, bool CL>
__global__ void __launch_bounds__(reg_max_threads(V * K))
    reg_kernel(const KArgs a) {
    reg_body<OP, T, V, K, AL, CL, false>(a);
}

// Whole tiles (every pack of every row exists, every parameter vector is
// present): the same row program with no bounds guard.
template <int OP, typename T, int V, int K>
__global__ void __launch_bounds__(reg_max_threads(V * K))
    reg_full_kernel(const KArgs a) {
    reg_body<OP, T, V, K, true, false, true>(a);
}

// The same with a register cap (where reg_full_capped applies; the cap
// also admits the largest CTA the thread bound allows).
template <int OP, typename T, int V, int K>
__global__ void __maxnreg__(kFullCapRegs)
    reg_full_capped_kernel(const KArgs a) {
    static_assert(kFullCapRegs * 512 <= 65536,
                  "the cap must admit the largest CTA (512 threads)");
    reg_body<OP, T, V, K, true, false, true>(a);
}

// =========================================================================
// Loop path (rows wider than the register budget)
// =========================================================================
// Calls f(vals, nvalid, off) for every pack of the thread's part of the row
// body, U packs' loads in flight at a time; then the head element, if any,
// as f(&hv, 1, -1 - worker) (off < 0 marks the head: column = -1 - off).
template <int V, bool AL, int U, class LoadF, class F>
__device__ __forceinline__ void stream_row(int worker, int W, int hd, int nb,
                                           bool active, LoadF load, F f) {
    if (!active) return;
    int64_t p = worker;
    const int64_t step = (int64_t)U * W;
    for (; (p + (int64_t)(U - 1) * W + 1) * V <= nb; p += step) {
        float t[U][V];
#pragma unroll
        for (int u = 0; u < U; ++u) load((int)((p + u * W) * V), V, t[u]);
#pragma unroll
        for (int u = 0; u < U; ++u) f(t[u], V, (int)((p + u * W) * V));
    }
    for (; p * V < nb; p += W) {
        const int off = (int)(p * V);
        const int nv = nb - off < V ? nb - off : V;
        float t[V];
        load(off, nv, t);
        f(t, nv, off);
    }
    if constexpr (!AL && V > 1) {
        if (worker < hd) {
            float t[V];
            load(-1 - worker, 1, t);
            f(t, 1, -1 - worker);
        }
    }
}

template <int OP, typename T, int V, bool AL, bool CL>
__global__ void __launch_bounds__(kLoopMaxThreads) loop_kernel(const KArgs a) {
    kernel_prologue<OP, T, CL>(a);
    // Packs in flight per thread.  RMSNorm, softmax and log-softmax (one
    // input, light per-pack work, a second pass that re-reads the row): 8,
    // or 4 for 8-value packs (128 bytes), measured faster on wide rows.  The
    // others keep 4, or 2 for 8-value packs: the one-pass row sum and
    // cross-entropy measured slower with 8, and LayerNorm and the residual
    // operators would leave the register budget.
    constexpr bool kDeep =
        OP == OP_RMSNORM || OP == OP_SOFTMAX || OP == OP_LOG_SOFTMAX;
    constexpr int U = kDeep ? (V >= 8 ? 4 : 8) : (V >= 8 ? 2 : 4);
    __shared__ RedScratch red;
    int parity = 0;
    const T *X = static_cast<const T *>(a.x);
    const T *Wt = static_cast<const T *>(a.w);
    const T *Bt = static_cast<const T *>(a.b);
    T *Y = static_cast<T *>(a.y);
    const int W = a.W;             // threads of this CTA per row
    // CTAs per row (thread-block cluster); the CL=false kernels fold every
    // cluster step away.
    const int csize = CL ? a.csize : 1;
    const int rank = csize > 1 ? (int)cluster_ctarank() : 0;
    const int WT = W * csize;      // workers per row
    const int worker = rank * W + (int)(threadIdx.x & (W - 1));
    const int slot = threadIdx.x >> a.log2W;
    const int64_t g0 = csize > 1 ? (int64_t)cluster_id_x() : blockIdx.x;
    const int64_t gstride =
        csize > 1 ? (int64_t)num_clusters_x() : (int64_t)gridDim.x;
    int cpar = 0;
    const int cols = a.cols;
    const int64_t ngroups = (a.rows + a.B - 1) / a.B;
    const bool yvec = AL || a.y_vec;

    for (int64_t g = g0; g < ngroups; g += gstride) {
        prefetch_next_group<OP, T>(a, g, ngroups, gstride, rank);
        const int64_t row = g * a.B + slot;
        const bool active = row < a.rows;
        const RowGeom<T, V, AL> geo(X, active ? row : 0, cols);
        const int64_t base = geo.base;
        const int hd = geo.hd, nb = geo.nb;
        const T *xb = X + base + hd;
        const T *xrow = X + base;
        // Loads the (residual-added) input values of one pack or the head.
        auto load_x = [&](int off, int nv, float *t) {
            if (off < 0) {
                t[0] = to_f(xrow[-1 - off]);
                if constexpr (has_residual<OP>())
                    t[0] = __fadd_rn(
                        t[0], to_f(static_cast<const T *>(a.res)[base - 1 - off]));
                return;
            }
            if (nv == V) {
                ld_vec<T, V>(xb + off, t);
            } else {
#pragma unroll
                for (int e = 0; e < V; ++e)
                    t[e] = e < nv ? to_f(xb[off + e]) : 0.f;
            }
            if constexpr (has_residual<OP>()) {
                const T *rb = static_cast<const T *>(a.res) + base + hd;
                float r[V];
                if (nv == V && (AL || a.r_vec)) {
                    ld_vec<T, V>(rb + off, r);
                } else {
#pragma unroll
                    for (int e = 0; e < V; ++e)
                        r[e] = e < nv ? to_f(rb[off + e]) : 0.f;
                }
#pragma unroll
                for (int e = 0; e < V; ++e) t[e] = __fadd_rn(t[e], r[e]);
            }
        };
        // Column of a head element (off < 0).
        auto column = [&](int off) { return -1 - off; };

        if constexpr (OP == OP_RMSNORM || OP == OP_RESIDUAL_RMSNORM) {
            float ss = 0.f;
            stream_row<V, AL, U>(worker, WT, hd, nb, active, load_x,
                                 [&](const float *t, int nv, int) {
#pragma unroll
                                     for (int e = 0; e < V; ++e)
                                         if (e < nv) ss = fmaf(t[e], t[e], ss);
                                 });
            ss = team_allreduce<SumOp>(ss, W, csize, red, parity, cpar);
            const float r = rsqrtf(ss / (float)cols + a.eps);
            T *yb = Y + base + hd;
            T *H = static_cast<T *>(a.h);
            T *hb = H ? H + base + hd : nullptr;
            const bool hvec = AL || a.h_vec;
            stream_row<V, AL, U>(
                worker, WT, hd, nb, active, load_x,
                [&](const float *t, int nv, int off) {
                    if (off < 0) {
                        const int c = column(off);
                        Y[base + c] = from_f<T>(t[0] * r * param_at(Wt, c, 1.f));
                        if (OP == OP_RESIDUAL_RMSNORM && H)
                            H[base + c] = from_f<T>(t[0]);
                        return;
                    }
                    float wv[V], o[V];
                    param_pack<T, V>(Wt, hd + off, nv, AL, 1.f, wv);
#pragma unroll
                    for (int e = 0; e < V; ++e) o[e] = t[e] * r * wv[e];
                    store_pack<T, V, AL>(yb, off, nb, true, yvec, o);
                    if (OP == OP_RESIDUAL_RMSNORM && hb)
                        store_pack<T, V, AL>(hb, off, nb, true, hvec, t);
                });
        } else if constexpr (OP == OP_LAYERNORM ||
                             OP == OP_RESIDUAL_LAYERNORM) {
            // Shifted moments about the row's first value (as on the
            // register path): one pass and one reduction for the
            // statistics, then the output pass.
            float x0 = 0.f;
            load_x(-1, 1, &x0);  // column 0 of the row
            float s1 = 0.f, s2 = 0.f;
            stream_row<V, AL, U>(worker, WT, hd, nb, active, load_x,
                                 [&](const float *t, int nv, int) {
#pragma unroll
                                     for (int e = 0; e < V; ++e)
                                         if (e < nv) {
                                             const float d = t[e] - x0;
                                             s1 += d;
                                             s2 = fmaf(d, d, s2);
                                         }
                                 });
            team_allreduce_sum2(s1, s2, W, csize, red, parity, cpar);
            const float md = s1 / (float)cols;
            const float mean = x0 + md;
            const float rstd = rsqrtf(
                fmaxf(fmaf(-md, md, s2 / (float)cols), 0.f) + a.eps);
            T *yb = Y + base + hd;
            T *H = static_cast<T *>(a.h);
            T *hb = H ? H + base + hd : nullptr;
            const bool hvec = AL || a.h_vec;
            stream_row<V, AL, U>(
                worker, WT, hd, nb, active, load_x,
                [&](const float *t, int nv, int off) {
                    if (off < 0) {
                        const int c = column(off);
                        Y[base + c] = from_f<T>(fmaf((t[0] - mean) * rstd,
                                                     param_at(Wt, c, 1.f),
                                                     param_at(Bt, c, 0.f)));
                        if (OP == OP_RESIDUAL_LAYERNORM && H)
                            H[base + c] = from_f<T>(t[0]);
                        return;
                    }
                    float gv[V], bv[V], o[V];
                    param_pack<T, V>(Wt, hd + off, nv, AL, 1.f, gv);
                    param_pack<T, V>(Bt, hd + off, nv, AL, 0.f, bv);
#pragma unroll
                    for (int e = 0; e < V; ++e)
                        o[e] = fmaf((t[e] - mean) * rstd, gv[e], bv[e]);
                    store_pack<T, V, AL>(yb, off, nb, true, yvec, o);
                    if (OP == OP_RESIDUAL_LAYERNORM && hb)
                        store_pack<T, V, AL>(hb, off, nb, true, hvec, t);
                });
        } else if constexpr (OP == OP_SOFTMAX || OP == OP_CROSS_ENTROPY ||
                             OP == OP_LOG_SOFTMAX) {
            // Running (max, sum of exp(x - max)) of the thread's values:
            // the sum is rescaled only when a pack raises the max (or turns
            // it NaN), so a pack costs one exponential per value; while
            // every value so far is -inf there is nothing to add (and
            // exp(-inf - -inf) would be NaN).
            float m = -INFINITY, s = 0.f;
            stream_row<V, AL, U>(worker, WT, hd, nb, active, load_x,
                                 [&](const float *t, int nv, int) {
                                     float pm = -INFINITY;
#pragma unroll
                                     for (int e = 0; e < V; ++e)
                                         if (e < nv) pm = nanmax(pm, t[e]);
                                     const float mm = nanmax(m, pm);
                                     if (mm != m) {
                                         s *= exp_shifted(m - mm);
                                         m = mm;
                                     }
                                     if (m != -INFINITY) {
                                         float ps = 0.f;
#pragma unroll
                                         for (int e = 0; e < V; ++e)
                                             if (e < nv)
                                                 ps += exp_shifted(t[e] - m);
                                         s += ps;
                                     }
                                 });
            team_allreduce_lse(m, s, W, csize, red, parity, cpar);
            if constexpr (OP == OP_SOFTMAX) {
                const float inv = 1.f / s;
                T *yb = Y + base + hd;
                stream_row<V, AL, U>(
                    worker, WT, hd, nb, active, load_x,
                    [&](const float *t, int nv, int off) {
                        if (off < 0) {
                            Y[base + column(off)] =
                                from_f<T>(exp_shifted(t[0] - m) * inv);
                            return;
                        }
                        float o[V];
#pragma unroll
                        for (int e = 0; e < V; ++e) o[e] = exp_shifted(t[e] - m) * inv;
                        store_pack<T, V, AL>(yb, off, nb, true, yvec, o);
                    });
            } else if constexpr (OP == OP_LOG_SOFTMAX) {
                const float ls = logf(s);
                T *yb = Y + base + hd;
                stream_row<V, AL, U>(
                    worker, WT, hd, nb, active, load_x,
                    [&](const float *t, int nv, int off) {
                        if (off < 0) {
                            Y[base + column(off)] = from_f<T>((t[0] - m) - ls);
                            return;
                        }
                        float o[V];
#pragma unroll
                        for (int e = 0; e < V; ++e) o[e] = (t[e] - m) - ls;
                        store_pack<T, V, AL>(yb, off, nb, true, yvec, o);
                    });
            } else {
                if (active && worker == 0) {
                    const int32_t lab = __ldg(a.labels + row);
                    const LabelInfo li = label_info(a, lab, cols);
                    const float xl = li.valid ? to_f(X[base + lab]) : NAN;
                    a.out[row] = li.ignored ? 0.f : (m + logf(s)) - xl;
                }
            }
        } else if constexpr (OP == OP_ROW_SUM) {
            float s = 0.f, c = 0.f;
            stream_row<V, AL, U>(worker, WT, hd, nb, active, load_x,
                                 [&](const float *t, int nv, int) {
#pragma unroll
                                     for (int e = 0; e < V; ++e)
                                         if (e < nv) {
                                             float u, err;
                                             two_sum(s, t[e], u, err);
                                             s = u;
                                             c += err;
                                         }
                                 });
            team_allreduce_compensated(s, c, W, csize, red, parity, cpar);
            if (active && worker == 0) a.out[row] = s + c;
        }
    }
    // Peers may still read this CTA's cluster slots.
    if (csize > 1) cluster_sync();
}

}  // namespace mt

#include "mt_stage.cuh"

namespace mt {

// =========================================================================
// Launch helpers
// =========================================================================
using KernelFn = void (*)(KArgs);

template <int OP, typename T, int V, int K>
__host__ KernelFn full_kernel() {
    if constexpr (reg_full_capped(OP, V * K, V * (int)sizeof(T),
                                  (int)sizeof(T)))
        return reg_full_capped_kernel<OP, T, V, K>;
    else
        return reg_full_kernel<OP, T, V, K>;
}

template <int OP, typename T, int V, bool AL, bool CL, bool FU = false>
__host__ KernelFn reg_kernel_for_chunks(int K) {
    if constexpr (FU) {
        switch (K) {
            case 1: return full_kernel<OP, T, V, 1>();
            case 2: return full_kernel<OP, T, V, 2>();
            case 4: return full_kernel<OP, T, V, 4>();
            case 8: return full_kernel<OP, T, V, 8>();
            case 16: return full_kernel<OP, T, V, 16>();
            default: return nullptr;
        }
    } else {
        switch (K) {
            case 1: return reg_kernel<OP, T, V, 1, AL, CL>;
            case 2: return reg_kernel<OP, T, V, 2, AL, CL>;
            case 4: return reg_kernel<OP, T, V, 4, AL, CL>;
            case 8: return reg_kernel<OP, T, V, 8, AL, CL>;
            case 16: return reg_kernel<OP, T, V, 16, AL, CL>;
            default: return nullptr;
        }
    }
}

// A pack of one FP32 value needs no alignment head, so it has only the
// aligned kernels.  Cluster (split-row) kernels exist for 16-byte packs.
// Whole-tile register kernels (KM_FULL) exist for one CTA per row group.
template <int OP, typename T, int V, bool CL>
__host__ KernelFn kernel_for_cl(const mt_plan_t &p, int mode) {
    constexpr bool kOnlyAligned = (V == 1 && sizeof(T) == 4);
    const bool aligned = kOnlyAligned || mode != KM_UNALIGNED;
    if (p.path == MT_PATH_STAGE) {
        // Staged runs: 16-byte units, aligned rows.
        if constexpr (stage_supported<OP>() && V * sizeof(T) == 16) {
            if (aligned) return stage_kernel<OP, T, CL>;
        }
        return nullptr;
    }
    if (p.path == MT_PATH_LOOP) {
        if (aligned) return loop_kernel<OP, T, V, true, CL>;
        return loop_kernel<OP, T, V, kOnlyAligned, CL>;
    }
    if constexpr (!CL) {
        if (mode == KM_FULL)
            return reg_kernel_for_chunks<OP, T, V, true, false, true>(
                p.chunks);
    }
    if (aligned) return reg_kernel_for_chunks<OP, T, V, true, CL>(p.chunks);
    return reg_kernel_for_chunks<OP, T, V, kOnlyAligned, CL>(p.chunks);
}

template <int OP, typename T, int V>
__host__ KernelFn kernel_for(const mt_plan_t &p, int mode) {
    if constexpr (V * sizeof(T) == 16) {
        if (p.cluster > 1) return kernel_for_cl<OP, T, V, true>(p, mode);
    }
    if (p.cluster > 1) return nullptr;
    return kernel_for_cl<OP, T, V, false>(p, mode);
}

// Instantiated values per thread per chunk: FP32 V = 1, 2, 4 (4-, 8- and
// 16-byte packs); FP16/BF16 V = 2, 4, 8 (4-, 8- and 16-byte packs).
template <int OP, typename T>
__host__ KernelFn select_kernel(const mt_plan_t &p, int mode) {
    if constexpr (sizeof(T) == 4) {
        switch (p.values_per_thread) {
            case 1: return kernel_for<OP, T, 1>(p, mode);
            case 2: return kernel_for<OP, T, 2>(p, mode);
            case 4: return kernel_for<OP, T, 4>(p, mode);
        }
    } else {
        switch (p.values_per_thread) {
            case 2: return kernel_for<OP, T, 2>(p, mode);
            case 4: return kernel_for<OP, T, 4>(p, mode);
            case 8: return kernel_for<OP, T, 8>(p, mode);
        }
    }
    return nullptr;
}

template <int OP, typename T>
__host__ cudaError_t launch_op(const mt_plan_t &p, const KArgs &a,
                               int mode, cudaStream_t stream) {
    KernelFn k = select_kernel<OP, T>(p, mode);
    if (k == nullptr) return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (a.pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (a.csize > 8) {
        // 16 CTAs per cluster is beyond the portable size of 8.
        if (cudaError_t e =
                allow_nonportable_cluster(reinterpret_cast<const void *>(k)))
            return e;
    }
    size_t smem = 0;
    if (p.path == MT_PATH_STAGE) {
        smem = (size_t)stage_run_bytes(a.cols, (int)sizeof(T), a.csize);
        if (cudaError_t e = allow_stage_smem(reinterpret_cast<const void *>(k)))
            return e;
    }
    if (a.csize > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = (unsigned)a.csize;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid);
    cfg.blockDim = dim3((unsigned)(p.threads_per_row * p.rows_per_block));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = n ? attr : nullptr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, k, a);
}

template <int OP, typename T>
__host__ cudaError_t occupancy_op(const mt_plan_t &p, int mode, int64_t cols,
                                  int *blocks_per_sm) {
    KernelFn k = select_kernel<OP, T>(p, mode);
    if (k == nullptr) return cudaErrorInvalidValue;
    size_t smem = 0;
    if (p.path == MT_PATH_STAGE) {
        smem = (size_t)stage_run_bytes(cols, (int)sizeof(T),
                                       p.cluster > 1 ? p.cluster : 1);
        if (cudaError_t e = allow_stage_smem(reinterpret_cast<const void *>(k)))
            return e;
    }
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        blocks_per_sm, k, p.threads_per_row * p.rows_per_block, smem);
}

}  // namespace mt

// One translation unit per (operator, storage type) defines its launcher
// pair through this macro.
#define MT_DEFINE_LAUNCHER(name, OPV, TYPE)                                  \
    namespace mt {                                                           \
    cudaError_t name(const mt_plan_t &plan, const KArgs &a, int mode,        \
                     cudaStream_t stream) {                                  \
        return launch_op<OPV, TYPE>(plan, a, mode, stream);                  \
    }                                                                        \
    cudaError_t name##_occupancy(const mt_plan_t &plan, int mode,            \
                                 int64_t cols, int *blocks_per_sm) {         \
        return occupancy_op<OPV, TYPE>(plan, mode, cols, blocks_per_sm);     \
    }                                                                        \
    cudaError_t name##_timeouts(unsigned long long *n) {                     \
        return cudaMemcpyFromSymbol(n, g_stage_timeouts, sizeof(*n));        \
    }                                                                        \
    }
