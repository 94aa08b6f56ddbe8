// rows.cuh -- register-cached row kernels: each row (or, in the cluster
// tier, each piece of a row) is read from HBM exactly once into registers,
// reduced, rescaled in registers and written exactly once.
//
// Geometry (template parameter G = threads per row or per row piece):
//   G <= 32  : a group of G lanes per row, 128-thread CTAs holding 128/G rows
//              ("several rows per warp" for short rows, "one warp per row");
//   G >= 64  : one CTA of G threads per row, warp butterflies + one
//              shared-memory stage ("one block per row");
//   CLUSTER  : a thread-block cluster of cs CTAs per row, CTA partials
//              merged through distributed shared memory, so a row longer
//              than one CTA's registers is still read once ("several blocks
//              per row", split-row).
// Row-length policy of "Softmax 与归一化" (anrans.github.io), table
// "按行长度选择并行方式"; register row cache of "两个融合算子：RMSNorm 与
// online softmax" (daleiyang.github.io), §4·三 "N3：把 x 留在寄存器".
//
// Each thread owns EPT elements of its row as units of U elements (U = 16
// bytes of input for the vector path, U = 1 for the element-wise path); unit
// j of thread t is unit (u0 + j * G + t), so consecutive lanes touch
// consecutive 16-byte vectors (coalesced).
#pragma once

#include "reduce.cuh"

namespace osr {

struct RowArgs {
    const void *x;      // input rows
    void *res;          // fused: residual, read and overwritten
    const void *gamma;  // norms: [N] scale
    const void *beta;   // LayerNorm: [N] shift
    void *y;            // output rows
    float *row_max;     // softmax statistics, may be null
    float *row_sum;     // (the log-sum-exp kernel writes log-sum-exp here)
    int64_t *row_arg;   // log-sum-exp kernel: index of the row maximum, may be null
    void *ws;           // split tier: per-piece partial states
    int64_t M;          // rows
    int64_t N;          // row length in elements
    int64_t row0;       // first row handled by this launch (split batches)
    int64_t chunk;      // cluster / split: units per CTA piece
    int cs;             // cluster: CTAs per row; split: pieces per row
    float eps;
    int flags;          // kFlag* test hooks (0 in normal use)
};

// Test hook: the staged tier's copy barrier gets no arrival, so its bounded
// wait runs out and the kernel reports a fault instead of computing.
constexpr int kFlagNoArrive = 1;
// Softmax kernels: write log-softmax, (x - m) - log d, instead of exp(x - m) / d.
constexpr int kFlagLog = 2;

template <int G>
struct RowsGeom {
    static constexpr int kThreads = G <= 32 ? 128 : G;
    static constexpr int kRowsPerCta = kThreads / G;
    static constexpr int kWarps = kThreads / 32;
};

struct Slice {
    int64_t row;
    int64_t u0, u1;  // unit range of this CTA's piece of the row
    int t;           // thread index within the row group
    bool ok;         // the row exists
};

template <int G, bool CLUSTER>
__device__ __forceinline__ Slice make_slice(const RowArgs &a, int64_t nunits) {
    Slice s;
    if constexpr (G <= 32) {
        s.row = (int64_t)blockIdx.x * RowsGeom<G>::kRowsPerCta + threadIdx.x / G;
        s.t = threadIdx.x & (G - 1);
        s.u0 = 0;
        s.u1 = nunits;
    } else if constexpr (!CLUSTER) {
        s.row = blockIdx.x;
        s.t = threadIdx.x;
        s.u0 = 0;
        s.u1 = nunits;
    } else {
        // 1-D grid, cluster dims (cs, 1, 1): CTAs [r*cs, (r+1)*cs) form the
        // cluster of row r and %cluster_ctarank == blockIdx.x % cs
        s.row = blockIdx.x / a.cs;
        s.t = threadIdx.x;
        s.u0 = (int64_t)cluster_ctarank() * a.chunk;
        s.u1 = s.u0 + a.chunk < nunits ? s.u0 + a.chunk : nunits;
    }
    s.ok = s.row < a.M;
    return s;
}

// ============================================================ softmax
// Per thread: chunk summary of its cached elements (max, then sum of
// exp(x - max), overwriting the cache with those exps) -- the chunk-summary
// form of "两个融合算子" §4·四 "S4" with the chunk = the thread's elements.
// The row's (m, d) follows by max-then-sum over the row's threads (and CTAs);
// each thread then rescales its cached exps by e^(m_t - m) / d, so every
// element costs one exp.
template <Dt DI, Dt DO, int G, int EPT, int U, bool CLUSTER>
__global__ void __launch_bounds__(RowsGeom<G>::kThreads)
softmax_rows_kernel(const RowArgs a) {
    constexpr int NU = EPT / U;
    const int64_t nunits = a.N / U;
    const Slice s = make_slice<G, CLUSTER>(a, nunits);
    const char *xrow = reinterpret_cast<const char *>(a.x) + s.row * a.N * Elem<DI>::kBytes;
    pdl_wait();

    float v[NU][U];
#pragma unroll
    for (int j = 0; j < NU; ++j) {
        const int64_t ui = s.u0 + (int64_t)j * G + s.t;
        if (s.ok && ui < s.u1) {
            load_unit<DI, U>(xrow, ui * U, v[j]);
        } else {
#pragma unroll
            for (int k = 0; k < U; ++k) v[j][k] = -INFINITY;  // contributes e^-inf = 0
        }
    }

    float mt = -FLT_MAX;
#pragma unroll
    for (int j = 0; j < NU; ++j)
#pragma unroll
        for (int k = 0; k < U; ++k) mt = fmaxf(mt, v[j][k]);
    // log-softmax keeps the inputs; softmax replaces them by their exps
    const bool logm = (a.flags & kFlagLog) != 0;
    float dt = 0.f;
#pragma unroll
    for (int j = 0; j < NU; ++j)
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const float e = exp_shifted(v[j][k], mt);
            dt += e;
            v[j][k] = logm ? v[j][k] : e;
        }

    RowNorm rn;
    if constexpr (G <= 32) {
        rn = group_norm<G>(mt, dt);
    } else {
        __shared__ float red_m[32], red_d[32];
        rn = block_norm<RowsGeom<G>::kWarps>(mt, dt, red_m, red_d);
    }
    if constexpr (CLUSTER) {
        __shared__ float2 slot;
        rn = cluster_norm(mt, rn, a.cs, &slot);
    }

    const float scale = rn.f / rn.d;
    const float logd = logf(rn.d);
    if (a.row_max != nullptr && s.ok && s.t == 0 && s.u0 == 0) {
        a.row_max[s.row] = rn.m;
        if (a.row_sum != nullptr) a.row_sum[s.row] = rn.d;
    }

    char *yrow = reinterpret_cast<char *>(a.y) + s.row * a.N * Elem<DO>::kBytes;
#pragma unroll
    for (int j = 0; j < NU; ++j) {
        const int64_t ui = s.u0 + (int64_t)j * G + s.t;
        if (s.ok && ui < s.u1) {
            float o[U];
#pragma unroll
            for (int k = 0; k < U; ++k) o[k] = logm ? (v[j][k] - rn.m) - logd : v[j][k] * scale;
            store_unit<DO, U>(yrow, ui * U, o);
        }
    }
    pdl_trigger();
    if constexpr (CLUSTER) cluster_wait_acquire();
}

// ============================================================ RMSNorm
// y = x * rsqrt(mean(x^2) + eps) * gamma; with FUSED, x + residual is first
// rounded to the storage type, written back to the residual, and the
// rounded sum is what gets normalised ("GPU Kernel 工程（04）" 八.3 "fused
// residual + RMSNorm"; the stored value is normalised so that the output
// equals RMSNorm of the new residual).
// bfloat16 rows on the 16-byte path stay packed in registers (4 registers
// per 8 elements) and are widened when used, which halves the cache's
// register footprint and raises occupancy.
template <Dt D, int G, int EPT, int U, bool CLUSTER, bool FUSED>
__global__ void __launch_bounds__(RowsGeom<G>::kThreads)
rmsnorm_rows_kernel(const RowArgs a) {
    constexpr bool kPacked = D == Dt::BF16 && U == 8;
    constexpr int NU = EPT / U;
    constexpr int NP = kPacked ? NU : 1;  // packed vectors held
    constexpr int NF = kPacked ? 1 : NU;  // fp32 units held
    const int64_t nunits = a.N / U;
    const Slice s = make_slice<G, CLUSTER>(a, nunits);
    const int64_t row_off = s.row * a.N * Elem<D>::kBytes;
    const char *xrow = reinterpret_cast<const char *>(a.x) + row_off;
    pdl_wait();

    uint4 pk[NP], gp[NP];
    float v[NF][U], g[NF][U];
#pragma unroll
    for (int j = 0; j < NU; ++j) {
        const int64_t ui = s.u0 + (int64_t)j * G + s.t;
        const bool in = s.ok && ui < s.u1;
        if constexpr (kPacked) {
            pk[j] = make_uint4(0, 0, 0, 0);
            if (in) {
                pk[j] = ld16<Hint::Stream>(xrow + ui * 16);
                if constexpr (FUSED) {
                    char *rrow = reinterpret_cast<char *>(a.res) + row_off;
                    const uint4 rq = ld16<Hint::Stream>(rrow + ui * 16);
                    float xf[8], rf[8];
                    unpack8(pk[j], xf);
                    unpack8(rq, rf);
#pragma unroll
                    for (int k = 0; k < 8; ++k) xf[k] += rf[k];
                    pk[j] = pack8(xf);
                    __stcs(reinterpret_cast<uint4 *>(rrow + ui * 16), pk[j]);
                }
            }
        } else {
            if (in) {
                load_unit<D, U>(xrow, ui * U, v[j]);
                if constexpr (FUSED) {
                    char *rrow = reinterpret_cast<char *>(a.res) + row_off;
                    float r[U];
                    load_unit<D, U>(rrow, ui * U, r);
#pragma unroll
                    for (int k = 0; k < U; ++k) v[j][k] = round_to<D>(v[j][k] + r[k]);
                    store_unit<D, U>(rrow, ui * U, v[j]);
                }
            } else {
#pragma unroll
                for (int k = 0; k < U; ++k) v[j][k] = 0.f;
            }
        }
    }

    // gamma is shared by every row: read-only path, fetched before the
    // reduction so its latency overlaps it
#pragma unroll
    for (int j = 0; j < NU; ++j) {
        const int64_t ui = s.u0 + (int64_t)j * G + s.t;
        const bool in = s.ok && ui < s.u1;
        if constexpr (kPacked) {
            gp[j] = in ? ld16<Hint::ReadOnly>(reinterpret_cast<const char *>(a.gamma) + ui * 16)
                       : make_uint4(0, 0, 0, 0);
        } else {
            if (in) {
                load_unit<D, U, Hint::ReadOnly>(a.gamma, ui * U, g[j]);
            } else {
#pragma unroll
                for (int k = 0; k < U; ++k) g[j][k] = 0.f;
            }
        }
    }

    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < NU; ++j) {
        if constexpr (kPacked) {
            float f[8];
            unpack8(pk[j], f);
#pragma unroll
            for (int k = 0; k < 8; ++k) ss = fmaf(f[k], f[k], ss);
        } else {
#pragma unroll
            for (int k = 0; k < U; ++k) ss = fmaf(v[j][k], v[j][k], ss);
        }
    }

    if constexpr (G <= 32) {
        ss = group_sum<G>(ss);
    } else {
        __shared__ float red[32];
        ss = block_sum<RowsGeom<G>::kWarps>(ss, red);
    }
    if constexpr (CLUSTER) {
        __shared__ float2 slot;
        ss = cluster_sum(ss, a.cs, &slot);
    }
    const float r = rsqrtf(ss / (float)a.N + a.eps);

    char *yrow = reinterpret_cast<char *>(a.y) + row_off;
#pragma unroll
    for (int j = 0; j < NU; ++j) {
        const int64_t ui = s.u0 + (int64_t)j * G + s.t;
        if (s.ok && ui < s.u1) {
            if constexpr (kPacked) {
                float f[8], gf[8];
                unpack8(pk[j], f);
                unpack8(gp[j], gf);
#pragma unroll
                for (int k = 0; k < 8; ++k) f[k] = f[k] * r * gf[k];
                __stcs(reinterpret_cast<uint4 *>(yrow + ui * 16), pack8(f));
            } else {
                float o[U];
#pragma unroll
                for (int k = 0; k < U; ++k) o[k] = v[j][k] * r * g[j][k];
                store_unit<D, U>(yrow, ui * U, o);
            }
        }
    }
    pdl_trigger();
    if constexpr (CLUSTER) cluster_wait_acquire();
}

// ============================================================ LayerNorm
// y = (x - mu) / sqrt(var + eps) * gamma + beta with the two-pass statistics
// of "Softmax 与归一化" (anrans.github.io), "LayerNorm 与 RMSNorm", and its
// exercise 1 (two passes over the row cached in registers).  The values are
// first shifted by a pivot -- the row's first element, the same for every
// thread and CTA of the row -- so the binary32 sums work on numbers of the
// row's spread rather than its mean (the mean-101 stress case of that
// exercise would otherwise lose five digits to the rounding of the mean):
//   mu_s = (1/H) sum (x - p),  var = (1/H) sum ((x - p) - mu_s)^2,
//   y = ((x - p) - mu_s) * rsqrt(var + eps) * gamma + beta.
// Cluster tier: both sums are taken across the cluster's CTAs through
// distributed shared memory, two exchanges with one barrier each.  (Merging
// per-thread (n, mean, M2) states with Chan's formula in a single reduction
// measured 28 % slower: its divisions cost more than the second barrier.)
__device__ __forceinline__ float cluster_gather_sum(float v, int cs, float *slot) {
    if (threadIdx.x == 0) *slot = v;
    cluster_arrive_release();
    cluster_wait_acquire();
    const int q = threadIdx.x & 15;
    float t = 0.f;
    if (q < cs) {
        float r;
        asm volatile("ld.shared::cluster.f32 %0, [%1];"
                     : "=f"(r)
                     : "r"(mapa_shared(smem_u32(slot), q))
                     : "memory");
        t = r;
    }
    return group_sum<16>(t);
}

template <Dt D, int G, int EPT, int U, bool CLUSTER>
__global__ void __launch_bounds__(RowsGeom<G>::kThreads)
layernorm_rows_kernel(const RowArgs a) {
    constexpr bool kPacked = D == Dt::BF16 && U == 8;
    constexpr int NU = EPT / U;
    constexpr int NP = kPacked ? NU : 1;
    constexpr int NF = kPacked ? 1 : NU;
    const int64_t nunits = a.N / U;
    const Slice s = make_slice<G, CLUSTER>(a, nunits);
    const int64_t row_off = s.row * a.N * Elem<D>::kBytes;
    const char *xrow = reinterpret_cast<const char *>(a.x) + row_off;
    pdl_wait();

    float p = 0.f;  // pivot: x[row][0]
    if (s.ok) {
        float t[1];
        load_unit<D, 1, Hint::Keep>(xrow, 0, t);
        p = t[0];
    }
    // packed rows prefetch gamma and beta before the reductions, so their
    // latency overlaps them; fp32 rows read them when used
    uint4 pk[NP], gp[NP], bp[NP];
    float v[NF][U];
    uint32_t valid = 0;  // bit j: unit j of this thread exists
#pragma unroll
    for (int j = 0; j < NU; ++j) {
        const int64_t ui = s.u0 + (int64_t)j * G + s.t;
        const bool in = s.ok && ui < s.u1;
        valid |= in ? 1u << j : 0u;
        if constexpr (kPacked) {
            pk[j] = in ? ld16<Hint::Stream>(xrow + ui * 16) : make_uint4(0, 0, 0, 0);
            gp[j] = in ? ld16<Hint::ReadOnly>(reinterpret_cast<const char *>(a.gamma) + ui * 16)
                       : make_uint4(0, 0, 0, 0);
            bp[j] = in ? ld16<Hint::ReadOnly>(reinterpret_cast<const char *>(a.beta) + ui * 16)
                       : make_uint4(0, 0, 0, 0);
        } else if (in) {
            load_unit<D, U>(xrow, ui * U, v[j]);
        }
    }
    // the thread's values, shifted by the pivot, unit by unit
    auto shifted = [&](int j, float (&f)[U]) {
        if constexpr (kPacked) {
            unpack8(pk[j], f);
        } else {
#pragma unroll
            for (int k = 0; k < U; ++k) f[k] = v[j][k];
        }
#pragma unroll
        for (int k = 0; k < U; ++k) f[k] -= p;
    };

    float s1 = 0.f;
#pragma unroll
    for (int j = 0; j < NU; ++j)
        if (valid >> j & 1u) {
            float f[U];
            shifted(j, f);
#pragma unroll
            for (int k = 0; k < U; ++k) s1 += f[k];
        }
    __shared__ float red1[32], red2[32];
    __shared__ float slot1, slot2;
    if constexpr (G <= 32) {
        s1 = group_sum<G>(s1);
    } else {
        s1 = block_sum<RowsGeom<G>::kWarps>(s1, red1);
    }
    if constexpr (CLUSTER) s1 = cluster_gather_sum(s1, a.cs, &slot1);
    const float mu = s1 / (float)a.N;

    float s2 = 0.f;
#pragma unroll
    for (int j = 0; j < NU; ++j)
        if (valid >> j & 1u) {
            float f[U];
            shifted(j, f);
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const float c = f[k] - mu;
                s2 = fmaf(c, c, s2);
            }
        }
    if constexpr (G <= 32) {
        s2 = group_sum<G>(s2);
    } else {
        s2 = block_sum<RowsGeom<G>::kWarps>(s2, red2);
    }
    if constexpr (CLUSTER) {
        s2 = cluster_gather_sum(s2, a.cs, &slot2);
        cluster_arrive_relaxed();
    }
    const float r = rsqrtf(s2 / (float)a.N + a.eps);

    char *yrow = reinterpret_cast<char *>(a.y) + row_off;
#pragma unroll
    for (int j = 0; j < NU; ++j) {
        const int64_t ui = s.u0 + (int64_t)j * G + s.t;
        if (valid >> j & 1u) {
            float f[U], o[U], gg[U], bb[U];
            shifted(j, f);
            if constexpr (kPacked) {
                unpack8(gp[j], gg);
                unpack8(bp[j], bb);
            } else {
                load_unit<D, U, Hint::ReadOnly>(a.gamma, ui * U, gg);
                load_unit<D, U, Hint::ReadOnly>(a.beta, ui * U, bb);
            }
#pragma unroll
            for (int k = 0; k < U; ++k) o[k] = fmaf((f[k] - mu) * r, gg[k], bb[k]);
            store_unit<D, U>(yrow, ui * U, o);
        }
    }
    pdl_trigger();
    if constexpr (CLUSTER) cluster_wait_acquire();
}

}  // namespace osr
