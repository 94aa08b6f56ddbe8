// layernorm_kernels.cuh -- LayerNorm kernels: the register-cached row/cluster
// kernel and the two split-row passes.
#pragma once

#include <type_traits>

#include "row_common.cuh"

namespace osr {

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
// On 16-byte rows the arithmetic runs on binary32 pairs (f32x2), a quarter
// fewer instructions: the kernel is issue-bound, not memory-bound, with the
// scalar form.  Cluster tier: both sums are taken across the cluster's CTAs,
// each by one barrier-free exchange (cluster_sum).  (Merging per-thread (n,
// mean, M2) states with Chan's formula in a single reduction measured 28 %
// slower, with the exchanges behind cluster barriers: its divisions cost
// more than the second exchange.)
template <Dt D, int G, int EPT, int U, bool CLUSTER>
__global__ void __launch_bounds__(RowsGeom<G>::kThreads)
layernorm_rows_kernel(const RowArgs a) {
    // 16-byte units are kept as raw vectors and worked on in binary32 pairs
    // (f32x2: one instruction per two elements); element units are scalars.
    constexpr bool kVec = U > 1;
    constexpr int NU = EPT / U;
    constexpr int NQ = kVec ? NU : 1;   // raw vectors held
    constexpr int NS = kVec ? 1 : NU;   // scalars held
    constexpr int PAIRS = U / 2;        // binary32 pairs per vector
    const int64_t nunits = a.N / U;
    const Slice s = make_slice<G, CLUSTER>(a, nunits);
    const int64_t row_off = s.row * a.N * Elem<D>::kBytes;
    const char *xrow = reinterpret_cast<const char *>(a.x) + row_off;
    const char *gam = reinterpret_cast<const char *>(a.gamma);
    const char *bet = reinterpret_cast<const char *>(a.beta);
    if constexpr (CLUSTER) cluster_push_init(cluster_push_area<0>(), cluster_push_area<1>(), a.cs);
    pdl_wait();

    float p = 0.f;  // pivot: x[row][0]
    if (s.ok) {
        float t[1];
        load_unit<D, 1, Hint::Keep>(xrow, 0, t);
        p = t[0];
    }
    uint4 q[NQ];
    float v[NS];
    uint32_t valid = 0;  // bit j: unit j of this thread exists
#pragma unroll
    for (int j = 0; j < NU; ++j) {
        const int64_t ui = s.u0 + (int64_t)j * G + s.t;
        const bool in = s.ok && ui < s.u1;
        valid |= in ? 1u << j : 0u;
        if constexpr (kVec) {
            q[j] = in ? ld16<Hint::Stream>(xrow + ui * 16) : make_uint4(0, 0, 0, 0);
        } else if (in) {
            float t[1];
            load_unit<D, 1>(xrow, ui, t);
            v[j] = t[0];
        }
    }
    uint64_t p2 = f2_make(p, p);  // the pivot (bfloat16: moved near the mean for a second pass)
    // binary32 vectors: the pivot-shifted pairs are formed once and kept (the
    // same registers as the raw vectors; 4.30 -> 4.13 us on 256 x 5120).
    // bfloat16 vectors stay packed and are widened in each pass: keeping the
    // wide pairs costs 52 instead of 38 registers and measured 2 % slower.
    constexpr bool kKeep = kVec && D == Dt::F32;
    uint64_t d2[kKeep ? NU : 1][kKeep ? PAIRS : 1];
    if constexpr (kKeep) {
#pragma unroll
        for (int j = 0; j < NU; ++j)
#pragma unroll
            for (int k = 0; k < PAIRS; ++k) d2[j][k] = f2_sub(f2_of<D>(q[j], k), p2);
    }
    auto shifted2 = [&](int j, int k) {  // pair k of unit j, minus the pivot
        if constexpr (kKeep) return d2[j][k];
        else return f2_sub(f2_of<D>(q[j], k), p2);
    };

    // Statistics of the pivot-shifted values d = x - p.
    // binary32 rows: the two-pass form, mu = sum(d)/H, then
    // var = sum((d - mu)^2)/H.  A pivot hundreds of standard deviations from
    // the mean costs them digits in x - p.
    // bfloat16 rows: one pass for sum(d) and sum(d^2), reduced together,
    // var = sum(d^2)/H - mu^2 (x - p is exact there: a difference of two
    // 8-bit significands).  The subtraction loses log10(1 + mu^2/var)
    // digits, so when mu^2 > 0.9 mean(d^2) (the pivot far from the mean) a
    // second pass runs, the corrected two-pass algorithm (Chan, Golub &
    // LeVeque, "Algorithms for computing the sample variance", 1983) about
    // P = p + mu, a binary32 number next to the mean: with c = x - P,
    // mu = sum(c)/H and var = sum(c^2)/H - mu^2, and the output offset is
    // small as well.
    constexpr bool kOnePass = kVec && D == Dt::BF16;
    __shared__ float red1[32], red2[32];
    float s1 = 0.f, q2 = 0.f;
    if constexpr (kVec) {
        uint64_t acc = f2_make(0.f, 0.f), acc2 = f2_make(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < NU; ++j)
            if (valid >> j & 1u) {
#pragma unroll
                for (int k = 0; k < PAIRS; ++k) {
                    const uint64_t d = shifted2(j, k);
                    acc = f2_add(acc, d);
                    if constexpr (kOnePass) acc2 = f2_fma(d, d, acc2);
                }
            }
        s1 = f2_lo(acc) + f2_hi(acc);
        if constexpr (kOnePass) q2 = f2_lo(acc2) + f2_hi(acc2);
    } else {
#pragma unroll
        for (int j = 0; j < NU; ++j)
            if (valid >> j & 1u) s1 += v[j] - p;
    }
    // the row's sums of a and b: threads, warps (one shared-memory stage),
    // cluster CTAs (exchange number X)
    auto row_sums = [&](float &sa, float &sb, float *ra, float *rb, auto X) {
        if constexpr (G <= 32) {
            sa = group_sum<G>(sa);
            sb = group_sum<G>(sb);
        } else {
            constexpr int NW = RowsGeom<G>::kWarps;
            const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
            sa = group_sum<32>(sa);
            sb = group_sum<32>(sb);
            if (lane == 0) {
                ra[warp] = sa;
                rb[warp] = sb;
            }
            __syncthreads();
            sa = group_sum<NW>(ra[lane & (NW - 1)]);
            sb = group_sum<NW>(rb[lane & (NW - 1)]);
        }
        if constexpr (CLUSTER) {
            constexpr int ID = decltype(X)::value;
            ClusterPush *x = cluster_push_area<ID>();
            const bool got = cluster_push(x, make_uint4(__float_as_uint(sa), __float_as_uint(sb), 0u, 0u), a.cs, ID == 0);
            const int lane = threadIdx.x & 31;
            sa = group_sum<32>(lane < a.cs ? __uint_as_float(x->slot[lane].x) : 0.f);
            sb = group_sum<32>(lane < a.cs ? __uint_as_float(x->slot[lane].y) : 0.f);
            if (!got) sa = __int_as_float(0x7fffffff);
        }
    };
    if constexpr (kOnePass) {
        row_sums(s1, q2, red1, red2, std::integral_constant<int, 0>());
    } else {
        if constexpr (G <= 32) {
            s1 = group_sum<G>(s1);
        } else {
            s1 = block_sum<RowsGeom<G>::kWarps>(s1, red1);
        }
        if constexpr (CLUSTER) s1 = cluster_sum(s1, a.cs, cluster_push_area<0>(), true);
    }
    float mu = s1 / (float)a.N;  // mean of the shifted values
    float s2 = 0.f;
    bool second = true;
    if constexpr (kOnePass) {
        const float e2 = q2 / (float)a.N;  // mean of d^2 = var + mu^2
        second = mu * mu > 0.9f * e2;      // the same in every thread and CTA of the row
        s2 = fmaxf(e2 - mu * mu, 0.f) * (float)a.N;
    }
    if (second) {
        if constexpr (kOnePass) {
            p2 = f2_make(p + mu, p + mu);  // shifted2 now gives x - P
            mu = 0.f;
        }
        const uint64_t m1 = f2_make(mu, mu);
        float t1 = 0.f, t2 = 0.f;
        if constexpr (kVec) {
            uint64_t acc = f2_make(0.f, 0.f), acc2 = f2_make(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < NU; ++j)
                if (valid >> j & 1u) {
#pragma unroll
                    for (int k = 0; k < PAIRS; ++k) {
                        const uint64_t c = f2_sub(shifted2(j, k), m1);
                        if constexpr (kOnePass) acc = f2_add(acc, c);
                        acc2 = f2_fma(c, c, acc2);
                    }
                }
            t1 = f2_lo(acc) + f2_hi(acc);
            t2 = f2_lo(acc2) + f2_hi(acc2);
        } else {
#pragma unroll
            for (int j = 0; j < NU; ++j)
                if (valid >> j & 1u) {
                    const float c = (v[j] - p) - mu;
                    t2 = fmaf(c, c, t2);
                }
        }
        if constexpr (kOnePass) {
            // second stage arrays: a warp may still read the first ones
            __shared__ float red3[32], red4[32];
            row_sums(t1, t2, red3, red4, std::integral_constant<int, 1>());
            const float dm = t1 / (float)a.N;  // the mean of x - P
            mu += dm;
            s2 = fmaxf(t2 - t1 * dm, 0.f);
        } else {
            // binary32: the sum of squares about mu1 (the correction of mu1
            // is below the rounding of x - p there, and cost 7 % on
            // 256 x 5120)
            if constexpr (G <= 32) {
                t2 = group_sum<G>(t2);
            } else {
                t2 = block_sum<RowsGeom<G>::kWarps>(t2, red2);
            }
            if constexpr (CLUSTER) t2 = cluster_sum(t2, a.cs, cluster_push_area<1>(), false);
            s2 = t2;
        }
    }
    const uint64_t mu2 = f2_make(mu, mu);
    const float r = rsqrtf(s2 / (float)a.N + a.eps);
    const uint64_t r2 = f2_make(r, r);
    // bfloat16 rows: z = (x - p) r - mu r in one fused multiply-add.  x - p
    // is exact there and |mu| r stays near 1 or below (the second pass moves
    // the pivot next to the mean whenever mu is large), so the rounding of
    // mu r adds at most about 2^-24 to z: one instruction less per pair.
    const uint64_t nmur2 = f2_make(-(mu * r), -(mu * r));

    char *yrow = reinterpret_cast<char *>(a.y) + row_off;
#pragma unroll
    for (int j = 0; j < NU; ++j) {
        const int64_t ui = s.u0 + (int64_t)j * G + s.t;
        if (!(valid >> j & 1u)) continue;
        if constexpr (kVec) {
            // gamma and beta are read when used: prefetching them into
            // registers before the reductions measured 10 % slower (69
            // instead of 38 registers, fewer CTAs per SM)
            const uint4 g16 = ld16<Hint::ReadOnly>(gam + ui * 16);
            const uint4 b16 = ld16<Hint::ReadOnly>(bet + ui * 16);
            uint64_t o[PAIRS];
#pragma unroll
            for (int k = 0; k < PAIRS; ++k) {
                uint64_t z;
                if constexpr (kOnePass) z = f2_fma(shifted2(j, k), r2, nmur2);
                else z = f2_mul(f2_sub(shifted2(j, k), mu2), r2);
                o[k] = f2_fma(z, f2_of<D>(g16, k), f2_of<D>(b16, k));
            }
            uint4 w;
            if constexpr (D == Dt::BF16) {
                w = make_uint4(bf16x2_from_f2(o[0]), bf16x2_from_f2(o[1]), bf16x2_from_f2(o[2]),
                               bf16x2_from_f2(o[3]));
            } else {
                w = make_uint4(__float_as_uint(f2_lo(o[0])), __float_as_uint(f2_hi(o[0])),
                               __float_as_uint(f2_lo(o[1])), __float_as_uint(f2_hi(o[1])));
            }
            __stcs(reinterpret_cast<uint4 *>(yrow + ui * 16), w);
        } else {
            float gg[1], bb[1];
            load_unit<D, 1, Hint::ReadOnly>(a.gamma, ui, gg);
            load_unit<D, 1, Hint::ReadOnly>(a.beta, ui, bb);
            const float o[1] = {fmaf(((v[j] - p) - mu) * r, gg[0], bb[0])};
            store_unit<D, 1>(yrow, ui, o);
        }
    }
    pdl_trigger();
}

// ------------------------------------------------------------ LayerNorm, split
// Pass 1: each piece's (n, mean, M2) of the pivot-shifted values (the pivot,
// x[row][0], is stored with them, so pass 2 never reads x[row][0] after a
// piece has overwritten it in place): every tile
// is summarised by its own two passes in registers and folded into the
// thread's state with Chan's merge ("GPU Kernel 工程（04）" 八.2, Welford and
// Chan et al.), then the CTA's states are merged in a fixed tree.  Pass 2:
// every CTA of a row merges the row's S states in the same fixed tree (so all
// of them normalise with identical statistics) and streams its piece again.
struct Chan {
    float n, mean, m2;
};

__device__ __forceinline__ Chan chan_merge(Chan a, Chan b) {
    if (a.n == 0.f) return b;
    if (b.n == 0.f) return a;
    const float n = a.n + b.n, delta = b.mean - a.mean, fb = b.n / n;
    return {n, fmaf(delta, fb, a.mean), a.m2 + b.m2 + delta * delta * a.n * fb};
}

// Merge the CTA's per-thread states; the result is valid in thread 0.
template <int NW>
__device__ __forceinline__ Chan block_chan_to_thread0(Chan c, float4 *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        Chan o;
        o.n = __shfl_down_sync(0xffffffffu, c.n, off);
        o.mean = __shfl_down_sync(0xffffffffu, c.mean, off);
        o.m2 = __shfl_down_sync(0xffffffffu, c.m2, off);
        if (lane + off < 32) c = chan_merge(c, o);
    }
    if (lane == 0) red[warp] = make_float4(c.n, c.mean, c.m2, 0.f);
    __syncthreads();
    if (warp == 0) {
        c = Chan{0.f, 0.f, 0.f};
        if (lane < NW) {
            const float4 q = red[lane];
            c = Chan{q.x, q.y, q.z};
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            Chan o;
            o.n = __shfl_down_sync(0xffffffffu, c.n, off);
            o.mean = __shfl_down_sync(0xffffffffu, c.mean, off);
            o.m2 = __shfl_down_sync(0xffffffffu, c.m2, off);
            if (lane + off < 32) c = chan_merge(c, o);
        }
    }
    return c;
}

template <Dt D, int G, int EPT, int U>
__global__ void __launch_bounds__(G) layernorm_split_stats_kernel(const RowArgs a) {
    constexpr int NU = EPT / U;
    const int64_t nunits = a.N / U;
    const Piece q = make_piece(a, nunits);
    const char *xrow = reinterpret_cast<const char *>(a.x) + q.row * a.N * Elem<D>::kBytes;
    pdl_wait();
    float p;
    {
        float t[1];
        load_unit<D, 1, Hint::Keep>(xrow, 0, t);
        p = t[0];
    }
    Chan st{0.f, 0.f, 0.f};
    for (int64_t base = q.u0; base < q.u1; base += (int64_t)G * NU) {
        float v[NU][U];
        int cnt = 0;
        float s1 = 0.f;
#pragma unroll
        for (int j = 0; j < NU; ++j) {
            const int64_t ui = base + (int64_t)j * G + threadIdx.x;
            if (ui < q.u1) {
                load_unit<D, U, Hint::Keep>(xrow, ui * U, v[j]);
#pragma unroll
                for (int k = 0; k < U; ++k) {
                    v[j][k] -= p;
                    s1 += v[j][k];
                }
                cnt += U;
            }
        }
        if (cnt == 0) continue;
        const float tm = s1 / (float)cnt;
        float s2 = 0.f;
#pragma unroll
        for (int j = 0; j < NU; ++j) {
            const int64_t ui = base + (int64_t)j * G + threadIdx.x;
            if (ui < q.u1) {
#pragma unroll
                for (int k = 0; k < U; ++k) {
                    const float c = v[j][k] - tm;
                    s2 = fmaf(c, c, s2);
                }
            }
        }
        st = chan_merge(st, Chan{(float)cnt, tm, s2});
    }
    __shared__ float4 red[32];
    st = block_chan_to_thread0<G / 32>(st, red);
    if (threadIdx.x == 0)
        reinterpret_cast<float4 *>(a.ws)[q.row * a.cs + q.p] = make_float4(st.n, st.mean, st.m2, p);
    pdl_trigger();
}

template <Dt D, int G, int EPT, int U>
__global__ void __launch_bounds__(G) layernorm_split_apply_kernel(const RowArgs a) {
    constexpr int NU = EPT / U;
    const int64_t nunits = a.N / U;
    const Piece q = make_piece(a, nunits);
    const int64_t row_off = q.row * a.N * Elem<D>::kBytes;
    const char *xrow = reinterpret_cast<const char *>(a.x) + row_off;
    pdl_wait();
    Chan st{0.f, 0.f, 0.f};
    if (threadIdx.x < a.cs) {
        const float4 w = reinterpret_cast<const float4 *>(a.ws)[q.row * a.cs + threadIdx.x];
        st = Chan{w.x, w.y, w.z};
    }
    __shared__ float4 red[32];
    __shared__ float2 stats;
    st = block_chan_to_thread0<G / 32>(st, red);
    if (threadIdx.x == 0) stats = make_float2(st.mean, rsqrtf(st.m2 / (float)a.N + a.eps));
    const float p = reinterpret_cast<const float4 *>(a.ws)[q.row * a.cs].w;  // pass 1's pivot
    __syncthreads();
    const float mu = stats.x, r = stats.y;
    char *yrow = reinterpret_cast<char *>(a.y) + row_off;
    for (int64_t base = q.u0; base < q.u1; base += (int64_t)G * NU) {
        float v[NU][U], g[NU][U], b[NU][U];
#pragma unroll
        for (int j = 0; j < NU; ++j) {
            const int64_t ui = base + (int64_t)j * G + threadIdx.x;
            if (ui < q.u1) {
                load_unit<D, U>(xrow, ui * U, v[j]);
                load_unit<D, U, Hint::ReadOnly>(a.gamma, ui * U, g[j]);
                load_unit<D, U, Hint::ReadOnly>(a.beta, ui * U, b[j]);
            }
        }
#pragma unroll
        for (int j = 0; j < NU; ++j) {
            const int64_t ui = base + (int64_t)j * G + threadIdx.x;
            if (ui < q.u1) {
                float o[U];
#pragma unroll
                for (int k = 0; k < U; ++k) o[k] = fmaf(((v[j][k] - p) - mu) * r, g[j][k], b[j][k]);
                store_unit<D, U>(yrow, ui * U, o);
            }
        }
    }
    pdl_trigger();
}

}  // namespace osr
