// k_lse.cu -- per-row log-sum-exp and argmax without writing probabilities.
//
// A sampler that draws greedily needs only the index of the row maximum, and
// one that works in log space needs only log(sum_j e^(x_j)) = m + log d:
// "Softmax 与归一化" (anrans.github.io), exercise 2 "大词表采样" -- sampling
// does not need the softmax row written out.  This kernel therefore reads
// each row once and writes two numbers per row: HBM traffic is the input
// alone.
//
// Each thread streams its units in tiles and keeps a running (m, d): the
// online normaliser's update, taken once per tile (the running maximum
// raised by the tile's maximum, the sum rescaled, then the tile's exps
// added against the new maximum).  Across threads, CTAs and cluster CTAs:
// the row maximum, then the smallest index holding it, then the sum of
// d e^(m_t - m).
#include <cuda_runtime.h>

#include "launch.h"
#include "lse.h"

namespace osr {

constexpr int64_t kNoIndex = 0x7fffffffffffffffLL;
// elements per thread per tile: twice the row kernels' 16, so each thread
// keeps 64 (bf16) to 128 (fp32) bytes of loads in flight in a streaming loop
constexpr int kLseEpt = 32;
constexpr int kLseStagedHeader = 128;  // the copies' mbarrier, padded

// per half: the larger number (a NaN loses to a number)
__device__ __forceinline__ uint32_t lse_max_bf16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

template <int W>
__device__ __forceinline__ int64_t group_min_i64(int64_t v) {
#pragma unroll
    for (int off = W / 2; off > 0; off >>= 1) {
        const int64_t o = __shfl_xor_sync(0xffffffffu, v, off);
        v = o < v ? o : v;
    }
    return v;
}

struct MaxArgSum {
    float m;
    float d;
    int64_t i;
};

template <int W>
__device__ __forceinline__ MaxArgSum group_mas(MaxArgSum t) {
    MaxArgSum r;
    r.m = group_max<W>(t.m);
    r.i = group_min_i64<W>(t.m == r.m ? t.i : kNoIndex);
    r.d = group_sum<W>(t.d * md_factor(t.m, r.m));
    return r;
}

// A thread's tile of the streaming kernel: NU units kept raw, 16-byte
// vectors (U > 1) or single elements widened to binary32 (U = 1).
template <bool B>
struct LseFull {
    static constexpr bool value = B;
};
template <int U>
struct RawOf {
    using T = uint4;
};
template <>
struct RawOf<1> {
    using T = float;
};
template <int U>
using Raw = typename RawOf<U>::T;

template <Dt DI, int U>
__device__ __forceinline__ Raw<U> raw_neg_inf() {
    if constexpr (U == 1) {
        return -INFINITY;
    } else {
        const uint32_t n = DI == Dt::BF16 ? 0xff80ff80u : 0xff800000u;
        return make_uint4(n, n, n, n);
    }
}
// element k of a unit, exactly widened
template <Dt DI, int U>
__device__ __forceinline__ float raw_elem(const Raw<U> &q, int k) {
    if constexpr (U == 1) {
        return q;
    } else if constexpr (DI == Dt::BF16) {
        const uint32_t w = k < 2 ? q.x : k < 4 ? q.y : k < 6 ? q.z : q.w;
        return (k & 1) ? bf16_hi(w) : bf16_lo(w);
    } else {
        return __uint_as_float(k == 0 ? q.x : k == 1 ? q.y : k == 2 ? q.z : q.w);
    }
}
// elements 2p and 2p + 1 of the tile as an f32x2 pair
template <Dt DI, int U, int NU>
__device__ __forceinline__ uint64_t raw_pair(const Raw<U> (&q)[NU], int p) {
    if constexpr (U == 1)
        return f2_make(q[2 * p], q[2 * p + 1]);
    else
        return f2_of<DI>(q[p / (U / 2)], p % (U / 2));
}
// the tile's maximum, as a tree (bfloat16 on packed pairs); a NaN loses
// unless every element is NaN
template <Dt DI, int U, int NU>
__device__ __forceinline__ float raw_tile_max(const Raw<U> (&q)[NU]) {
    if constexpr (U > 1 && DI == Dt::BF16) {
        uint32_t w[NU];
#pragma unroll
        for (int j = 0; j < NU; ++j)
            w[j] = lse_max_bf16x2(lse_max_bf16x2(q[j].x, q[j].y), lse_max_bf16x2(q[j].z, q[j].w));
#pragma unroll
        for (int h = NU / 2; h >= 1; h /= 2)
#pragma unroll
            for (int j = 0; j < h; ++j) w[j] = lse_max_bf16x2(w[j], w[j + h]);
        return fmaxf(bf16_lo(w[0]), bf16_hi(w[0]));
    } else {
        float v[NU];
#pragma unroll
        for (int j = 0; j < NU; ++j) {
            if constexpr (U == 1)
                v[j] = q[j];
            else
                v[j] = fmaxf(fmaxf(__uint_as_float(q[j].x), __uint_as_float(q[j].y)),
                             fmaxf(__uint_as_float(q[j].z), __uint_as_float(q[j].w)));
        }
#pragma unroll
        for (int h = NU / 2; h >= 1; h /= 2)
#pragma unroll
            for (int j = 0; j < h; ++j) v[j] = fmaxf(v[j], v[j + h]);
        return v[0];
    }
}

// PEEL: rows that do not start on a 16-byte boundary, or whose length is not
// a multiple of the vector width.  Each row's body, from its first 16-byte
// boundary, streams in 16-byte vectors as above; its head (the h < U
// elements before that boundary) and its tail (the < U elements after the
// last whole vector) are folded in one element a lane, the head before the
// body and the tail after it (CTA 0 of a cluster).  Groups are at least U
// lanes wide.  The bf16 256-thread form is held to 32 registers (eight CTAs
// an SM, as the aligned one): 1024 rows of 50257 elements 22.7 -> 19.4 us,
// the time of 50256-element aligned rows.
template <Dt DI, int G, int U, bool CLUSTER, bool PEEL = false>
__global__ void __launch_bounds__(RowsGeom<G>::kThreads,
                                  CLUSTER ? lse_cluster_ctas_per_sm(DI)
                                          : (PEEL && DI == Dt::BF16 && G == 256) ? 8 : 0)
lse_argmax_kernel(const RowArgs a) {
    constexpr int NU = kLseEpt / U;
    static_assert(!PEEL || (U > 1 && G >= U), "a peeled row needs vectors and a lane per edge element");
    const int64_t nunits = a.N / U;
    Slice s = make_slice<G, CLUSTER>(a, nunits);
    const char *row0 = reinterpret_cast<const char *>(a.x) + s.row * a.N * Elem<DI>::kBytes;
    const char *xrow = row0;
    int64_t h = 0, nb = nunits;  // head elements, body vectors
    int tl = 0;                  // tail elements
    if constexpr (PEEL) {
        h = (int64_t)(((16u - (uint32_t)(reinterpret_cast<uintptr_t>(row0) & 15u)) & 15u) / Elem<DI>::kBytes);
        if (h > a.N) h = a.N;
        nb = (a.N - h) / U;
        tl = (int)(a.N - h - nb * U);
        if (s.u1 > nb) s.u1 = nb;
        xrow = row0 + h * Elem<DI>::kBytes;  // 16-byte aligned
    }
    // cluster: each CTA stores its (m, d, index) into slot [its rank] of
    // every CTA (st.async, counted on the receiver's xbar); no cluster
    // barrier after this start-up one
    __shared__ __align__(8) uint64_t xbar_word;
    __shared__ uint4 xslot[16];
    const uint32_t xbar = smem_u32(&xbar_word);
    if constexpr (CLUSTER) {
        if (threadIdx.x == 0) {
            mbar_init(xbar, 1);
            mbar_arrive_expect_tx(xbar, (uint32_t)a.cs * 16u);
            fence_mbar_init();
        }
        __syncthreads();
        cluster_arrive_relaxed();  // this CTA's xbar is initialised
    }
    pdl_wait();

    // The thread's running maximum m only grows: a tile that raises it
    // rescales the running sum by e^(m_old - m_new) and records its base.
    // The tile's exps are then taken against the running maximum (so no
    // second exp per tile), summed on f32x2 pairs, and the tile's sum added
    // whole to the running one.  The first index holding the maximum is
    // searched once, after the group's maximum is known, and only by the
    // threads that hold it: in the tile they recorded, which is still in
    // registers when it was the last one (a thread visits its elements in
    // increasing index order, so a later tile with the same maximum never
    // moves the first index).  An in-loop search would run on whichever
    // lanes raised their maximum in that tile, and the warp would pay for
    // it on almost every tile.
    float m_run = -INFINITY;
    uint64_t d2 = f2_make(0.f, 0.f);
    int64_t tbase = -1, last = -1;
    int64_t xidx = kNoIndex;  // PEEL: the edge element that set the running maximum
    Raw<U> q[NU];
    // PEEL: element e of the row folded in like a one-element tile
    auto fold_edge = [&](int64_t e) {
        float v[1];
        load_unit<DI, 1>(row0, e, v);
        if (v[0] > m_run) {
            const float f = exp_shifted(m_run, v[0]);
            d2 = f2_mul(d2, f2_make(f, f));
            m_run = v[0];
            tbase = -1;
            xidx = e;
        }
        d2 = f2_add(d2, f2_make(exp_shifted(v[0], md_shift(m_run)), 0.f));
    };
    const bool edges = PEEL && s.ok && s.u0 == 0;  // this CTA folds the row's edges
    if constexpr (PEEL) {
        if (edges && s.t < h) fold_edge(s.t);
    }
    auto load = [&](int64_t base, auto full) {
#pragma unroll
        for (int j = 0; j < NU; ++j) {
            const int64_t ui = base + (int64_t)j * G + s.t;
            if (decltype(full)::value || ui < s.u1) {
                if constexpr (U > 1) {
                    q[j] = ld16<Hint::Stream>(xrow + ui * 16);
                } else {
                    float v[1];
                    load_unit<DI, 1>(xrow, ui, v);
                    q[j] = v[0];
                }
            } else {
                q[j] = raw_neg_inf<DI, U>();
            }
        }
    };
    if (s.ok && s.u1 > s.u0) {
        const int64_t step = (int64_t)G * NU;
        last = s.u0 + (s.u1 - s.u0 - 1) / step * step;
        const uint64_t l2e = f2_make(1.4426950408889634f, 1.4426950408889634f);
        auto run = [&](int64_t base, auto full) {
            load(base, full);
            const float tm = raw_tile_max<DI, U, NU>(q);
            if (tm > m_run) {  // false for -inf and for an all-NaN tile
                // e^(m_run - tm) by the terms' own exp: 0 from m_run = -inf
                // (and for tm = +inf), no guard needed
                const float f = exp_shifted(m_run, tm);
                d2 = f2_mul(d2, f2_make(f, f));
                m_run = tm;
                tbase = base;
                if constexpr (PEEL) xidx = kNoIndex;
            }
            const float ms = md_shift(m_run);
            const uint64_t m2 = f2_make(ms, ms);
            uint64_t acc = f2_make(0.f, 0.f);
#pragma unroll
            for (int p = 0; p < NU * U / 2; ++p) {
                const uint64_t e = f2_mul(f2_sub(raw_pair<DI, U>(q, p), m2), l2e);
                acc = f2_add(acc, f2_make(ex2_approx(f2_lo(e)), ex2_approx(f2_hi(e))));
            }
            d2 = f2_add(d2, acc);
        };
        for (int64_t base = s.u0; base < last; base += step) run(base, LseFull<true>{});
        run(last, LseFull<false>{});
    }
    if constexpr (PEEL) {
        if (edges && s.t < tl) fold_edge(h + nb * U + s.t);
    }
    const float dsum = f2_lo(d2) + f2_hi(d2);
    // first index of m in the recorded tile (reloaded unless it was the last)
    // (PEEL: or the edge element that set it, which comes first)
    auto first_index = [&]() -> int64_t {
        if (PEEL && xidx != kNoIndex) return xidx;
        if (tbase != last) load(tbase, LseFull<true>{});
        int64_t ti = kNoIndex;
#pragma unroll
        for (int j = NU - 1; j >= 0; --j)
#pragma unroll
            for (int k = U - 1; k >= 0; --k)
                if (raw_elem<DI, U>(q[j], k) == m_run) ti = h + (tbase + (int64_t)j * G + s.t) * U + k;
        return ti;  // the last hit is the first
    };
    const bool holds = tbase >= 0 || (PEEL && xidx != kNoIndex);  // a recorded place of m_run

    MaxArgSum r;
    if constexpr (G <= 32) {
        r.m = group_max<G>(m_run);
        const int64_t ti = holds && m_run == r.m ? first_index() : kNoIndex;
        r.i = group_min_i64<G>(ti);
        r.d = group_sum<G>(dsum * md_factor(m_run, r.m));
    } else {
        constexpr int NW = RowsGeom<G>::kWarps;
        __shared__ float s_m[32], s_d[32];
        __shared__ long long s_i[32];
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        float m = group_max<32>(m_run);
        if (lane == 0) s_m[warp] = m;
        __syncthreads();
        m = group_max<NW>(s_m[lane & (NW - 1)]);
        const int64_t ti = holds && m_run == m ? first_index() : kNoIndex;
        const int64_t wi = group_min_i64<32>(ti);
        const float wd = group_sum<32>(dsum * md_factor(m_run, m));
        if (lane == 0) {
            s_d[warp] = wd;
            s_i[warp] = wi;
        }
        __syncthreads();
        r.m = m;
        r.d = group_sum<NW>(s_d[lane & (NW - 1)]);
        r.i = group_min_i64<NW>(s_i[lane & (NW - 1)]);
    }
    if constexpr (CLUSTER) {
        cluster_wait_acquire();  // every peer's xbar is initialised
        if (threadIdx.x < a.cs) {
            const uint4 v = make_uint4(__float_as_uint(r.m), __float_as_uint(r.d), (uint32_t)r.i,
                                       (uint32_t)((uint64_t)r.i >> 32));
            st_async_v4(mapa_shared(smem_u32(&xslot[cluster_ctarank()]), threadIdx.x),
                        mapa_shared(xbar, threadIdx.x), v);
        }
        // bounded (2 s): a state that never arrives gives NaN and -1
        const bool got = mbar_wait_bounded(xbar, 0, 2000000000ull);
        // lanes q and q + 16 take CTA q's state, the same order in every CTA
        const int q = threadIdx.x & 15;
        MaxArgSum p{-INFINITY, 0.f, kNoIndex};
        if (q < a.cs) {
            const uint4 v = xslot[q];
            p = MaxArgSum{__uint_as_float(v.x), __uint_as_float(v.y),
                          (int64_t)(((uint64_t)v.w << 32) | v.z)};
        }
        r = group_mas<16>(p);
        if (!got) {
            r.m = __int_as_float(0x7fffffff);
            r.i = kNoIndex;
        }
    }
    if (s.ok && s.t == 0 && s.u0 == 0) {
        if (a.row_sum != nullptr) a.row_sum[s.row] = r.m + logf(r.d);
        if (a.row_arg != nullptr) a.row_arg[s.row] = r.i == kNoIndex ? -1 : r.i;
    }
    pdl_trigger();
}

// Staged variant for rows spread over a cluster (16-byte rows): each CTA
// bulk-copies its whole piece into shared memory at once (every byte in
// flight together, where the streaming kernel above waits for one tile of
// loads after another), then takes its maximum with the first index holding
// it, and its sum of exp(x - max), from shared memory.  The CTAs' (m, d,
// index) go to every CTA of the cluster by st.async, as above.
template <Dt DI>
__global__ void __launch_bounds__(256) lse_staged_kernel(const RowArgs a) {
    constexpr int U = Elem<DI>::kVec;
    constexpr int T = 256;
    constexpr int NW = T / 32;
    extern __shared__ __align__(128) unsigned char smem[];
    const uint32_t bar = smem_u32(smem);
    const unsigned char *stage = smem + kLseStagedHeader;
    __shared__ __align__(8) uint64_t xbar_word;
    __shared__ uint4 xslot[16];
    __shared__ float s_m[NW], s_d[NW];
    __shared__ long long s_i[NW];
    const uint32_t xbar = smem_u32(&xbar_word);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    const int64_t nunits = a.N / U;
    const int64_t row = blockIdx.x / a.cs;
    const uint32_t rank = cluster_ctarank();
    const int64_t u0 = (int64_t)rank * a.chunk;
    const int64_t u1 = u0 + a.chunk < nunits ? u0 + a.chunk : nunits;
    const int n = u1 > u0 ? (int)(u1 - u0) : 0;
    const char *src = reinterpret_cast<const char *>(a.x) + (row * nunits + u0) * 16;

    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        mbar_init(xbar, 1);
        mbar_arrive_expect_tx(xbar, (uint32_t)a.cs * 16u);
        fence_mbar_init();
    }
    __syncthreads();
    cluster_arrive_relaxed();  // this CTA's barriers are initialised
    pdl_wait();
    if (threadIdx.x == 0) {
        const uint64_t policy = l2_evict_first_policy();  // read once
        const uint32_t bytes = (uint32_t)n * 16u;
        mbar_arrive_expect_tx(bar, bytes);
        for (uint32_t off = 0; off < bytes; off += 32768u) {
            const uint32_t len = bytes - off < 32768u ? bytes - off : 32768u;
            bulk_load_g2s_hint(smem_u32(stage) + off, src + off, len, bar, policy);
        }
    }
    bool ok = __syncthreads_and(mbar_wait_bounded(bar, 0, 1000000000ull));
    if (!ok) mbar_wait_bounded(bar, 0, 1000000000ull);  // own copies still landing

    // the CTA's maximum and the first index holding it (each thread visits
    // its vectors in increasing index order and keeps the first vector whose
    // maximum beats its running one; NaN never wins), then its sum of exps
    // on f32x2 pairs
    float tm = -INFINITY;
    int ju = -1;  // the vector holding this thread's maximum
    if (ok) {
        for (int u = threadIdx.x; u < n; u += T) {
            const uint4 q = *reinterpret_cast<const uint4 *>(stage + u * 16);
            float um;
            if constexpr (DI == Dt::BF16) {
                const uint32_t w = lse_max_bf16x2(lse_max_bf16x2(q.x, q.y), lse_max_bf16x2(q.z, q.w));
                um = fmaxf(bf16_lo(w), bf16_hi(w));
            } else {
                um = fmaxf(fmaxf(__uint_as_float(q.x), __uint_as_float(q.y)),
                           fmaxf(__uint_as_float(q.z), __uint_as_float(q.w)));
            }
            if (um > tm) {
                tm = um;
                ju = u;
            }
        }
    }
    int64_t ti = kNoIndex;
    if (ju >= 0) {
        float v[U];
        load_unit<DI, U, Hint::Keep>(stage, (int64_t)ju * U, v);
#pragma unroll
        for (int k = U - 1; k >= 0; --k)
            if (v[k] == tm) ti = (u0 + ju) * U + k;  // the last hit is the first
    }
    float m = group_max<32>(tm);
    if (lane == 0) s_m[warp] = m;
    __syncthreads();
    m = group_max<NW>(s_m[lane & (NW - 1)]);
    const int64_t wi = group_min_i64<32>(tm == m ? ti : kNoIndex);
    float td = 0.f;
    if (ok) {
        const uint64_t m2 = f2_make(md_shift(m), md_shift(m)),
                       l2e = f2_make(1.4426950408889634f, 1.4426950408889634f);
        uint64_t acc = f2_make(0.f, 0.f);
        for (int u = threadIdx.x; u < n; u += T) {
            const uint4 q = *reinterpret_cast<const uint4 *>(stage + u * 16);
#pragma unroll
            for (int k = 0; k < U / 2; ++k) {
                const uint64_t e = f2_mul(f2_sub(f2_of<DI>(q, k), m2), l2e);
                acc = f2_add(acc, f2_make(ex2_approx(f2_lo(e)), ex2_approx(f2_hi(e))));
            }
        }
        td = f2_lo(acc) + f2_hi(acc);
    }
    const float wd = group_sum<32>(td);
    if (lane == 0) {
        s_d[warp] = wd;
        s_i[warp] = wi;
    }
    __syncthreads();
    MaxArgSum r{m, group_sum<NW>(s_d[lane & (NW - 1)]), group_min_i64<NW>(s_i[lane & (NW - 1)])};

    cluster_wait_acquire();  // every peer's xbar is initialised
    if (threadIdx.x < a.cs) {
        const uint4 v = make_uint4(__float_as_uint(r.m), __float_as_uint(r.d), (uint32_t)r.i,
                                   (uint32_t)((uint64_t)r.i >> 32));
        st_async_v4(mapa_shared(smem_u32(&xslot[rank]), threadIdx.x), mapa_shared(xbar, threadIdx.x), v);
    }
    ok = mbar_wait_bounded(xbar, 0, 2000000000ull) && ok;
    const int q = threadIdx.x & 15;
    MaxArgSum p{-INFINITY, 0.f, kNoIndex};
    if (q < a.cs) {
        const uint4 v = xslot[q];
        p = MaxArgSum{__uint_as_float(v.x), __uint_as_float(v.y), (int64_t)(((uint64_t)v.w << 32) | v.z)};
    }
    r = group_mas<16>(p);
    if (threadIdx.x == 0 && u0 == 0) {
        // a copy or state that never arrived (bounded waits) gives NaN and -1
        if (a.row_sum != nullptr) a.row_sum[row] = ok ? r.m + logf(r.d) : __int_as_float(0x7fffffff);
        if (a.row_arg != nullptr) a.row_arg[row] = ok && r.i != kNoIndex ? r.i : -1;
    }
    pdl_trigger();
}

namespace {

using KernelFn = void (*)(RowArgs);

cudaError_t launch_fn(KernelFn k, int64_t grid, int threads, int cs, const RowArgs &a,
                      cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(threads);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    int n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n++].val.programmaticStreamSerializationAllowed = use_pdl() ? 1 : 0;
    if (cs > 0) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = (unsigned)cs;
        attr[n].val.clusterDim.y = 1;
        attr[n++].val.clusterDim.z = 1;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, k, a);
}

template <Dt DI, int U, bool PEEL = false>
cudaError_t launch_lse_u(const RowArgs &a, int g, bool cluster, int64_t grid, cudaStream_t st) {
    KernelFn fn = nullptr;
    if (cluster) {
        if (g == 256) fn = lse_argmax_kernel<DI, 256, U, true, PEEL>;
        if (!fn) return cudaErrorInvalidConfiguration;
        if (a.cs > 8) {
            const cudaError_t e =
                cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
        }
        return launch_fn(fn, grid, 256, a.cs, a, st);
    }
#define OSR_MAKE(G) \
    if (g == G) fn = lse_argmax_kernel<DI, G, U, false, PEEL>;
    if constexpr (PEEL) {
        // a lane per edge element: groups of at least U lanes
        if constexpr (U <= 4) { OSR_MAKE(4) }
        OSR_MAKE(8) OSR_MAKE(16) OSR_MAKE(32) OSR_MAKE(64) OSR_MAKE(128) OSR_MAKE(256) OSR_MAKE(512)
        OSR_MAKE(1024)
    } else {
        OSR_MAKE(1) OSR_MAKE(2) OSR_MAKE(4) OSR_MAKE(8) OSR_MAKE(16) OSR_MAKE(32) OSR_MAKE(64)
        OSR_MAKE(128) OSR_MAKE(256) OSR_MAKE(512) OSR_MAKE(1024)
    }
#undef OSR_MAKE
    if (!fn) return cudaErrorInvalidConfiguration;
    return launch_fn(fn, grid, g <= 32 ? RowsGeom<1>::kThreads : g, 0, a, st);
}

}  // namespace

template <Dt DI>
cudaError_t launch_lse_staged(const RowArgs &a, int64_t grid, size_t smem, cudaStream_t st) {
    const KernelFn fn = lse_staged_kernel<DI>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess && a.cs > 8) e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = use_pdl() ? 1 : 0;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)a.cs;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, fn, a);
}

template <Dt DI>
cudaError_t launch_lse(const RowArgs &a, int g, bool cluster, bool vec, int64_t grid,
                       cudaStream_t st) {
    if (vec) return launch_lse_u<DI, Elem<DI>::kVec>(a, g, cluster, grid, st);
    return launch_lse_u<DI, 1>(a, g, cluster, grid, st);
}

template <Dt DI>
cudaError_t launch_lse_peel(const RowArgs &a, int g, bool cluster, int64_t grid, cudaStream_t st) {
    return launch_lse_u<DI, Elem<DI>::kVec, true>(a, g, cluster, grid, st);
}

template cudaError_t launch_lse<Dt::F32>(const RowArgs &, int, bool, bool, int64_t, cudaStream_t);
template cudaError_t launch_lse_peel<Dt::F32>(const RowArgs &, int, bool, int64_t, cudaStream_t);
template cudaError_t launch_lse_peel<Dt::BF16>(const RowArgs &, int, bool, int64_t, cudaStream_t);
template cudaError_t launch_lse<Dt::BF16>(const RowArgs &, int, bool, bool, int64_t, cudaStream_t);
template cudaError_t launch_lse_staged<Dt::F32>(const RowArgs &, int64_t, size_t, cudaStream_t);
template cudaError_t launch_lse_staged<Dt::BF16>(const RowArgs &, int64_t, size_t, cudaStream_t);

}  // namespace osr
