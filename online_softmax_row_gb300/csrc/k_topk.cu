// k_topk.cu -- top-k sampling prologue of vocabulary rows: per row the k
// largest logits (largest first, equal values by lower index, NaN above every
// number), their column indices, the softmax of those k logits and the
// log-sum-exp of the whole row, from one read of the row.
//
// "Softmax 与归一化" (anrans.github.io), exercise 2 "大词表采样": sampling
// needs no softmax row written out -- top-k sampling selects the k largest
// logits first and normalises only those, and a long row with few rows is
// spread over several CTAs whose partial results are merged.  The selection
// counts elements by digit buckets, the ballot-and-count pattern that
// "两个融合算子：RMSNorm 与 online softmax" (daleiyang.github.io) §3 names for
// top-k bucketing, here with shared-memory histograms.
//
// One thread-block cluster of cs CTAs per row; CTA r copies elements
// [r * chunk, (r + 1) * chunk) of the row into shared memory (cp.async: the
// row is read from HBM once) and works on that copy:
//   bound   -- each thread's largest number; per warp the ceil(k/8)-th
//              largest of those, and g = the smallest over the warps: at
//              least k elements of the CTA are >= g, so the row's k-th largest
//              is >= g and nothing below g can be selected;
//   sweep   -- one pass: the CTA's (m, d) = (max, sum of e^(x - max)) for the
//              log-sum-exp, and every element not below g appended to a
//              short list as a (key, column) word (keys: an order-preserving
//              integer map, -0 as +0, NaN above every number; words order by
//              key, then by smaller column, and all differ);
//   merge   -- one exchange: each CTA stores its (m, d) and list length
//              into every CTA (st.async, counted on the receiver's
//              mbarrier); the row's (m, d) by the (m, d) merge of the CTAs'
//              (lse = m + log d);
//   select  -- every CTA stores its list into CTA 0 the same way, and CTA 0,
//              with the union of the lists (it holds every element at or
//              above the k-th largest), finds the k-th largest key T by
//              8-bit radix passes over it, takes the words above T and the
//              largest of those equal to T, and writes them in order (values
//              rebuilt from their keys, zeros and NaNs re-read from the row;
//              columns; the softmax of the k values).
// When a list overflows (k > 256 gives no bound; heavy ties at the bound) or
// the union does not fit, the cluster selects together instead: radix passes
// over the lists or the whole pieces with the histograms summed through
// distributed shared memory each pass (behind cluster barriers), and the
// equal keys shared out by a prefix over the CTAs.  The result is unique (a
// total order), so it is deterministic.  The exchanges' waits are bounded
// (2 s); one that runs out writes NaN / -1 for the row.
#include <cuda_runtime.h>

#include <type_traits>

#include "launch.h"
#include "topk.h"

namespace osr {

namespace {

constexpr int kWarps = kTopkThreads / 32;

// Order-preserving key: larger value -> larger unsigned key.  -0 is keyed as
// +0 and every NaN as the quiet NaN above +inf.
__device__ __forceinline__ uint32_t topk_key(uint32_t bits, Dt dt) {
    if (dt == Dt::BF16) {
        if ((bits & 0x7fffu) > 0x7f80u) bits = 0x7fc0u;
        if (bits == 0x8000u) bits = 0u;
        return (bits & 0x8000u) ? (~bits & 0xffffu) : (bits | 0x8000u);
    }
    if ((bits & 0x7fffffffu) > 0x7f800000u) bits = 0x7fc00000u;
    if (bits == 0x80000000u) bits = 0u;
    return (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
}

__device__ __forceinline__ float raw_to_f32(uint32_t bits, Dt dt) {
    return __uint_as_float(dt == Dt::BF16 ? bits << 16 : bits);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// Remote shared-memory loads.  volatile keeps them after the cluster
// barrier (itself volatile, with a memory clobber); they have no clobber of
// their own, so several can be in flight at once.
__device__ __forceinline__ uint32_t ld_dsmem_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint64_t ld_dsmem_u64(uint32_t addr) {
    uint64_t v;
    asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(addr));
    return v;
}

// dst[0, cnt) <- cnt words of another CTA's shared memory at `src`, four
// remote loads in flight per thread
__device__ __forceinline__ void copy_words(uint64_t *dst, uint32_t src, uint32_t cnt) {
    for (uint32_t i0 = threadIdx.x; i0 < cnt; i0 += 4 * kTopkThreads) {
        uint64_t v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t i = i0 + j * kTopkThreads;
            v[j] = i < cnt ? ld_dsmem_u64(src + i * 8) : 0ull;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t i = i0 + j * kTopkThreads;
            if (i < cnt) dst[i] = v[j];
        }
    }
}

__device__ __forceinline__ void cluster_sync_all() {
    cluster_arrive_release();
    cluster_wait_acquire();
}

// Inclusive sum over the CTA's threads in thread order; `scratch` holds
// kWarps values.  With END_SYNC it ends with the CTA synchronised (scratch
// free again); without, the caller synchronises before reusing scratch.
template <bool END_SYNC = true>
__device__ __forceinline__ uint32_t block_inclusive_scan(uint32_t v, uint32_t *scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t o = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += o;
    }
    if (lane == 31) scratch[warp] = v;
    __syncthreads();
    uint32_t before = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) before += w < warp ? scratch[w] : 0u;
    if (END_SYNC) __syncthreads();
    return v + before;
}

__device__ __forceinline__ float block_max_f(float v, float *scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = group_max<32>(v);
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    v = group_max<kWarps>(scratch[lane & (kWarps - 1)]);
    __syncthreads();
    return v;
}

// The CTA's sum (a fixed tree); END_SYNC as in block_inclusive_scan.
template <bool END_SYNC = true>
__device__ __forceinline__ float block_sum_f(float v, float *scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = group_sum<32>(v);
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    v = group_sum<kWarps>(scratch[lane & (kWarps - 1)]);
    if (END_SYNC) __syncthreads();
    return v;
}

// The number a key stands for (-0 comes back as +0, NaN as the quiet NaN).
template <Dt DI>
__device__ __forceinline__ float key_value(uint32_t key) {
    if constexpr (DI == Dt::BF16) {
        const uint32_t b = (key & 0x8000u) ? (key & 0x7fffu) : (~key & 0xffffu);
        return __uint_as_float(b << 16);
    } else {
        return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
    }
}

// Larger of two numbers, NaN if either is NaN (the sweep's pre-filter must
// not drop a NaN, which ranks above every number).
__device__ __forceinline__ float max_nan_f32(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// per half: the larger number, NaN if either is NaN
__device__ __forceinline__ uint32_t max_nan_bf16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint32_t max_bf16x2(uint32_t a, uint32_t b) {
    uint32_t r;  // per half: the larger number (a NaN loses to a number)
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Float value of element e of a 16-byte vector of raw values.
template <Dt DI>
__device__ __forceinline__ float raw_value_at(const uint4 &q, int e) {
    if constexpr (DI == Dt::BF16) {
        const uint32_t w = e < 2 ? q.x : e < 4 ? q.y : e < 6 ? q.z : q.w;
        return (e & 1) ? bf16_hi(w) : bf16_lo(w);
    } else {
        return __uint_as_float(e == 0 ? q.x : e == 1 ? q.y : e == 2 ? q.z : q.w);
    }
}

template <Dt DI>
__device__ __forceinline__ uint32_t raw_bits_at(const uint4 &q, int e) {
    if constexpr (DI == Dt::BF16) {
        const uint32_t w = e < 2 ? q.x : e < 4 ? q.y : e < 6 ? q.z : q.w;
        return (e & 1) ? w >> 16 : w & 0xffffu;
    } else {
        return e == 0 ? q.x : e == 1 ? q.y : e == 2 ? q.z : q.w;
    }
}

// Warp-wide sort of one float per lane, largest in lane 0 (bitonic network
// on shuffles; no NaN among the inputs).
__device__ __forceinline__ float warp_sort_desc(float v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const float o = __shfl_xor_sync(0xffffffffu, v, stride);
            const bool lower = (lane & stride) == 0, desc = (lane & size) == 0;
            v = lower == desc ? fmaxf(v, o) : fminf(v, o);
        }
    }
    return v;
}

template <Dt DI, int U>
__global__ void __launch_bounds__(kTopkThreads, 4) topk_kernel(const TopkArgs a) {
    using Raw = typename std::conditional<DI == Dt::BF16, uint16_t, uint32_t>::type;
    constexpr int KB = DI == Dt::BF16 ? 16 : 32;  // key bits
    constexpr int PASSES = KB / 8;
    extern __shared__ __align__(16) unsigned char smem[];
    Raw *piece = reinterpret_cast<Raw *>(smem);             // the piece, raw
    uint64_t *words = reinterpret_cast<uint64_t *>(smem);    // reuses the piece region
    uint32_t *hist = reinterpret_cast<uint32_t *>(smem + a.region0);
    uint32_t *hist_pub = hist + 256;                         // [2][256]
    uint64_t *list = reinterpret_cast<uint64_t *>(hist_pub + 2 * 256);
    uint64_t *cand = list + kTopkListCap;
    __shared__ float s_red[kWarps], s_gw[kWarps];
    __shared__ uint32_t s_scan[kWarps];
    __shared__ float s_ez[kTopkRankMaxK];
    __shared__ uint32_t pub_cand, list_n, s_bin, s_krem;
    __shared__ uint64_t s_top;
    // exchanges without a cluster barrier: st.async into the receiver's
    // shared memory, counted on its mbarrier.  xbar[0]: every CTA's
    // (m, d, list length) into xstate[its rank] of every CTA; xbar[1]: on
    // the short path, every CTA's list into CTA 0's union
    __shared__ __align__(8) uint64_t xbar_words[3];
    __shared__ uint4 xstate[kTopkMaxCluster];
    __shared__ float2 xg[kTopkMaxCluster];  // xbar[2]: every CTA's bound g

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cs = a.cs;
    const uint32_t rank = cluster_ctarank();
    const int64_t row = blockIdx.x / (uint32_t)cs;
    const int64_t e0 = (int64_t)rank * a.chunk;
    const int64_t e1 = e0 + a.chunk < a.N ? e0 + a.chunk : a.N;
    const int n = e1 > e0 ? (int)(e1 - e0) : 0;  // elements of this CTA's piece
    const Raw *xrow = reinterpret_cast<const Raw *>(a.x) + row * a.N;
    const int64_t k = a.k;
    const uint32_t inv = 0xffffffffu;
    // (key, column) <-> one 64-bit word ordered by key, then by smaller column
    auto word = [&](uint32_t key, int64_t col) {
        return ((uint64_t)key << 32) | (uint64_t)(inv - (uint32_t)col);
    };
    auto candidate = [&](uint64_t w) {
        const uint32_t pos = atomicAdd(&pub_cand, 1u);
        if (pos < (uint32_t)k) cand[pos] = w;  // at most k by construction
    };
    // every element of the piece as (value, raw bits, column), in any order
    auto sweep_piece = [&](auto &&f) {
        if constexpr (U > 1) {
            const uint4 *pv = reinterpret_cast<const uint4 *>(piece);
            for (int i = tid; i < n / U; i += kTopkThreads) {
                const uint4 q = pv[i];
#pragma unroll
                for (int e = 0; e < U; ++e) f(raw_value_at<DI>(q, e), raw_bits_at<DI>(q, e), e0 + i * U + e);
            }
        } else {
            for (int i = tid; i < n; i += kTopkThreads) {
                const uint32_t b = piece[i];
                f(raw_to_f32(b, DI), b, e0 + i);
            }
        }
    };

    const uint32_t xbar0 = smem_u32(&xbar_words[0]), xbar1 = smem_u32(&xbar_words[1]),
                   xbar2 = smem_u32(&xbar_words[2]);
    if (tid == 0) {
        pub_cand = 0;
        list_n = 0;
        mbar_init(xbar0, 1);
        mbar_init(xbar1, 1);
        mbar_init(xbar2, 1);
        mbar_arrive_expect_tx(xbar0, (uint32_t)cs * 16u);
        mbar_arrive_expect_tx(xbar2, (uint32_t)cs * 8u);
        fence_mbar_init();
    }
    __syncthreads();
    cluster_arrive_relaxed();  // this CTA's barriers are initialised
    pdl_wait();

    // ---- load the piece (the row is read from HBM once, every copy in
    //      flight at once) and take each thread's largest number (NaN skipped)
    float tmax = -INFINITY;
    if constexpr (U > 1) {
        const char *src = reinterpret_cast<const char *>(xrow + e0);
        uint4 *pv = reinterpret_cast<uint4 *>(piece);
        const int nv = n / U;  // n is a multiple of U on the vector path
        for (int i = tid; i < nv; i += kTopkThreads) cp_async16(smem_u32(pv + i), src + (int64_t)i * 16);
        cp_async_wait_all();  // this thread's own copies; it reads only those here
        if constexpr (DI == Dt::BF16) {
            uint32_t mx = 0xff80ff80u;  // (-inf, -inf)
            for (int i = tid; i < nv; i += kTopkThreads) {
                const uint4 q = pv[i];
                mx = max_bf16x2(mx, max_bf16x2(max_bf16x2(q.x, q.y), max_bf16x2(q.z, q.w)));
            }
            tmax = fmaxf(bf16_lo(mx), bf16_hi(mx));
        } else {
            for (int i = tid; i < nv; i += kTopkThreads) {
                const uint4 q = pv[i];
                tmax = fmaxf(tmax, fmaxf(fmaxf(__uint_as_float(q.x), __uint_as_float(q.y)),
                                         fmaxf(__uint_as_float(q.z), __uint_as_float(q.w))));
            }
        }
    } else {
        // a piece off the 16-byte grid: placed in shared memory as many bytes
        // past a boundary as it lies in global memory, so its whole 16-byte
        // chunks go by cp.async as on the vector path and only the few
        // elements before the first boundary and after the last are loaded
        // one by one (the region has 16 bytes to spare for the shift)
        const char *src = reinterpret_cast<const char *>(xrow + e0);
        const uint32_t mis = (uint32_t)(reinterpret_cast<uintptr_t>(src) & 15u);
        piece = reinterpret_cast<Raw *>(smem + mis);
        const int head = (int)(mis ? (16u - mis) / sizeof(Raw) : 0u) < n ? (int)(mis ? (16u - mis) / sizeof(Raw) : 0u) : n;
        const int nch = (int)((int64_t)(n - head) * (int64_t)sizeof(Raw) / 16);
        const int t0 = head + nch * (int)(16 / sizeof(Raw));
        const char *body = src + head * sizeof(Raw);
        unsigned char *dst = smem + mis + head * sizeof(Raw);  // 16-byte aligned
        for (int i = tid; i < nch; i += kTopkThreads) cp_async16(smem_u32(dst + i * 16), body + (int64_t)i * 16);
        for (int i = tid; i < head; i += kTopkThreads) piece[i] = xrow[e0 + i];
        for (int i = t0 + tid; i < n; i += kTopkThreads) piece[i] = xrow[e0 + i];
        cp_async_wait_all();
        __syncthreads();  // every thread's copies have landed
        for (int i = tid; i < n; i += kTopkThreads) tmax = fmaxf(tmax, raw_to_f32(piece[i], DI));
    }

    // ---- a lower bound g of the row's k-th largest element.  With
    //      q = ceil(k/8), take in each warp the q-th largest lane maximum and
    //      let g be the smallest of those: at least 8q >= k threads hold a
    //      number >= g, so nothing below g is among the k largest (a NaN
    //      ranks above every number and is always kept).  k > 256: no bound.
    const uint32_t qk = (uint32_t)((k + kWarps - 1) / kWarps);
    const float sorted = warp_sort_desc(tmax);
    const float gw = __shfl_sync(0xffffffffu, sorted, (int)((qk <= 32 ? qk : 32) - 1));
    if (lane == 0) s_gw[warp] = gw;
    const float cmax = block_max_f(tmax, s_red);  // its barriers publish s_gw too
    float g = -INFINITY;
    if (qk <= 32) {
        g = INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) g = fminf(g, s_gw[w]);
    }

    // Every CTA's g is a lower bound of the row's k-th largest (it holds k
    // elements >= g), so their maximum is one too: sent to every CTA now,
    // read after the exps, so the lists keep only elements >= that maximum.
    cluster_wait_acquire();  // every peer's barriers are initialised
    if (tid < cs) st_async_f2(mapa_shared(smem_u32(&xg[rank]), tid), mapa_shared(xbar2, tid), g, 0.f);
    auto row_bound = [&]() {
        float gr = g;
        if (mbar_wait_bounded(xbar2, 0, 2000000000ull))  // else the exchange below fails
            for (int r = 0; r < cs; ++r) gr = fmaxf(gr, xg[r].x);
        return gr;
    };

    // ---- one sweep: this CTA's (m, d) for the log-sum-exp, and the elements
    //      not below g, as (key, column) words, into a short list
    const float mc = fmaxf(cmax, -FLT_MAX);
    float dt = 0.f;
    auto keep = [&](uint32_t bits, int64_t col) {
        const uint32_t pos = atomicAdd(&list_n, 1u);
        if (pos < (uint32_t)kTopkListCap) list[pos] = word(topk_key(bits, DI), col);
    };
    if constexpr (U > 1) {
        // two passes.  First every vector's exps (two running sums, shorter
        // add chains) and a bit per vector whose largest value (NaN kept) is
        // not below g; then, for those few vectors only, the elements into
        // the list.  Measured on the vocabulary rows: one pass with the
        // element tests and appends inside took 5.7 us, the exps alone 2.7.
        const uint4 *pv = reinterpret_cast<const uint4 *>(piece);
        // the exps on binary32 pairs (sub, mul, add .f32x2; each lane rounds
        // as the scalar instruction): lane 0 sums the even elements, lane 1
        // the odd ones
        const uint64_t m2 = f2_make(mc, mc), l2e = f2_make(1.4426950408889634f, 1.4426950408889634f);
        uint64_t acc = f2_make(0.f, 0.f);
        uint64_t hit = 0;  // bit j: vector tid + j * kTopkThreads (at most 64 a thread)
        for (int i = tid, j = 0; i < n / U; i += kTopkThreads, ++j) {
            const uint4 q = pv[i];
            float um;
            if constexpr (DI == Dt::BF16) {
                const uint32_t w = max_nan_bf16x2(max_nan_bf16x2(q.x, q.y), max_nan_bf16x2(q.z, q.w));
                um = max_nan_f32(bf16_lo(w), bf16_hi(w));
            } else {
                um = max_nan_f32(max_nan_f32(__uint_as_float(q.x), __uint_as_float(q.y)),
                                 max_nan_f32(__uint_as_float(q.z), __uint_as_float(q.w)));
            }
#pragma unroll
            for (int k = 0; k < U / 2; ++k) {
                const uint64_t t = f2_mul(f2_sub(f2_of<DI>(q, k), m2), l2e);
                acc = f2_add(acc, f2_make(ex2_approx(f2_lo(t)), ex2_approx(f2_hi(t))));
            }
            hit |= (uint64_t)!(um < g) << j;
        }
        const float d0 = f2_lo(acc), d1 = f2_hi(acc);
        const float gr = row_bound();
        while (hit != 0) {
            const int j = __ffsll((long long)hit) - 1;
            hit &= hit - 1;
            const int i = tid + j * kTopkThreads;
            const uint4 q = pv[i];
#pragma unroll
            for (int e = 0; e < U; ++e)
                if (!(raw_value_at<DI>(q, e) < gr)) keep(raw_bits_at<DI>(q, e), e0 + (int64_t)i * U + e);
        }
        dt = d0 + d1;
    } else {
        const float gr = row_bound();
        sweep_piece([&](float v, uint32_t bits, int64_t col) {
            dt += exp_shifted(v, mc);
            if (!(v < gr)) keep(bits, col);
        });
    }
    dt = block_sum_f(dt, s_red);  // also orders the list appends
    const uint32_t nl = list_n;

    // ---- exchange: the row's (m, d) by the merge of the CTAs' (m, d), and
    //      the lists' lengths
    if (tid < cs)
        st_async_v4(mapa_shared(smem_u32(&xstate[rank]), tid), mapa_shared(xbar0, tid),
                    make_uint4(__float_as_uint(mc), __float_as_uint(dt), nl, 0u));
    auto fail = [&]() {  // a state or list that never arrived (bounded waits: 2 s)
        for (int64_t t = tid; rank == 0 && t < k; t += kTopkThreads) {
            a.values[row * k + t] = __uint_as_float(0x7fc00000u);
            a.indices[row * k + t] = -1;
            if (a.probs != nullptr) a.probs[row * k + t] = __uint_as_float(0x7fc00000u);
        }
        if (rank == 0 && tid == 0 && a.lse != nullptr) a.lse[row] = __uint_as_float(0x7fc00000u);
        pdl_trigger();
    };
    if (!__syncthreads_and(mbar_wait_bounded(xbar0, 0, 2000000000ull))) {
        fail();
        return;
    }
    float m = -FLT_MAX, d = 0.f;
    uint32_t over = 0, total = 0;
    for (int r = 0; r < cs; ++r) {
        const uint32_t rn = xstate[r].z;
        m = fmaxf(m, __uint_as_float(xstate[r].x));
        over |= rn > (uint32_t)kTopkListCap;
        total += rn < (uint32_t)kTopkListCap ? rn : (uint32_t)kTopkListCap;
    }
    for (int r = 0; r < cs; ++r)
        d += __uint_as_float(xstate[r].y) * expf(__uint_as_float(xstate[r].x) - m);
    if (rank == 0 && a.lse != nullptr && tid == 0) a.lse[row] = m + logf(d);

    // The row's own value of a word.  A key stands for one bit pattern except
    // the keys of zero (+0 and -0) and of NaN (every NaN): those two are
    // re-read from the row (in L2), the rest rebuilt from the key.  An index
    // outside the row could only come from a selection that found fewer than
    // k candidates: reported as NaN, never read.
    const uint32_t zero_key = topk_key(0u, DI), nan_key = topk_key(DI == Dt::BF16 ? 0x7fc0u : 0x7fc00000u, DI);
    auto store = [&](int64_t t, uint64_t w, float p) {
        const uint32_t key = (uint32_t)(w >> 32), j = inv - (uint32_t)w;
        const bool in_row = j < (uint32_t)a.N;
        a.values[row * k + t] = !in_row ? __uint_as_float(0x7fc00000u)
                                : key == zero_key || key == nan_key ? raw_to_f32(xrow[j], DI)
                                                                    : key_value<DI>(key);
        a.indices[row * k + t] = in_row ? (int64_t)j : -1;
        if (a.probs != nullptr) a.probs[row * k + t] = p;
    };
    // Radix selection of the k-th largest key T among keys delivered by
    // `each` (8 bits per pass from the top).  `merge(b)` gives the count of
    // digit b in the histogram the choice is made from (the cluster's sum,
    // or the CTA's own); returns T and leaves in krem how many keys equal to
    // T belong to the k largest.
    uint32_t krem = (uint32_t)k;
    auto radix_select = [&](auto &&each, auto &&merge) {
        uint32_t prefix = 0;
        krem = (uint32_t)k;
#pragma unroll 1
        for (int p = 0; p < PASSES; ++p) {
            const int shift = KB - 8 * (p + 1);
            hist[tid] = 0u;
            __syncthreads();
            each([&](uint32_t key, int64_t) {
                if (p == 0 || (key >> (shift + 8)) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
            });
            __syncthreads();
            // S_b = keys in play with digit >= b, an inclusive scan in
            // descending digit order: thread t takes digit 255 - t
            const uint32_t Hr = merge(255 - tid);
            // s_scan, s_bin and s_krem are next written after at least two
            // more barriers, which every reader passes first: no barrier
            // closes the scan or the pass
            const uint32_t S = block_inclusive_scan<false>(Hr, s_scan);
            if (S >= krem && S - Hr < krem) {
                s_bin = 255u - (uint32_t)tid;
                s_krem = krem - (S - Hr);
            }
            __syncthreads();
            prefix = (prefix << 8) | s_bin;
            krem = s_krem;
        }
        return prefix;
    };

    bool in_cand = false;  // CTA 0's k words: in `cand` (short path) or in `words`
    if (!over && total <= a.region0 / 8) {
        // ---- the short path: the union of the lists holds every element at
        //      or above the k-th largest (each CTA's bound lies below it).
        //      Every CTA stores its list into CTA 0's union (which reuses the
        //      piece region, no longer read once the states went out); CTA 0
        //      selects from it alone.
        uint32_t off = 0;
        for (int r = 0; r < (int)rank; ++r) off += xstate[r].z;
        if (rank == 0 && tid == 0) mbar_arrive_expect_tx(xbar1, total * 8u);
        const uint32_t to_words = mapa_shared(smem_u32(words + off), 0), to_bar = mapa_shared(xbar1, 0);
        for (uint32_t i = tid; i < nl; i += kTopkThreads) st_async_u64(to_words + i * 8u, to_bar, list[i]);
        if (rank != 0) {
            pdl_trigger();
            return;
        }
        if (!__syncthreads_and(mbar_wait_bounded(xbar1, 0, 2000000000ull))) {
            fail();
            return;
        }
        // every thread has read the list length; the radix passes' barriers
        // order this reset before the gathering below
        if (tid == 0) list_n = 0;
        auto each_u = [&](auto &&f) {
            for (uint32_t i = tid; i < total; i += kTopkThreads) f((uint32_t)(words[i] >> 32), (int64_t)i);
        };
        const uint32_t T = radix_select(each_u, [&](int b) { return hist[b]; });
        // keys above T, and the krem largest words among those equal to T
        // (equal keys: the smaller columns; every word differs).  The equal
        // words are gathered into `list` (free now) and ranked among
        // themselves.
        for (uint32_t i = tid; i < total; i += kTopkThreads) {
            const uint64_t w = words[i];
            const uint32_t key = (uint32_t)(w >> 32);
            if (key > T) candidate(w);
            if (key == T) {
                const uint32_t pos = atomicAdd(&list_n, 1u);
                if (pos < (uint32_t)kTopkListCap) list[pos] = w;
            }
        }
        __syncthreads();
        const uint32_t ne = list_n;
        if (ne <= (uint32_t)kTopkListCap) {
            for (uint32_t i = tid; i < ne; i += kTopkThreads) {
                const uint64_t w = list[i];
                uint32_t larger = 0;
                for (uint32_t j = 0; j < ne; ++j) larger += list[j] > w;
                if (larger < krem) candidate(w);
            }
        } else {  // too many equal keys to gather: rank them over the union
            for (uint32_t i = tid; i < total; i += kTopkThreads) {
                const uint64_t w = words[i];
                if ((uint32_t)(w >> 32) != T) continue;
                uint32_t larger = 0;
                for (uint32_t j = 0; j < total; ++j) larger += (uint32_t)(words[j] >> 32) == T && words[j] > w;
                if (larger < krem) candidate(w);
            }
        }
        in_cand = true;
    } else {
        // ---- otherwise the cluster selects together, over the lists (or,
        //      when a list overflowed, over the whole pieces).  Published
        //      histograms alternate between two buffers per exchange, so a
        //      CTA never overwrites one another CTA may still read.
        const bool full = over != 0;  // cluster-uniform
        auto each = [&](auto &&f) {
            if (full) {
                sweep_piece([&](float, uint32_t bits, int64_t col) { f(topk_key(bits, DI), col); });
            } else {
                for (uint32_t i = tid; i < nl; i += kTopkThreads) {
                    const uint64_t w = list[i];
                    f((uint32_t)(w >> 32), (int64_t)(inv - (uint32_t)w));
                }
            }
        };
        int xb = 0;
        uint32_t *pub = nullptr;
        auto cluster_merge = [&](int b) {
            pub = hist_pub + xb * 256;
            pub[tid] = hist[tid];
            xb ^= 1;
            cluster_sync_all();
            uint32_t H = 0;
            for (int r = 0; r < cs; ++r) H += ld_dsmem_u32(mapa_shared(smem_u32(pub + b), r));
            return H;
        };
        const uint32_t T = radix_select(each, cluster_merge);
        // the last histograms count, per CTA, the keys equal to T: bin (T & 255)
        uint32_t eq_before = 0;
        for (int r = 0; r < (int)rank; ++r)
            eq_before += ld_dsmem_u32(mapa_shared(smem_u32(pub + (T & 255u)), r));
        const uint32_t eq_here = pub[T & 255u];
        const uint32_t quota = krem > eq_before ? (krem - eq_before < eq_here ? krem - eq_before : eq_here) : 0u;
        const bool all_eq = quota == eq_here;
        each([&](uint32_t key, int64_t col) {
            if (key > T || (all_eq && key == T && quota > 0)) candidate(word(key, col));
        });
        if (!all_eq && quota > 0) {
            // a partial share (one CTA of the row at most): the lowest-indexed
            // equal keys.  Each thread walks a contiguous range of the piece,
            // so index order is (thread, position): count, scan, take in order.
            const int L = (n + kTopkThreads - 1) / kTopkThreads;
            const int j0 = tid * L < n ? tid * L : n, j1 = j0 + L < n ? j0 + L : n;
            uint32_t c = 0;
            for (int j = j0; j < j1; ++j) c += topk_key(piece[j], DI) == T;
            const uint32_t incl = block_inclusive_scan(c, s_scan);
            uint32_t r = incl - c;  // equal keys before this thread's range
            for (int j = j0; j < j1 && r < quota; ++j)
                if (topk_key(piece[j], DI) == T) {
                    candidate(word(T, e0 + j));
                    ++r;
                }
        }
        cluster_sync_all();  // every CTA's candidates are complete
        if (rank == 0) {
            uint32_t off = 0;
            for (int r = 0; r < cs; ++r) {
                uint32_t cnt = ld_dsmem_u32(mapa_shared(smem_u32(&pub_cand), r));
                cnt = off + cnt <= (uint32_t)k ? cnt : (off < (uint32_t)k ? (uint32_t)k - off : 0u);
                copy_words(words + off, mapa_shared(smem_u32(cand), r), cnt);
                off += cnt;
            }
        }
        cluster_sync_all();  // no CTA leaves while CTA 0 reads its candidates
        if (rank != 0) {
            pdl_trigger();
            return;
        }
    }
    __syncthreads();

    // ---- CTA 0 writes the k words in order: values, columns, the softmax of
    //      the k values (largest first, so v0 is their maximum), summed in
    //      output order
    if (k <= kTopkRankMaxK) {
        // output position = the number of larger words (all words differ)
        const uint64_t *kw = in_cand ? cand : words;
        int64_t t = 0;
        uint64_t w = 0;
        if (tid < k) {
            w = kw[tid];
            for (int j = 0; j < k; ++j) t += kw[j] > w;
            if (t == 0) s_top = w;
        }
        __syncthreads();
        const float v0 = key_value<DI>((uint32_t)(s_top >> 32));  // the largest value
        if (tid < k) s_ez[t] = expf(key_value<DI>((uint32_t)(w >> 32)) - v0);
        __syncthreads();
        const float rz = __frcp_rn(block_sum_f<false>(tid < k ? s_ez[tid] : 0.f, s_red));
        if (tid < k) store(t, w, s_ez[t] * rz);
    } else {
        if (in_cand) {
            for (int i = tid; i < k; i += kTopkThreads) words[i] = cand[i];
            __syncthreads();
        }
        // a bitonic network on a.sort_n >= k words (zero words sort last)
        for (int i = (int)k + tid; i < a.sort_n; i += kTopkThreads) words[i] = 0ull;
        __syncthreads();
        for (int size = 2; size <= a.sort_n; size <<= 1) {
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                for (int i = tid; i < a.sort_n / 2; i += kTopkThreads) {
                    const int lo = 2 * i - (i & (stride - 1));
                    const int hi = lo + stride;
                    const uint64_t A = words[lo], B = words[hi];
                    if ((lo & size) == 0 ? A < B : A > B) {
                        words[lo] = B;
                        words[hi] = A;
                    }
                }
                __syncthreads();
            }
        }
        const float v0 = key_value<DI>((uint32_t)(words[0] >> 32));  // the largest value
        float z = 0.f;
        for (int t = tid; t < k; t += kTopkThreads) z += expf(key_value<DI>((uint32_t)(words[t] >> 32)) - v0);
        const float rz = __frcp_rn(block_sum_f(z, s_red));
        for (int t = tid; t < k; t += kTopkThreads)
            store(t, words[t], expf(key_value<DI>((uint32_t)(words[t] >> 32)) - v0) * rz);
    }
    pdl_trigger();
}

using TopkFn = void (*)(TopkArgs);

template <Dt DI>
TopkFn topk_fn(bool vec) {
    return vec ? topk_kernel<DI, Elem<DI>::kVec> : topk_kernel<DI, 1>;
}

cudaError_t prepare(TopkFn fn, int cs, size_t smem) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess && cs > 8)
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
}

}  // namespace

template <Dt DI>
cudaError_t launch_topk(const TopkArgs &a, bool vec, size_t smem, cudaStream_t st) {
    const TopkFn fn = topk_fn<DI>(vec);
    cudaError_t e = prepare(fn, a.cs, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.M * a.cs));
    cfg.blockDim = dim3(kTopkThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)a.cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = use_pdl() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, fn, a);
}

template <Dt DI>
cudaError_t topk_occupancy(bool vec, int cs, size_t smem, int *n) {
    *n = 0;
    const TopkFn fn = topk_fn<DI>(vec);
    cudaError_t e = prepare(fn, cs, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cs * 16u);
    cfg.blockDim = dim3(kTopkThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(n, fn, &cfg);
}

template cudaError_t launch_topk<Dt::F32>(const TopkArgs &, bool, size_t, cudaStream_t);
template cudaError_t launch_topk<Dt::BF16>(const TopkArgs &, bool, size_t, cudaStream_t);
template cudaError_t topk_occupancy<Dt::F32>(bool, int, size_t, int *);
template cudaError_t topk_occupancy<Dt::BF16>(bool, int, size_t, int *);

}  // namespace osr
