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
// One thread-block cluster of cs CTAs per row; CTA r caches elements
// [r * chunk, (r + 1) * chunk) of the row in shared memory as order-keys (so
// the row is read from HBM once) and all passes below run over that copy:
//   select  -- radix selection of the k-th largest key, 8 bits per pass from
//              the top (2 passes for bfloat16, 4 for binary32; the first runs
//              while the row is loaded): every CTA histograms the digit of its
//              elements whose higher digits equal the chosen prefix, the cs
//              histograms are summed through distributed shared memory, and
//              every CTA picks the same bin;
//   lse     -- the first pass also takes the row maximum m, the second the
//              sum d of e^(x - m); lse = m + log d;
//   gather  -- elements with key above the k-th largest key T are taken; of
//              those equal to T the lowest-indexed ones are taken (a prefix
//              over the cluster's CTAs; inside the one CTA whose share is
//              partial, an in-order scan), exactly k in all;
//   sort    -- CTA 0 pulls the k candidates of all CTAs, sorts them by (key
//              descending, index ascending) with a bitonic network and writes
//              values (re-read from the row), indices, probabilities and lse.
// The result is unique (a total order), so it is deterministic.
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

__device__ __forceinline__ uint32_t ld_dsmem_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ uint64_t ld_dsmem_u64(uint32_t addr) {
    uint64_t v;
    asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void cluster_sync_all() {
    cluster_arrive_release();
    cluster_wait_acquire();
}

// Inclusive sum over the CTA's threads in thread order; `scratch` holds
// kWarps values.  Ends with the CTA synchronised.
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
    __syncthreads();
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

__device__ __forceinline__ float block_sum_f(float v, float *scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = group_sum<32>(v);
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    v = group_sum<kWarps>(scratch[lane & (kWarps - 1)]);
    __syncthreads();
    return v;
}

__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, uint32_t *scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = __reduce_max_sync(0xffffffffu, v);
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    uint32_t r = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) r = scratch[w] > r ? scratch[w] : r;
    __syncthreads();
    return r;
}

// Keys of the elements of a 16-byte vector of raw values (8 bfloat16 or 4
// binary32), packed the same way.
template <Dt DI>
__device__ __forceinline__ uint4 keys_of(const uint4 &q) {
    if constexpr (DI == Dt::BF16) {
        auto k2 = [](uint32_t w) {
            return topk_key(w & 0xffffu, Dt::BF16) | (topk_key(w >> 16, Dt::BF16) << 16);
        };
        return make_uint4(k2(q.x), k2(q.y), k2(q.z), k2(q.w));
    } else {
        return make_uint4(topk_key(q.x, DI), topk_key(q.y, DI), topk_key(q.z, DI),
                          topk_key(q.w, DI));
    }
}

// Key e of a 16-byte vector of keys.
template <Dt DI>
__device__ __forceinline__ uint32_t key_at(const uint4 &q, int e) {
    if constexpr (DI == Dt::BF16) {
        const uint32_t w = e < 2 ? q.x : e < 4 ? q.y : e < 6 ? q.z : q.w;
        return (e & 1) ? w >> 16 : w & 0xffffu;
    } else {
        return e == 0 ? q.x : e == 1 ? q.y : e == 2 ? q.z : q.w;
    }
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

template <Dt DI, int U>
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const TopkArgs a) {
    using Key = typename std::conditional<DI == Dt::BF16, uint16_t, uint32_t>::type;
    constexpr int KB = DI == Dt::BF16 ? 16 : 32;  // key bits
    constexpr int PASSES = KB / 8;
    constexpr uint32_t kKeyInf = DI == Dt::BF16 ? 0xff80u : 0xff800000u;  // NaN keys lie above
    extern __shared__ __align__(16) unsigned char smem[];
    Key *keys = reinterpret_cast<Key *>(smem);              // the piece, as keys
    uint64_t *sortbuf = reinterpret_cast<uint64_t *>(smem);  // reuses the piece region
    uint32_t *hist_w = reinterpret_cast<uint32_t *>(smem + a.region0);
    uint32_t *hist_pub = hist_w + kWarps * 256;            // [2][256]
    uint64_t *cand = reinterpret_cast<uint64_t *>(hist_pub + 2 * 256);
    __shared__ float s_red[kWarps];
    __shared__ uint32_t s_scan[kWarps];
    __shared__ float pub_d;
    __shared__ uint32_t pub_kmax, pub_eq, pub_cand, s_bin, s_krem;

    const int tid = threadIdx.x, warp = tid >> 5;
    const int cs = a.cs;
    const uint32_t rank = cluster_ctarank();
    const int64_t row = blockIdx.x / cs;
    const int64_t e0 = (int64_t)rank * a.chunk;
    const int64_t e1 = e0 + a.chunk < a.N ? e0 + a.chunk : a.N;
    const int n = e1 > e0 ? (int)(e1 - e0) : 0;  // elements of this CTA's piece
    const Key *xrow = reinterpret_cast<const Key *>(a.x) + row * a.N;
    uint32_t *hw = hist_w + warp * 256;
    const uint32_t inv = 0xffffffffu;
    auto candidate = [&](uint32_t key, int i) {  // (key, column) -> sort word, kept
        const uint32_t pos = atomicAdd(&pub_cand, 1u);
        if (pos < (uint32_t)a.k)  // at most k by construction; never past the list
            cand[pos] = ((uint64_t)key << 32) | (uint64_t)(inv - (uint32_t)(e0 + i));
    };
    // every key of the piece, with its element index, in any order
    auto sweep = [&](auto &&f) {
        if constexpr (U > 1) {
            const uint4 *kv = reinterpret_cast<const uint4 *>(keys);
            for (int i = tid; i < n / U; i += kTopkThreads) {
                const uint4 q = kv[i];
#pragma unroll
                for (int e = 0; e < U; ++e) f(key_at<DI>(q, e), i * U + e);
            }
        } else {
            for (int i = tid; i < n; i += kTopkThreads) f((uint32_t)keys[i], i);
        }
    };

#pragma unroll
    for (int w = 0; w < kWarps; ++w) hist_w[w * 256 + tid] = 0u;
    if (tid == 0) pub_cand = 0;
    __syncthreads();
    pdl_wait();

    // ---- load: raw values -> keys in shared memory (the row is read from HBM
    //      once), with pass 0 on the way: the largest key of a number and the
    //      histogram of the top digit
    uint32_t kmax = 0;  // 0: no number seen
    auto visit0 = [&](uint32_t key) {
        if (key <= kKeyInf && key > kmax) kmax = key;
        atomicAdd(&hw[key >> (KB - 8)], 1u);
    };
    if constexpr (U > 1) {
        const uint4 *src = reinterpret_cast<const uint4 *>(xrow + e0);
        uint4 *dst = reinterpret_cast<uint4 *>(keys);
        const int nv = n / U;  // n is a multiple of U on the vector path
        for (int i0 = tid; i0 < nv; i0 += 4 * kTopkThreads) {
            uint4 q[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = i0 + j * kTopkThreads;
                q[j] = i < nv ? __ldcs(src + i) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = i0 + j * kTopkThreads;
                if (i < nv) {
                    const uint4 kq = keys_of<DI>(q[j]);
                    dst[i] = kq;
#pragma unroll
                    for (int e = 0; e < U; ++e) visit0(key_at<DI>(kq, e));
                }
            }
        }
    } else {
        for (int i = tid; i < n; i += kTopkThreads) {
            const uint32_t key = topk_key(xrow[e0 + i], DI);
            keys[i] = (Key)key;
            visit0(key);
        }
    }

    // ---- radix selection of the k-th largest key, with the row's m and d
    uint32_t prefix = 0;  // the chosen digits so far
    uint32_t krem = (uint32_t)a.k;
    float m = -FLT_MAX, d = 0.f;
#pragma unroll 1
    for (int p = 0; p < PASSES; ++p) {
        const int shift = KB - 8 * (p + 1);
        if (p == 0) {
            kmax = block_max_u32(kmax, s_scan);  // also orders the histogram atomics
            if (tid == 0) pub_kmax = kmax;
        } else {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) hist_w[w * 256 + tid] = 0u;
            __syncthreads();
            float acc = 0.f;
            sweep([&](uint32_t key, int) {
                if (p == 1) acc += exp_shifted(key_value<DI>(key), m);
                if ((key >> (shift + 8)) == prefix) atomicAdd(&hw[(key >> shift) & 255u], 1u);
            });
            if (p == 1) {
                acc = block_sum_f(acc, s_red);
                if (tid == 0) pub_d = acc;
            } else {
                __syncthreads();
            }
        }
        uint32_t h = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) h += hist_w[w * 256 + tid];
        uint32_t *pub = hist_pub + (p & 1) * 256;
        pub[tid] = h;
        cluster_sync_all();
        // the cluster's histogram and statistics, read in rank order
        uint32_t H = 0, km = 0;
        float ds = 0.f;
        for (int r = 0; r < cs; ++r) {
            H += ld_dsmem_u32(mapa_shared(smem_u32(pub + tid), r));
            if (p == 0) {
                const uint32_t o = ld_dsmem_u32(mapa_shared(smem_u32(&pub_kmax), r));
                km = o > km ? o : km;
            }
            if (p == 1) ds += ld_dsmem_f32(mapa_shared(smem_u32(&pub_d), r));
        }
        if (p == 0) m = km == 0 ? -FLT_MAX : fmaxf(key_value<DI>(km), -FLT_MAX);
        if (p == 1) d = ds;
        // S_b = elements in play with digit >= b, an inclusive scan in
        // descending digit order: thread t takes digit 255 - t.  (The
        // per-warp histograms are free again: the cluster barrier above
        // follows every thread's reads of them.)
        hist_w[255 - tid] = H;
        __syncthreads();
        const uint32_t Hr = hist_w[tid];
        const uint32_t S = block_inclusive_scan(Hr, s_scan);
        if (S >= krem && S - Hr < krem) {
            s_bin = 255u - (uint32_t)tid;
            s_krem = krem - (S - Hr);
        }
        __syncthreads();
        prefix = (prefix << 8) | s_bin;
        krem = s_krem;
        __syncthreads();
    }
    const uint32_t T = prefix;  // key of the k-th largest element
    // krem: how many elements equal to T are taken (the lowest-indexed ones)

    // ---- gather: every key above T; the count of keys equal to T
    uint32_t eqc = 0;
    sweep([&](uint32_t key, int i) {
        if (key > T) candidate(key, i);
        eqc += key == T;
    });
    eqc = block_inclusive_scan(eqc, s_scan);  // thread 255 holds the CTA's count
    if (tid == kTopkThreads - 1) pub_eq = eqc;
    cluster_sync_all();
    uint32_t eq_before = 0;
    for (int r = 0; r < (int)rank; ++r) eq_before += ld_dsmem_u32(mapa_shared(smem_u32(&pub_eq), r));
    const uint32_t eq_here = pub_eq;
    const uint32_t quota = krem > eq_before ? (krem - eq_before < eq_here ? krem - eq_before : eq_here) : 0u;
    if (quota == eq_here && quota > 0) {
        sweep([&](uint32_t key, int i) {
            if (key == T) candidate(key, i);
        });
    } else if (quota > 0) {
        // a partial share (one CTA of the row at most): the lowest-indexed
        // equal keys.  Each thread walks a contiguous range of the piece, so
        // index order is (thread, position): count, scan, take in order.
        const int L = (n + kTopkThreads - 1) / kTopkThreads;
        const int j0 = tid * L, j1 = j0 + L < n ? j0 + L : n;
        uint32_t c = 0;
        for (int j = j0; j < j1; ++j) c += (uint32_t)keys[j] == T;
        const uint32_t incl = block_inclusive_scan(c, s_scan);
        uint32_t r = incl - c;  // equal keys before this thread's range
        for (int j = j0; j < j1 && r < quota; ++j)
            if ((uint32_t)keys[j] == T) {
                candidate(T, j);
                ++r;
            }
    }
    cluster_sync_all();  // every CTA's candidates are complete

    if (rank == 0) {
        // pull the k candidates (rank order), pad the network with zero words
        // (below every real key), then sort descending
        uint32_t off = 0;
        for (int r = 0; r < cs; ++r) {
            const uint32_t cnt = ld_dsmem_u32(mapa_shared(smem_u32(&pub_cand), r));
            const uint32_t src = mapa_shared(smem_u32(cand), r);
            for (uint32_t i = tid; i < cnt && off + i < (uint32_t)a.sort_n; i += kTopkThreads)
                sortbuf[off + i] = ld_dsmem_u64(src + i * 8);
            off += cnt;
        }
        for (int i = (int)a.k + tid; i < a.sort_n; i += kTopkThreads) sortbuf[i] = 0ull;
    }
    cluster_sync_all();  // no CTA leaves while CTA 0 reads its candidates
    if (rank != 0) {
        pdl_trigger();
        return;
    }
    __syncthreads();
    for (int size = 2; size <= a.sort_n; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = tid; i < a.sort_n / 2; i += kTopkThreads) {
                const int lo = 2 * i - (i & (stride - 1));
                const int hi = lo + stride;
                const uint64_t A = sortbuf[lo], B = sortbuf[hi];
                const bool desc = (lo & size) == 0;
                if (desc ? A < B : A > B) {
                    sortbuf[lo] = B;
                    sortbuf[hi] = A;
                }
            }
            __syncthreads();
        }
    }

    // ---- outputs: values re-read from the row (L2), indices, softmax of the
    //      k values (largest first, so v0 is their maximum), lse.  (An index
    //      outside the row can only come from a selection that did not find k
    //      candidates: it is reported as -1 with a NaN value, never read.)
    const int64_t k = a.k;
    auto value_at = [&](uint32_t j) {
        return j < (uint32_t)a.N ? raw_to_f32(xrow[j], DI) : __uint_as_float(0x7fc00000u);
    };
    const float v0 = value_at(inv - (uint32_t)sortbuf[0]);
    float zsum = 0.f;
    for (int t = tid; t < k; t += kTopkThreads) {
        const uint32_t j = inv - (uint32_t)sortbuf[t];
        const float v = value_at(j);
        a.values[row * k + t] = v;
        a.indices[row * k + t] = j < (uint32_t)a.N ? (int64_t)j : -1;
        zsum += expf(v - v0);
    }
    if (a.probs != nullptr) {
        zsum = block_sum_f(zsum, s_red);
        for (int t = tid; t < k; t += kTopkThreads)
            a.probs[row * k + t] = expf(value_at(inv - (uint32_t)sortbuf[t]) - v0) / zsum;
    }
    if (a.lse != nullptr && tid == 0) a.lse[row] = m + logf(d);
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
