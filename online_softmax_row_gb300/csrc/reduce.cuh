// reduce.cuh -- reductions of a row's partial results across the threads,
// warps and cluster CTAs that share the row, with every participant ending
// up holding the identical (bit-for-bit) result.
//
// Two monoids:
//   sum of squares (RMSNorm), identity 0;
//   the online-softmax normaliser state (m, d) with the merge
//     (m1, d1) (+) (m2, d2) = (max(m1, m2), d1 e^(m1 - m) + d2 e^(m2 - m)),
//   identity (-inf, 0) -- represented as (-FLT_MAX, 0) so that merging two
//   empty states never evaluates (-inf) - (-inf).
// Merge and identity: "两个融合算子：RMSNorm 与 online softmax"
// (daleiyang.github.io), §5·三 "结合律：为什么能做树形归约" (associativity,
// identity, the -FLT_MAX substitute) and §3·三 "联合归约：把 (m, s) 当成一个整体";
// "RMSNorm、Softmax 与在线归约" (notes.kuangjux.top), "从逐元素更新到合并两个 tile".
//
// Every exchange is an xor butterfly.  Because each merge below is exactly
// commutative in floating point (a + b == b + a; the (m, d) merge picks the
// larger m and scales the other side), the two partners of every butterfly
// step compute the same value, so after the last step all lanes agree bit
// for bit.  Block and cluster stages have every warp redo the final
// butterfly on the same inputs, so all warps (and all CTAs) agree too.
#pragma once

#include "device_common.cuh"

namespace osr {

struct MD {
    float m, d;
};

__device__ __forceinline__ MD md_identity() { return {-FLT_MAX, 0.f}; }

// One exp per merge: the side with the larger m is scaled by e^0 = 1.
__device__ __forceinline__ MD md_merge(MD a, MD b) {
    if (a.m < b.m) {
        const MD t = a;
        a = b;
        b = t;
    }
    return {a.m, fmaf(b.d, expf(b.m - a.m), a.d)};
}

// ---------------------------------------------------------------- in a group
// W lanes (a power of two, aligned within the warp) hold one row's partials.

template <int W>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
    for (int off = W / 2; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

template <int W>
__device__ __forceinline__ MD group_md(MD s) {
#pragma unroll
    for (int off = W / 2; off > 0; off >>= 1) {
        MD o;
        o.m = __shfl_xor_sync(0xffffffffu, s.m, off);
        o.d = __shfl_xor_sync(0xffffffffu, s.d, off);
        s = md_merge(s, o);
    }
    return s;
}

// ---------------------------------------------------------------- in a CTA
// NW warps share one row.  Stage 1: butterfly inside each warp.  Stage 2:
// each warp's lane 0 parks its result in shared memory; after one barrier
// every warp reads all NW results and runs the same butterfly over them.
// `red` is a 32-entry shared array used once per kernel.

template <int NW>
__device__ __forceinline__ float block_sum(float v, float *red) {
    v = group_sum<32>(v);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if constexpr (NW == 1) return v;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    return group_sum<NW>(red[lane & (NW - 1)]);
}

template <int NW>
__device__ __forceinline__ MD block_md(MD s, float2 *red) {
    s = group_md<32>(s);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if constexpr (NW == 1) return s;
    if (lane == 0) red[warp] = make_float2(s.m, s.d);
    __syncthreads();
    const float2 r = red[lane & (NW - 1)];
    return group_md<NW>(MD{r.x, r.y});
}

// ---------------------------------------------------------------- in a cluster
// cs CTAs (cs <= 32) share one row.  Each CTA publishes its CTA-level result
// in its own shared memory, the cluster barrier makes it visible, and every
// warp of every CTA gathers the cs results through distributed shared memory
// (lane r reads CTA r) and runs the same 32-lane butterfly on them.  The
// relaxed arrive that follows marks "done reading peers"; the caller must
// execute cluster_wait_acquire() once before it exits so that no CTA leaves
// while a peer may still read its shared memory.

__device__ __forceinline__ MD cluster_md(MD s, int cs, float2 *slot) {
    if (threadIdx.x == 0) *slot = make_float2(s.m, s.d);
    cluster_arrive_release();
    cluster_wait_acquire();
    const int lane = threadIdx.x & 31;
    MD q = md_identity();
    if (lane < cs) {
        const float2 r = ld_dsmem_f2(mapa_shared(smem_u32(slot), lane));
        q = MD{r.x, r.y};
    }
    q = group_md<32>(q);
    cluster_arrive_relaxed();
    return q;
}

__device__ __forceinline__ float cluster_sum(float s, int cs, float2 *slot) {
    if (threadIdx.x == 0) *slot = make_float2(s, 0.f);
    cluster_arrive_release();
    cluster_wait_acquire();
    const int lane = threadIdx.x & 31;
    float q = 0.f;
    if (lane < cs) q = ld_dsmem_f2(mapa_shared(smem_u32(slot), lane)).x;
    q = group_sum<32>(q);
    cluster_arrive_relaxed();
    return q;
}

}  // namespace osr
