// device_common.cuh -- storage types, 16-byte vector I/O and cluster /
// distributed-shared-memory primitives for sm_103a.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <float.h>
#include <stdint.h>

namespace osr {

enum class Dt : int { F32 = 0, BF16 = 1 };

template <Dt D>
struct Elem;
template <>
struct Elem<Dt::F32> {
    static constexpr int kBytes = 4;
    static constexpr int kVec = 4;  // elements per 16-byte vector
};
template <>
struct Elem<Dt::BF16> {
    static constexpr int kBytes = 2;
    static constexpr int kVec = 8;
};

// ---------------------------------------------------------------- conversions

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// two floats -> two bfloat16 (round to nearest even), lo in the low half
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&b);
}

__device__ __forceinline__ float round_bf16(float v) {
    return __bfloat162float(__float2bfloat16_rn(v));
}

template <Dt D>
__device__ __forceinline__ float round_to(float v) {
    if constexpr (D == Dt::BF16) return round_bf16(v);
    return v;
}

// ---------------------------------------------------------------- exp
// e^(x - m) for x <= m, as 2^((x - m) log2 e) on the special-function unit
// (PTX ex2.approx.ftz.f32: about 2 ulp; -inf -> 0; results below the normal
// range flush to 0).  The difference is formed before scaling, so the only
// extra error is the rounding of the product, |x - m| log2 e 2^-24 in the
// exponent: 5e-6 relative at x - m = -80.
__device__ __forceinline__ float ex2_approx(float t) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(t));
    return r;
}
__device__ __forceinline__ float exp_shifted(float x, float m) {
    return ex2_approx((x - m) * 1.4426950408889634f);
}

// ---------------------------------------------------------------- packed bf16
// Eight bfloat16 values in a 16-byte vector, element k in half (k & 1) of
// word k / 2.  Widening is exact; packing rounds to nearest even.
__device__ __forceinline__ void unpack8(const uint4 &q, float (&f)[8]) {
    f[0] = bf16_lo(q.x); f[1] = bf16_hi(q.x);
    f[2] = bf16_lo(q.y); f[3] = bf16_hi(q.y);
    f[4] = bf16_lo(q.z); f[5] = bf16_hi(q.z);
    f[6] = bf16_lo(q.w); f[7] = bf16_hi(q.w);
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    uint4 q;
    q.x = pack_bf16x2(f[0], f[1]);
    q.y = pack_bf16x2(f[2], f[3]);
    q.z = pack_bf16x2(f[4], f[5]);
    q.w = pack_bf16x2(f[6], f[7]);
    return q;
}

// ---------------------------------------------------------------- f32x2
// Two binary32 lanes in one 64-bit register pair, for the packed arithmetic
// of sm_100-family SMs (PTX add / sub / mul / fma .rn.f32x2).  Each lane is
// rounded exactly as the scalar instruction rounds it, so a lane's result is
// unchanged; one instruction does the work of two.
__device__ __forceinline__ uint64_t f2_make(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
// lane 0 is the low word of the pair, lane 1 the high word
__device__ __forceinline__ float f2_lo(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float f2_hi(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
// bfloat16 pair (element 2k in the low half) <-> binary32 pair
__device__ __forceinline__ uint64_t f2_from_bf16x2(uint32_t w) {
    return f2_make(bf16_lo(w), bf16_hi(w));
}
__device__ __forceinline__ uint32_t bf16x2_from_f2(uint64_t v) {
    return pack_bf16x2(f2_lo(v), f2_hi(v));
}
// pair k (elements 2k, 2k+1) of a 16-byte vector of dtype D: four bfloat16
// pairs or two binary32 pairs
template <Dt D>
__device__ __forceinline__ uint64_t f2_of(const uint4 &q, int k) {
    if constexpr (D == Dt::BF16)
        return f2_from_bf16x2(k == 0 ? q.x : k == 1 ? q.y : k == 2 ? q.z : q.w);
    else
        return k == 0 ? f2_make(__uint_as_float(q.x), __uint_as_float(q.y))
                      : f2_make(__uint_as_float(q.z), __uint_as_float(q.w));
}

// ---------------------------------------------------------------- loads
// A "unit" is U consecutive elements: one 16-byte vector (U = kVec) or one
// scalar (U = 1).  `e` is the element offset of the unit from `base`.
// Streaming inputs are read with the evict-first (.cs) hint: each byte is
// read once, so it should not push reusable lines out of L2.

// Stream   : read once (ld.global.cs, evict-first);
// Keep     : default caching, for data read again soon (split-row pass 1);
// ReadOnly : never written during the kernel and shared by many CTAs
//            (gamma), through the non-coherent read-only path.
enum class Hint : int { Stream = 0, Keep = 1, ReadOnly = 2 };

template <Hint H>
__device__ __forceinline__ uint4 ld16(const void *p) {
    if constexpr (H == Hint::Stream)
        return __ldcs(reinterpret_cast<const uint4 *>(p));
    else if constexpr (H == Hint::ReadOnly)
        return __ldg(reinterpret_cast<const uint4 *>(p));
    else
        return *reinterpret_cast<const uint4 *>(p);
}

template <Dt D, int U, Hint H = Hint::Stream>
__device__ __forceinline__ void load_unit(const void *base, int64_t e, float (&v)[U]) {
    if constexpr (U == 1) {
        if constexpr (D == Dt::F32) {
            v[0] = reinterpret_cast<const float *>(base)[e];
        } else {
            const uint16_t b = reinterpret_cast<const uint16_t *>(base)[e];
            v[0] = __uint_as_float(uint32_t(b) << 16);
        }
    } else {
        static_assert(U == Elem<D>::kVec, "a vector unit is 16 bytes");
        const uint4 q = ld16<H>(reinterpret_cast<const char *>(base) + e * Elem<D>::kBytes);
        if constexpr (D == Dt::F32) {
            v[0] = __uint_as_float(q.x);
            v[1] = __uint_as_float(q.y);
            v[2] = __uint_as_float(q.z);
            v[3] = __uint_as_float(q.w);
        } else {
            v[0] = bf16_lo(q.x); v[1] = bf16_hi(q.x);
            v[2] = bf16_lo(q.y); v[3] = bf16_hi(q.y);
            v[4] = bf16_lo(q.z); v[5] = bf16_hi(q.z);
            v[6] = bf16_lo(q.w); v[7] = bf16_hi(q.w);
        }
    }
}

// ---------------------------------------------------------------- stores
// U elements of dtype D from binary32 values, rounded to nearest even.
// U = 1: one scalar; U = 4 or 8: 8..32 bytes as 16-byte (or, for 4 bfloat16,
// 8-byte) vector stores.  Outputs are written with the streaming (.cs) hint.

template <Dt D, int U>
__device__ __forceinline__ void store_unit(void *base, int64_t e, const float (&v)[U]) {
    if constexpr (U == 1) {
        if constexpr (D == Dt::F32)
            reinterpret_cast<float *>(base)[e] = v[0];
        else
            reinterpret_cast<__nv_bfloat16 *>(base)[e] = __float2bfloat16_rn(v[0]);
    } else if constexpr (D == Dt::F32) {
        static_assert(U % 4 == 0, "f32 vector stores cover 4 elements");
        float4 *p = reinterpret_cast<float4 *>(reinterpret_cast<float *>(base) + e);
#pragma unroll
        for (int k = 0; k < U / 4; ++k)
            __stcs(p + k, make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]));
    } else {
        static_assert(U == 4 || U == 8, "bf16 vector stores cover 4 or 8 elements");
        char *p = reinterpret_cast<char *>(base) + e * 2;
        if constexpr (U == 8) {
            uint4 q;
            q.x = pack_bf16x2(v[0], v[1]);
            q.y = pack_bf16x2(v[2], v[3]);
            q.z = pack_bf16x2(v[4], v[5]);
            q.w = pack_bf16x2(v[6], v[7]);
            __stcs(reinterpret_cast<uint4 *>(p), q);
        } else {
            uint2 q;
            q.x = pack_bf16x2(v[0], v[1]);
            q.y = pack_bf16x2(v[2], v[3]);
            __stcs(reinterpret_cast<uint2 *>(p), q);
        }
    }
}

// ---------------------------------------------------------------- dependent launch
// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start while the previous kernel in the stream drains;
// griddepcontrol.wait blocks until that kernel has completed and its writes
// are visible, so every kernel here calls it before its first global access
// (without the launch attribute it returns at once).  launch_dependents,
// issued after a CTA's last store, lets the next kernel start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- clusters
// Thread-block cluster barrier (split arrive / wait) and distributed shared
// memory access, as PTX.  Every thread of every CTA of the cluster executes
// each arrive and each wait exactly once per phase (.aligned).

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// address of the same shared variable in CTA `rank` of this cluster
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ float2 ld_dsmem_f2(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];"
                 : "=f"(v.x), "=f"(v.y)
                 : "r"(addr)
                 : "memory");
    return v;
}

// Asynchronous store of two floats into shared memory of a CTA of the
// cluster (addresses from mapa_shared), completing `8` bytes on that CTA's
// mbarrier, which the receiver waits on: no cluster barrier orders it.
__device__ __forceinline__ void st_async_f2(uint32_t addr, uint32_t remote_bar, float x, float y) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(addr),
                 "f"(x), "f"(y), "r"(remote_bar)
                 : "memory");
}

// The same for four 32-bit words (16 bytes, 16-byte aligned addresses).
__device__ __forceinline__ void st_async_v4(uint32_t addr, uint32_t remote_bar, uint4 v) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(addr),
                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(remote_bar)
                 : "memory");
}

// The same for one 64-bit word (8-byte aligned address).
__device__ __forceinline__ void st_async_u64(uint32_t addr, uint32_t remote_bar, uint64_t v) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b64 [%0], %1, [%2];" ::"r"(addr), "l"(v),
                 "r"(remote_bar)
                 : "memory");
}

// ---------------------------------------------------------------- bulk copies
// 1-D bulk asynchronous copies (the TMA engine, no tensor map) from global
// into this CTA's shared memory, completed through an mbarrier's
// transaction count.  Addresses and sizes are multiples of 16 bytes.

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
// make the initialised barrier visible to the async (TMA) proxy
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// one arrival that also announces `bytes` of incoming transactions
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_load_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                              uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}
// same copy with an L2 eviction-priority policy (createpolicy) attached
__device__ __forceinline__ void bulk_load_g2s_hint(uint32_t dst, const void *src, uint32_t bytes,
                                                   uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}
// L2 policy: lines fetched under it are the first to be evicted
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Wait for phase `parity` of the barrier, giving up after `limit_ns`
// nanoseconds; returns whether the phase completed.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > limit_ns) return false;
    return true;
}

}  // namespace osr
