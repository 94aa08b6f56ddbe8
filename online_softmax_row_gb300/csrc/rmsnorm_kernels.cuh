// rmsnorm_kernels.cuh -- RMSNorm and fused residual-add + RMSNorm kernels: the
// register-cached row/cluster kernel and the two split-row passes.
#pragma once

#include "row_common.cuh"

namespace osr {

// ============================================================ RMSNorm
// y = x * rsqrt(mean(x^2) + eps) * gamma; with FUSED, x + residual is first
// rounded to the storage type, written back to the residual, and the
// rounded sum is what gets normalised ("GPU Kernel 工程（04）" 八.3 "fused
// residual + RMSNorm"; the stored value is normalised so that the output
// equals RMSNorm of the new residual).
// bfloat16 rows on the 16-byte path stay packed in registers (4 registers
// per 8 elements) and are widened when used, which halves the cache's
// register footprint and raises occupancy.
//
// The packed bf16 fused kernel of 256 threads (rows of 2-4 Ki elements, the
// default for them) is held to 32 registers, eight CTAs an SM instead of six,
// by reading gamma after the reduction instead of before it.  Measured: 8192
// x 4096 40.19 -> 40.09 us, 16384 x 3584 69.5 -> 68.8, 2048 x 4096 12.04 ->
// 11.43, 1024 x 4096 7.25 -> 6.20; reading gamma late without the bound
// gained nothing.  Every other instantiation keeps its unbounded allocation
// (a minimum of 0 CTAs is the same as none; 1 would change them).
template <Dt D, int G, int EPT, int U, bool CLUSTER, bool FUSED>
__global__ void __launch_bounds__(RowsGeom<G>::kThreads, (FUSED && D == Dt::BF16 && G == 256 && !CLUSTER && U == 8) ? 8 : 0)
rmsnorm_rows_kernel(const RowArgs a) {
    constexpr bool kPacked = D == Dt::BF16 && U == 8;
    constexpr bool kLateGamma = FUSED && D == Dt::BF16 && G == 256 && !CLUSTER && U == 8;
    constexpr int NU = EPT / U;
    constexpr int NP = kPacked ? NU : 1;  // packed vectors held
    constexpr int NF = kPacked ? 1 : NU;  // fp32 units held
    const int64_t nunits = a.N / U;
    const Slice s = make_slice<G, CLUSTER>(a, nunits);
    const int64_t row_off = s.row * a.N * Elem<D>::kBytes;
    const char *xrow = reinterpret_cast<const char *>(a.x) + row_off;
    if constexpr (CLUSTER) cluster_push_init(cluster_push_area<0>(), nullptr, a.cs);
    pdl_wait();

    // The residual stores come after every load of the thread's units: the
    // pointers are not known to be distinct, so a load placed after a store
    // could not be moved ahead of it, and each unit would cost its own memory
    // round trip.
    char *rrow = reinterpret_cast<char *>(a.res) + row_off;
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
                    const uint4 rq = ld16<Hint::Stream>(rrow + ui * 16);
                    float xf[8], rf[8];
                    unpack8(pk[j], xf);
                    unpack8(rq, rf);
#pragma unroll
                    for (int k = 0; k < 8; ++k) xf[k] += rf[k];
                    pk[j] = pack8(xf);
                }
            }
        } else {
            if (in) {
                load_unit<D, U>(xrow, ui * U, v[j]);
                if constexpr (FUSED) {
                    float r[U];
                    load_unit<D, U>(rrow, ui * U, r);
#pragma unroll
                    for (int k = 0; k < U; ++k) v[j][k] = round_to<D>(v[j][k] + r[k]);
                }
            } else {
#pragma unroll
                for (int k = 0; k < U; ++k) v[j][k] = 0.f;
            }
        }
    }
    if constexpr (FUSED) {
#pragma unroll
        for (int j = 0; j < NU; ++j) {
            const int64_t ui = s.u0 + (int64_t)j * G + s.t;
            if (s.ok && ui < s.u1) {
                if constexpr (kPacked)
                    __stcs(reinterpret_cast<uint4 *>(rrow + ui * 16), pk[j]);
                else
                    store_unit<D, U>(rrow, ui * U, v[j]);
            }
        }
    }

    // gamma is shared by every row: read-only path, fetched before the
    // reduction so its latency overlaps it (after it where registers are
    // held to 32, see above)
    auto load_gamma = [&]() {
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
    };
    if constexpr (!kLateGamma) load_gamma();

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
    if constexpr (CLUSTER) ss = cluster_sum(ss, a.cs, cluster_push_area<0>(), true);
    const float r = rsqrtf(ss / (float)a.N + a.eps);
    if constexpr (kLateGamma) load_gamma();

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
}

// ------------------------------------------------------------ RMSNorm pass 1
template <Dt D, int G, int EPT, int U, bool FUSED>
__global__ void __launch_bounds__(G) rmsnorm_split_stats_kernel(const RowArgs a) {
    constexpr int NU = EPT / U;
    const int64_t nunits = a.N / U;
    const Piece q = make_piece(a, nunits);
    const int64_t row_off = q.row * a.N * Elem<D>::kBytes;
    const char *xrow = reinterpret_cast<const char *>(a.x) + row_off;
    pdl_wait();
    float ss = 0.f;
    for (int64_t base = q.u0; base < q.u1; base += (int64_t)G * NU) {
        float v[NU][U];
#pragma unroll
        for (int j = 0; j < NU; ++j) {
            const int64_t ui = base + (int64_t)j * G + threadIdx.x;
            if (ui < q.u1) {
                if constexpr (FUSED) {
                    char *rrow = reinterpret_cast<char *>(a.res) + row_off;
                    float r[U];
                    load_unit<D, U>(xrow, ui * U, v[j]);
                    load_unit<D, U>(rrow, ui * U, r);
#pragma unroll
                    for (int k = 0; k < U; ++k) v[j][k] = round_to<D>(v[j][k] + r[k]);
                    store_unit<D, U>(rrow, ui * U, v[j]);
                } else {
                    load_unit<D, U, Hint::Keep>(xrow, ui * U, v[j]);
                }
            } else {
#pragma unroll
                for (int k = 0; k < U; ++k) v[j][k] = 0.f;
            }
        }
#pragma unroll
        for (int j = 0; j < NU; ++j)
#pragma unroll
            for (int k = 0; k < U; ++k) ss = fmaf(v[j][k], v[j][k], ss);
    }
    __shared__ float red[32];
    ss = block_sum<SplitGeom<G>::kWarps>(ss, red);
    if (threadIdx.x == 0) reinterpret_cast<float *>(a.ws)[q.row * a.cs + q.p] = ss;
    pdl_trigger();
}

// ------------------------------------------------------------ RMSNorm pass 2
// Reads x (or, fused, the new residual written by pass 1) again.
template <Dt D, int G, int EPT, int U, bool FUSED>
__global__ void __launch_bounds__(G) rmsnorm_split_apply_kernel(const RowArgs a) {
    constexpr int NU = EPT / U;
    const int64_t nunits = a.N / U;
    const Piece q = make_piece(a, nunits);
    pdl_wait();
    float ss = 0.f;
    if (threadIdx.x < a.cs) ss = reinterpret_cast<const float *>(a.ws)[q.row * a.cs + threadIdx.x];
    __shared__ float red[32];
    ss = block_sum<SplitGeom<G>::kWarps>(ss, red);
    const float r = rsqrtf(ss / (float)a.N + a.eps);
    const int64_t row_off = q.row * a.N * Elem<D>::kBytes;
    const char *src = reinterpret_cast<const char *>(FUSED ? a.res : a.x) + row_off;
    char *yrow = reinterpret_cast<char *>(a.y) + row_off;
    for (int64_t base = q.u0; base < q.u1; base += (int64_t)G * NU) {
        float v[NU][U], g[NU][U];
#pragma unroll
        for (int j = 0; j < NU; ++j) {
            const int64_t ui = base + (int64_t)j * G + threadIdx.x;
            if (ui < q.u1) {
                load_unit<D, U>(src, ui * U, v[j]);
                load_unit<D, U, Hint::ReadOnly>(a.gamma, ui * U, g[j]);
            }
        }
#pragma unroll
        for (int j = 0; j < NU; ++j) {
            const int64_t ui = base + (int64_t)j * G + threadIdx.x;
            if (ui < q.u1) {
                float o[U];
#pragma unroll
                for (int k = 0; k < U; ++k) o[k] = v[j][k] * r * g[j][k];
                store_unit<D, U>(yrow, ui * U, o);
            }
        }
    }
    pdl_trigger();
}

}  // namespace osr
