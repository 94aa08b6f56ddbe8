// row_common.cuh -- arguments and geometry shared by the row kernels.
//
// Register-cached tiers: each row (or, in the cluster tier, each piece of a
// row) is read from HBM exactly once into registers, reduced, rescaled in
// registers and written exactly once.
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

// ============================================================ split-row tier
// Split-row tier for rows of any length: a row is cut into S pieces handled
// by S independent CTAs.
//   pass 1: each CTA streams its piece and writes one partial state to the
//           workspace ws[row][piece] -- (m, d) for softmax, the sum of
//           squares for the norms (the fused norm also writes the new
//           residual here);
//   pass 2: each CTA merges the S partials of its row in a fixed order (so
//           every piece of a row sees bit-identical statistics and repeated
//           runs are bit-identical), then streams its piece again and writes
//           the output.
// "Softmax 与归一化" (anrans.github.io), table "按行长度选择并行方式" (the
// "very long rows, few rows: several blocks per row, partial (m, d) then
// merge" row) and "第23讲：为什么Attention必须先算Max？" (lilinji.mintlify.site)
// §8.3 thought question 1 (rows beyond 65536).  The host keeps the second read
// in L2 by issuing the two passes over batches of rows whose pieces fit L2.
template <int G>
struct SplitGeom {
    static constexpr int kThreads = G;
    static constexpr int kWarps = G / 32;
};

// CTA (row, piece) of a split launch; rows are a.row0 + blockIdx.x / S.
struct Piece {
    int64_t row;
    int p;
    int64_t u0, u1;
};

__device__ __forceinline__ Piece make_piece(const RowArgs &a, int64_t nunits) {
    Piece q;
    q.row = a.row0 + blockIdx.x / a.cs;
    q.p = blockIdx.x % a.cs;
    q.u0 = (int64_t)q.p * a.chunk;
    q.u1 = q.u0 + a.chunk < nunits ? q.u0 + a.chunk : nunits;
    return q;
}

}  // namespace osr
