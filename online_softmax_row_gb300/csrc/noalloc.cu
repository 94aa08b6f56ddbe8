// noalloc.cu -- osr_softmax_rows_noalloc: the split-row softmax with its
// per-piece partials kept in a fixed, statically allocated device array
// instead of a workspace drawn from the stream-ordered allocator.
//
// Who needs it: callers that must not allocate device memory while they run
// -- serving loops that freeze their memory footprint after start-up, code on
// devices or drivers without stream-ordered memory pools
// (cudaDevAttrMemoryPoolsSupported == 0), and code running inside another
// allocator's callbacks, where calling back into an allocator can deadlock.
// This entry point calls no cudaMalloc*, cudaFree* or allocating library
// routine.
//
// The array below lives in the library's device image: every GPU that loads
// the library holds its OSR_NOALLOC_MAX_PARTIALS * 8 bytes until the process
// exits.  In host code its name is only a host-side stand-in, not a device
// address, so the host looks the real address up with cudaGetSymbolAddress
// once per device (with that device current) and passes it to the kernels.
#include <cuda_runtime.h>

#include <mutex>
#include <stdint.h>

#include "../../include/osr.h"
#include "launch.h"

namespace {

using osr::Dt;
using osr::Kind;
using osr::RowArgs;

// one (m, d) pair per (row, piece); 256-byte aligned like a cudaMalloc result
static __device__ __align__(256) float2 g_partials[OSR_NOALLOC_MAX_PARTIALS];

// CUDA failures are reported as OSR_ERR_CUDA; the error code is cleared
// from the runtime's per-thread state so later calls start clean.
osr_status fail(cudaError_t) {
    cudaGetLastError();
    return OSR_ERR_CUDA;
}

// Device address of g_partials on the current device, looked up once per
// device.  The first call on a device performs the lookup.
osr_status partials_address(float2 **out) {
    static std::mutex mu;
    static float2 *addr[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(e);
    if (dev < 0 || dev >= 64) return OSR_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_partials);
        if (e != cudaSuccess) return fail(e);
        addr[dev] = static_cast<float2 *>(p);
    }
    *out = addr[dev];
    return OSR_OK;
}

bool overlap(const void *a, int64_t an, const void *b, int64_t bn) {
    const char *pa = (const char *)a, *pb = (const char *)b;
    return pa < pb + bn && pb < pa + an;
}

// Memory the device reads and writes at the same address: device or managed
// memory, or page-locked host memory mapped into the unified address space
// (the kernels then reach it over the host link), as osr_softmax_rows takes.
bool on_device(const void *p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) return true;
    return at.type == cudaMemoryTypeHost && at.devicePointer == p;
}

cudaError_t launch_pass(osr_dtype in_dt, osr_dtype out_dt, Kind k, const RowArgs &a, bool vec,
                        int64_t grid, cudaStream_t st) {
    const int g = osr::kSplitThreads;
    if (in_dt == OSR_F32 && out_dt == OSR_F32)
        return osr::launch_softmax<Dt::F32, Dt::F32>(k, a, g, vec, grid, st);
    if (in_dt == OSR_F32 && out_dt == OSR_BF16)
        return osr::launch_softmax<Dt::F32, Dt::BF16>(k, a, g, vec, grid, st);
    if (in_dt == OSR_BF16 && out_dt == OSR_F32)
        return osr::launch_softmax<Dt::BF16, Dt::F32>(k, a, g, vec, grid, st);
    return osr::launch_softmax<Dt::BF16, Dt::BF16>(k, a, g, vec, grid, st);
}

}  // namespace

extern "C" osr_status osr_softmax_rows_noalloc(const void *x, void *y, int64_t M, int64_t N,
                                               osr_dtype in_dt, osr_dtype out_dt, void *stream) {
    if (M < 0 || N <= 0) return OSR_ERR_INVALID;
    if ((in_dt != OSR_F32 && in_dt != OSR_BF16) || (out_dt != OSR_F32 && out_dt != OSR_BF16))
        return OSR_ERR_INVALID;
    if (M == 0) return OSR_OK;
    if (!x || !y) return OSR_ERR_INVALID;
    // every row needs at least one (m, d) slot of the fixed array
    if (M > OSR_NOALLOC_MAX_PARTIALS || N > ((int64_t)1 << 40)) return OSR_ERR_UNSUPPORTED;
    const int in_b = in_dt == OSR_F32 ? 4 : 2, out_b = out_dt == OSR_F32 ? 4 : 2;
    const int64_t xb = M * N * in_b, yb = M * N * out_b;
    if (!(x == y && in_dt == out_dt) && overlap(x, xb, y, yb)) return OSR_ERR_ALIAS;
    if (!on_device(x) || !on_device(y)) return OSR_ERR_INVALID;

    float2 *partials = nullptr;
    osr_status s = partials_address(&partials);
    if (s != OSR_OK) return s;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(e);

    // shape of the split: pieces per row S and rows per (pass 1, pass 2)
    // batch b, as for the allocating split path, then S capped so that
    // M * S partials fit the fixed array
    const int vecn = in_dt == OSR_F32 ? 4 : 8;
    const bool vec = ((uintptr_t)x % 16 == 0) && ((uintptr_t)y % 16 == 0) && (N % vecn == 0);
    const int u = vec ? vecn : 1;
    const int64_t nunits = vec ? N / u : N;
    const int upt = osr::kEpt / u;  // the split softmax kernels' tile
    int64_t b = (48ll << 20) / (N * in_b);
    if (b < 1) b = 1;
    if (b > M) b = M;
    int64_t S = (2ll * sms + b - 1) / b;
    const int64_t most = (nunits + (int64_t)osr::kSplitThreads * upt - 1) /
                         ((int64_t)osr::kSplitThreads * upt);
    if (S > most) S = most;
    if (S > osr::kMaxPieces) S = osr::kMaxPieces;
    if (S > OSR_NOALLOC_MAX_PARTIALS / M) {
        // the array caps the pieces: take more rows per batch instead, so
        // that each launch still has about two CTAs per SM (their re-read in
        // pass 2 may then come partly from HBM rather than L2)
        S = OSR_NOALLOC_MAX_PARTIALS / M;
        if (S < 1) S = 1;
        const int64_t fill = (2ll * sms + S - 1) / S;
        if (b < fill) b = fill < M ? fill : M;
    }
    if (S > nunits) S = nunits;
    if (S < 1) S = 1;

    RowArgs a = {};
    a.x = x;
    a.y = y;
    a.M = M;
    a.N = N;
    a.cs = (int)S;
    a.chunk = (nunits + S - 1) / S;
    a.ws = partials;  // pass 1 writes every slot pass 2 reads: nothing to clear
    cudaStream_t st = (cudaStream_t)stream;
    for (int64_t r0 = 0; r0 < M; r0 += b) {
        const int64_t rows = M - r0 < b ? M - r0 : b;
        a.row0 = r0;
        e = launch_pass(in_dt, out_dt, Kind::SplitStats, a, vec, rows * S, st);
        if (e == cudaSuccess) e = launch_pass(in_dt, out_dt, Kind::SplitApply, a, vec, rows * S, st);
        if (e != cudaSuccess) return fail(e);
    }
    return OSR_OK;
}
