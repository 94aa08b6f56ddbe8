// dispatch.cu -- the C ABI (include/osr.h): argument validation, the
// length-based dispatcher, and execution of a plan on the caller's stream.
//
// Dispatch follows the row-length table of "Softmax 与归一化"
// (anrans.github.io), "按行长度选择并行方式": short rows -> several rows per
// warp; up to about a thousand elements -> one warp per row; thousands ->
// one block per row; rows longer than one block's registers -> several
// blocks per row.  Here the last step has two forms: a thread-block cluster
// whose CTAs exchange their partial statistics through distributed shared
// memory (row still read once), and, beyond what a cluster can hold, two
// passes through a small global workspace.
#include <cuda_runtime.h>

#include <atomic>
#include <map>
#include <mutex>
#include <stdio.h>
#include <tuple>
#include <stdlib.h>
#include <string.h>

#include "../../include/osr.h"
#include "../../include/osr_test.h"
#include "launch.h"
#include "lse.h"
#include "staged.h"
#include "topk.h"

namespace osr {
namespace {

thread_local int g_last_cuda_error = 0;

// osr_test_set_flags (include/osr_test.h): read once per staged launch
std::atomic<int> g_test_flags{0};

// osr_test_force_kernel (include/osr_test.h): a forced plan for tests,
// copied under a lock; the planners read it only while one is set
std::atomic<bool> g_force_set{false};
std::mutex g_force_mu;
char g_force[64] = "";

struct ForceSpec {
    char s[64];
    const char *get() const { return s[0] ? s : nullptr; }
};
ForceSpec forced_spec() {
    ForceSpec f;
    f.s[0] = 0;
    if (g_force_set.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(g_force_mu);
        memcpy(f.s, g_force, sizeof f.s);
    }
    return f;
}

osr_status cuda_fail(cudaError_t e) {
    g_last_cuda_error = (int)e;
    return OSR_ERR_CUDA;
}

constexpr int kL2BudgetBytes = 48 << 20;  // re-read set of one split batch

int elem_bytes(osr_dtype d) { return d == OSR_F32 ? 4 : 2; }
int vec_elems(osr_dtype d) { return d == OSR_F32 ? 4 : 8; }
bool dtype_ok(osr_dtype d) { return d == OSR_F32 || d == OSR_BF16; }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// elements per thread per tile of an operation's row kernels
int ept_of(Op op, osr_dtype dt, bool vec) {
    if (dt != OSR_BF16 || !vec) return kEpt;
    if (op == Op::Softmax) return softmax_ept<Dt::BF16, 8>();
    return op == Op::FusedAddRmsNorm ? norm_ept<Dt::BF16, 8, true>() : norm_ept<Dt::BF16, 8>();
}
int pow2ceil(int64_t v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

// ------------------------------------------------------------ device facts
// shared memory of an sm_100-family SM (1 KiB of it is reserved per CTA):
// the planners' default where no device is queried (osr_plan_describe)
constexpr int kSmemPerSmDefault = 228 << 10;

struct DeviceInfo {
    int sms = 0;
    int max_cluster = 8;
    int smem_per_sm = kSmemPerSmDefault;
};

osr_status device_info(DeviceInfo *out) {
    static std::mutex mu;
    static DeviceInfo cache[64];
    static bool have[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= 64) return OSR_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(mu);
    if (!have[dev]) {
        DeviceInfo d;
        int major = 0, cluster = 0;
        if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e);
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
            return cuda_fail(e);
        if ((e = cudaDeviceGetAttribute(&cluster, cudaDevAttrClusterLaunch, dev)) != cudaSuccess)
            return cuda_fail(e);
        if ((e = cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) !=
            cudaSuccess)
            return cuda_fail(e);
        d.max_cluster = cluster ? (major >= 10 ? 16 : 8) : 1;
        cache[dev] = d;
        have[dev] = true;
    }
    *out = cache[dev];
    return OSR_OK;
}

// ------------------------------------------------------------ planning
// Units: a unit is one 16-byte input vector on the vector path, else one
// element; each thread holds kEpt elements (kEpt / u units) per tile.

// Value of `key` in "tier:key=v,key=v"; keys match whole tokens only.
bool parse_kv(const char *s, const char *key, int64_t *v) {
    const size_t n = strlen(key);
    for (const char *p = strchr(s, ':'); p && *p; p = strchr(p + 1, ',')) {
        const char *k = p + 1;
        if (strncmp(k, key, n) == 0 && k[n] == '=') {
            char *end = nullptr;
            long long x = strtoll(k + n + 1, &end, 10);
            if (end == k + n + 1) return false;
            *v = x;
            return true;
        }
    }
    return false;
}

int64_t pow2_at_least(int64_t v) {
    int64_t c = 1;
    while (c < v) c <<= 1;
    return c;
}

// Whether the staged tier holds part of each piece in registers by default:
// fp32 input.  Measured over 16 shapes (fp32 rows of 24 Ki to 148 Ki
// elements, bfloat16 rows of 20 Ki to 148 Ki, 1 to 8192 rows): with
// registers fp32 rows ran up to 9 % faster (64 x 152064: 17.7 -> 16.2 us),
// bfloat16 rows 1-20 % slower.
bool staged_regs(osr_dtype in_dt, osr_dtype out_dt) {
    (void)out_dt;
    return in_dt == OSR_F32;
}

// Staged tier shape.
//
// regs: each thread holds kStagedRegUnits units in registers and the rest of
// its piece is staged.  The fewest pieces of at most 76 KiB (about half in
// registers, so four CTAs fit an SM); with fewer CTAs than SMs, 12 pieces
// (16 for one or two rows).
//
// Without registers: few rows (three CTAs per SM would need 8 or more per
// row): 12 CTAs per row, 16 for one or two rows.  Otherwise the fewest CTAs
// that each read and write at most 80 KiB (at most 16 CTAs), raised toward
// three CTAs per SM; above 8, rounded to a multiple of 4.  Measured on bf16 rows of
// 20 Ki to 256 Ki elements, to bf16 and to fp32: within 5 % of the best
// cluster size, where 48 KiB pieces rounded to a power of two (the rule
// before the barrier-free exchange) were up to 16 % off.
//
// The best shape is within 5 % of these on every measured case.
//
// force_cs: 0 decide; force_ru: -1 decide.  Returns false if no piece within
// the limits holds the row.
bool staged_shape(int64_t M, int64_t nunits, int64_t io_row_bytes, int sms, int max_cluster, bool regs,
                  int64_t force_cs, int64_t force_ru, int64_t force_g, Plan *p) {
    const int64_t row_bytes = nunits * 16;
    const int64_t ru = force_ru >= 0 ? force_ru : regs ? kStagedRegUnits : 0;
    const int64_t threads = force_g > 0 ? force_g : ru > 0 ? kStagedRegThreads : kStagedThreads;
    if (threads > 1024 || !staged_shape_ok((int)threads, (int)ru)) return false;
    const int64_t most = cdiv(nunits, threads);  // >= one unit per thread
    int64_t cs = force_cs;
    if (cs <= 0 && ru > 0) {
        cs = cdiv(row_bytes, kStagedRegPieceBytes);
        const int64_t wide = M <= 2 ? 16 : 12;
        if (M * cs < sms && cs < wide) cs = wide;
        if (cs > max_cluster) cs = max_cluster;
        if (cs > most) cs = most;
    } else if (cs <= 0) {
        int64_t need = cdiv(io_row_bytes, kStagedPieceIoBytes);
        if (need > max_cluster) need = max_cluster;  // the smallest pieces there are
        int64_t fill = cdiv(3 * (int64_t)sms, M);
        if (fill >= 8 && need <= 12) {
            // few rows: spread each row wide.  Measured on 1..64 rows of 64 Ki
            // to 152 Ki elements: 16 CTAs for one or two rows, 12 otherwise
            // (5-18 % faster than 8 or 16, e.g. 64 vocabulary rows 16.7 ->
            // 15.8 us); larger clusters pay more than their extra bandwidth
            cs = M <= 2 ? 16 : 12;
        } else {
            if (fill > most) fill = most;
            if (fill > max_cluster) fill = max_cluster;
            cs = need > fill ? need : fill;
            // above 8, the nearest multiple of 4 that still fits: clusters
            // of 12 packed better than 10, 11 or 13 (128 x 262144 bf16:
            // 27.0 us at 12, 29.4 at 13)
            if (cs > 8) {
                int64_t c4 = (cs + 2) / 4 * 4;
                while (c4 < max_cluster && 128 + cdiv(nunits, c4) * 16 > kStagedMaxSmem) c4 += 4;
                cs = c4;
            }
        }
        if (cs > max_cluster) cs = max_cluster;
        if (cs > most) cs = most;
    }
    if (cs < 1 || cs > max_cluster || cs > kStagedMaxCluster) return false;
    const int64_t chunk = cdiv(nunits, cs);
    const int64_t held = threads * ru;  // units a CTA holds in registers
    const int64_t smem = 128 + (chunk > held ? chunk - held : 0) * 16;
    if (smem > kStagedMaxSmem) return false;
    p->tier = Tier::Staged;
    p->g = (int)threads;
    p->cs = (int)cs;
    p->chunk = chunk;
    p->smem = (size_t)smem;
    p->ru = (int)ru;
    return true;
}

void split_shape(Op op, int64_t M, int64_t N, int64_t nunits, int in_bytes, int sms,
                 int64_t force_s, int64_t force_b, Plan *p) {
    if (op == Op::Softmax) p->ept = kEpt;  // the split softmax kernels' tile
    const int upt = p->ept / p->u;
    const int64_t row_bytes = N * in_bytes;
    int64_t b = force_b > 0 ? force_b : kL2BudgetBytes / (row_bytes > 0 ? row_bytes : 1);
    if (b < 1) b = 1;
    if (b > M) b = M;
    int64_t s = force_s;
    if (s <= 0) {
        s = cdiv(2 * (int64_t)sms, b);
        const int64_t most = cdiv(nunits, (int64_t)kSplitThreads * upt);  // >= one full tile
        if (s > most) s = most;
    }
    if (s > kMaxPieces) s = kMaxPieces;
    if (s > nunits) s = nunits;
    if (s < 1) s = 1;
    p->tier = Tier::Split;
    p->g = kSplitThreads;
    p->cs = (int)s;
    p->chunk = cdiv(nunits, s);
    p->batch_rows = b;
}

osr_status make_plan(Op op, int64_t M, int64_t N, osr_dtype in_dt, osr_dtype out_dt, bool vec,
                     int sms, int max_cluster, Plan *p) {
    *p = Plan();
    p->vec = vec;
    p->u = vec ? vec_elems(in_dt) : 1;
    p->ept = ept_of(op, in_dt, vec);
    const int upt = p->ept / p->u;
    const int64_t nunits = vec ? N / p->u : N;
    const int in_bytes = elem_bytes(in_dt);

    const ForceSpec force_spec = forced_spec();
    const char *force = force_spec.get();
    if (force && *force) {
        p->forced = true;
        int64_t g = 0, cs = 0, s = 0, b = 0;
        if (strncmp(force, "rows", 4) == 0) {
            if (!parse_kv(force, "g", &g)) return OSR_ERR_UNSUPPORTED;
            if (g < 1 || g > 1024 || (g & (g - 1)) || g * upt < nunits) return OSR_ERR_UNSUPPORTED;
            p->tier = Tier::Rows;
            p->g = (int)g;
            return OSR_OK;
        }
        if (strncmp(force, "cluster", 7) == 0) {
            if (!parse_kv(force, "g", &g)) g = 1024;
            if (!parse_kv(force, "cs", &cs)) cs = cdiv(nunits, g * upt);
            if ((g != 256 && g != 1024) || cs < 1 || cs > max_cluster || cs * g * upt < nunits)
                return OSR_ERR_UNSUPPORTED;
            p->tier = Tier::Cluster;
            p->g = (int)g;
            p->cs = (int)cs;
            p->chunk = cdiv(nunits, cs);
            if (p->chunk > g * upt) return OSR_ERR_UNSUPPORTED;
            return OSR_OK;
        }
        if (strncmp(force, "staged", 6) == 0) {
            if (op != Op::Softmax || !vec) return OSR_ERR_UNSUPPORTED;
            int64_t ru = -1;
            parse_kv(force, "cs", &cs);
            parse_kv(force, "r", &ru);
            parse_kv(force, "g", &g);
            if (cs <= 0) cs = 0;
            return staged_shape(M, nunits, N * (in_bytes + elem_bytes(out_dt)), sms, max_cluster,
                                staged_regs(in_dt, out_dt), cs, ru, g, p)
                       ? OSR_OK
                       : OSR_ERR_UNSUPPORTED;
        }
        if (strncmp(force, "split", 5) == 0) {
            parse_kv(force, "s", &s);
            parse_kv(force, "b", &b);
            if (s > kMaxPieces) return OSR_ERR_UNSUPPORTED;
            split_shape(op, M, N, nunits, in_bytes, sms, s, b, p);
            return OSR_OK;
        }
        return OSR_ERR_UNSUPPORTED;
    }

    // 1. the whole row in one group or CTA, register-cached.  Softmax with 32
    //    elements a thread stops at 512 threads: its 1024-thread CTA needs 59-63
    //    registers (one CTA per SM) and measured 7-25 % slower than staging
    //    the 64 KiB row in two CTAs' shared memory.
    const int g = pow2ceil(cdiv(nunits, upt));
    const int gmax = op == Op::Softmax && p->ept > kEpt && vec ? 512 : 1024;
    // a row that needs 1024 threads, or more than a CTA: a cluster of
    // 256-thread CTAs, up to 16 (1024-thread CTAs fit one an SM; measured
    // 16384-element fp32 rows 16-22 % faster for RMSNorm and LayerNorm,
    // 32768-element ones 27-36 %)
    const int64_t cs256 = cdiv(nunits, (int64_t)256 * upt);
    // fused add + RMSNorm on few rows (decode batches): latency is each
    // thread's chain of two loads, an add, a store, the reduction and two
    // more stores, so fewer vectors a thread run faster -- one 16-byte
    // vector a thread (up to 1024 threads) for up to 64 rows, twice the
    // threads (up to 512) for up to 256.  Measured on 3584-8192-element
    // rows: 15-30 % faster (bf16 16 x 4096: 2.43 -> 1.96 us; fp32 64 x
    // 3584: 3.81 -> 2.59 us), slower from 1024 rows on.
    if (op == Op::FusedAddRmsNorm && vec && g <= 1024) {
        int gs = g;
        if (M <= 64) {
            gs = pow2ceil(nunits < 1024 ? nunits : 1024);
        } else if (M <= 256 && 2 * g <= 512) {
            gs = 2 * g;
        }
        if (gs > g) {
            p->tier = Tier::Rows;
            p->g = gs;
            return OSR_OK;
        }
    }
    // LayerNorm on up to 256 16-byte bf16 rows: one vector a thread, up to
    // 512 threads (its two reductions and the pairs' arithmetic make each
    // thread's chain long; measured 1.04-1.29x faster on 2048-8192-element
    // rows, e.g. 64 x 2048: 2.84 -> 2.25 us).  RMSNorm and softmax measured
    // the same either way.
    if (op == Op::LayerNorm && vec && in_dt == OSR_BF16 && M <= 256 && g <= 512) {
        const int gs = pow2ceil(nunits < 512 ? nunits : 512);
        if (gs > g) {
            p->tier = Tier::Rows;
            p->g = gs;
            return OSR_OK;
        }
    }
    if (g <= gmax && (g <= 512 || cs256 > max_cluster)) {
        p->tier = Tier::Rows;
        p->g = g;
        return OSR_OK;
    }
    // 2. softmax on 16-byte rows longer than a CTA: a cluster per row,
    //    pieces staged in shared memory by bulk copies (one read)
    if (g > gmax && op == Op::Softmax && vec &&
        staged_shape(M, nunits, N * (in_bytes + elem_bytes(out_dt)), sms, max_cluster,
                     staged_regs(in_dt, out_dt), 0, -1, 0, p))
        return OSR_OK;
    // 3. a cluster of 256-thread CTAs (1024-thread ones beyond 16 of those),
    //    still register-cached (one read)
    const int64_t cs = cs256 <= max_cluster ? cs256 : cdiv(nunits, (int64_t)1024 * upt);
    if (cs <= max_cluster) {
        p->tier = Tier::Cluster;
        p->g = cs256 <= max_cluster ? 256 : 1024;
        p->cs = (int)cs;
        p->chunk = cdiv(nunits, cs);
        return OSR_OK;
    }
    // 4. two passes through a workspace
    split_shape(op, M, N, nunits, in_bytes, sms, 0, 0, p);
    return OSR_OK;
}

// Log-sum-exp / argmax geometry: the kernel streams, so any shape fits; it
// only has to spread the rows.  Short rows: a group of g <= 32 lanes per row.
// Otherwise one CTA per row, or a cluster of CTAs per row while there are
// too few rows to fill the GPU (sizes below; 16-CTA clusters were 70 %
// slower on 64 vocabulary rows).  A forced spec "lse:cs=<n>,st=<0|1>,
// g=<n>" picks the cluster size, the staged or streaming form and the group
// width (tests).
// rows of at least this many elements that are not 16-byte aligned (or not a
// whole number of vectors) stream their aligned bodies in vectors
constexpr int64_t kLsePeelMinN = 64;

struct LsePlan {
    bool peel = false;  // rows not 16-byte aligned: vector bodies, element edges
    int g = 1;
    int cs = 1;
    int64_t chunk = 0;
    int64_t grid = 0;
    bool staged = false;  // cluster rows staged in shared memory
    size_t smem = 0;      // staged: dynamic shared memory per CTA
};

LsePlan lse_plan(int64_t M, int64_t N, osr_dtype in_dt, bool vec, bool peel, int sms,
                 int smem_per_sm) {
    LsePlan lp;
    const ForceSpec force_spec = forced_spec();
    const char *force = force_spec.get();
    const bool forced = force && strncmp(force, "lse", 3) == 0;
    int64_t fg0 = 0;
    // a peeled row needs a lane per edge element: a forced narrower group
    // takes the element path
    if (peel && forced && parse_kv(force, "g", &fg0) && fg0 < vec_elems(in_dt)) peel = false;
    lp.peel = peel && !vec;
    vec = vec || lp.peel;  // the geometry of 16-byte units from here on
    const int u = vec ? vec_elems(in_dt) : 1;
    const int64_t nunits = vec ? N / u : N;
    const int upt = 32 / u;  // the kernel's 32 elements per thread per tile
    int g = pow2ceil(cdiv(nunits, upt));
    if (g > 256) g = 256;
    // 16-byte rows: narrower groups while each thread still streams at most
    // 16 units (256 bytes: four bf16 tiles, two fp32 tiles) and the grid
    // keeps at least 128 Ki threads.  Fewer threads a row mean fewer block
    // reductions a row and, from 32 lanes down, several rows a CTA reduced
    // by warp shuffles alone.  Measured at 65536 rows (fraction of the copy
    // peak): bf16 4096 elements 0.80 -> 0.99 (g 128 -> 32), 2048 elements
    // 0.58 -> 0.90 (64 -> 16), 1024 elements 0.59 -> 0.79 (32 -> 8); fp32
    // 2048 elements 0.99 -> 1.06 (64 -> 32).
    while (vec && g > 1 && cdiv(nunits, g / 2) <= 16 && M * (g / 2) >= 131072) g /= 2;
    // long 16-byte rows, 128 rows or more: one CTA of up to 1024 threads per
    // row instead of a cluster, as wide as keeps about 16 MB of tiles in
    // flight over the grid while each thread still streams two tiles or
    // more.  Measured on 152064-element rows (fraction of the copy peak,
    // against the clusters / 256-thread CTAs the planner chose before):
    // bf16 128 rows 0.58 against 0.56 (1024 threads), 256 rows 0.75 against
    // 0.67 (1024), 512 rows 0.85 against 0.81 (512); fp32 128 rows 0.84
    // against 0.80, 256 rows 0.94 against 0.92; bf16 32768-element rows at
    // 256 rows 0.44 against 0.39 (512).
    int gw = g;
    if (vec && g == 256 && M >= 128) {
        const int64_t tile = 16 * (int64_t)upt;  // bytes a thread loads per tile
        while (gw < 1024 && M * (gw * 2) * tile <= ((int64_t)1 << 24) && nunits >= (int64_t)gw * 4 * upt)
            gw *= 2;
    }
    int64_t fg = 0;
    if (forced && parse_kv(force, "g", &fg) && fg >= 1 && fg <= 1024 && (fg & (fg - 1)) == 0)
        g = gw = (int)fg;  // a forced group width (tests)
    if (lp.peel && g < u) g = u;
    if (g <= 32) {
        lp.g = g;
        lp.grid = cdiv(M, 128 / g);
        return lp;
    }
    // one CTA per row: as many threads as one tile of the row needs, up to
    // 256 (a 4096-element bf16 row at 256 threads left half of them idle:
    // 8192 such rows 36.2 -> 19.4 us at 128), or fewer or more as above
    lp.g = g;
    int64_t cs = 1;
    int64_t fcs = 0;
    const int64_t most = cdiv(nunits, 256 * (int64_t)upt);  // at least a full tile each
    // staged: 12 CTAs per row (16 for one or two rows), each piece
    // bulk-copied whole, for up to 8 rows long enough for 12 CTAs of full
    // tiles, whose pieces fit one wave.  Measured against 10 streaming CTAs
    // a row: 152064-element rows, 1 bf16 row 3.0 us against 3.4, 8 rows 3.6
    // against 3.8 (fp32 4.0 against 4.0), 12 rows 4.0 against 3.9 (fp32 4.7
    // against 4.3); 32768-element rows (4 CTAs of full tiles) 3.0 against
    // 2.7 at every row count from 1 to 24.
    bool staged_fit = false;
    int64_t cs_st = M <= 2 ? 16 : 12;
    if (cs_st > most) cs_st = most;
    if (vec && !lp.peel && M <= 8 && most >= 12) {
        const int64_t smem = 128 + cdiv(nunits, cs_st) * 16;
        const int64_t per_sm = (int64_t)smem_per_sm / (smem + 1024);  // 1 KiB reserved a CTA
        const int64_t slots = (per_sm < 8 ? per_sm : 8) * sms;
        staged_fit = smem <= kStagedMaxSmem && M * cs_st <= slots;
    }
    if (forced && parse_kv(force, "cs", &fcs) && fcs >= 1 && fcs <= 16) {
        cs = fcs;  // a forced cluster size (tests)
    } else if (staged_fit) {
        cs = cs_st;
    } else if (M * 10 * 10 <= (int64_t)9 * sms * lse_cluster_ctas_per_sm(in_dt == OSR_BF16 ? Dt::BF16 : Dt::F32)) {
        // 10 streaming CTAs a row while the grid fits one wave: the CTAs the
        // kernel holds an SM (5 bf16, 4 fp32) times the SMs, less a tenth
        // for clusters that do not pack into a GPC.  Measured on 152064-
        // element rows (us, against 8 / 12 a row): bf16 24 rows 4.5 against
        // 5.2 / 4.9, 48 rows 5.8 against 6.2 / 6.4, 64 rows 6.8 against
        // 7.1 / 8.8 (80 rows: 9.1 against 8.0 at 8, past one wave); fp32
        // 32 rows 6.1 against 6.4 / 6.2, 56 rows 8.0 against 8.5 (64 rows:
        // 10.7 against 9.2 at 8)
        cs = 10;
    } else if (gw > 256) {
        cs = 1;  // the wide CTAs above
    } else {
        // streaming: about 512 CTAs in all, a power of two per row, at most
        // 8.  Measured (bf16 / fp32, fraction of the copy peak): 152064-
        // element rows, 64 rows at 8 0.39 / 0.62 (10 a row: fp32 16 %
        // slower, the grid past one wave), 96 rows at 4 0.48 / 0.73;
        // 32768-element bf16 rows, 128 rows at 4 0.25 against 0.23 at 1.
        cs = 1;
        while (cs < 8 && M * cs * 2 <= 512) cs *= 2;
    }
    if (cs > most) cs = most;
    if (cs < 1) cs = 1;
    if (cs > 1) lp.g = 256;  // the cluster kernels run 256-thread CTAs
    else if (gw > 256) lp.g = gw;
    lp.cs = (int)cs;
    lp.chunk = cdiv(nunits, cs);
    lp.grid = M * cs;
    int64_t st = staged_fit ? 1 : 0;
    if (forced) parse_kv(force, "st", &st);
    if (cs > 1 && vec && !lp.peel && st != 0 && 128 + lp.chunk * 16 <= kStagedMaxSmem) {
        lp.staged = true;
        lp.smem = (size_t)(128 + lp.chunk * 16);
    }
    return lp;
}

void describe(const Plan &p, char *buf, size_t n) {
    const char *v = p.vec ? "vec" : "scalar";
    switch (p.tier) {
    case Tier::Rows:
        snprintf(buf, n, "rows g=%d ept=%d %s", p.g, p.ept, v);
        break;
    case Tier::Cluster:
        snprintf(buf, n, "cluster cs=%d g=%d ept=%d %s", p.cs, p.g, p.ept, v);
        break;
    case Tier::Split:
        snprintf(buf, n, "split s=%d b=%lld g=%d ept=%d %s", p.cs, (long long)p.batch_rows, p.g,
                 p.ept, v);
        break;
    case Tier::Staged:
        if (p.ru)
            snprintf(buf, n, "staged cs=%d g=%d piece=%lldB r=%d %s", p.cs, p.g, (long long)p.chunk * 16,
                     p.ru, v);
        else
            snprintf(buf, n, "staged cs=%d g=%d piece=%lldB %s", p.cs, p.g, (long long)p.chunk * 16, v);
        break;
    }
}

// ------------------------------------------------------------ execution

cudaError_t launch(Op op, osr_dtype in_dt, osr_dtype out_dt, Kind k, const RowArgs &a,
                   const Plan &p, int64_t grid, cudaStream_t st) {
    if (op == Op::Softmax) {
        if (in_dt == OSR_F32 && out_dt == OSR_F32)
            return launch_softmax<Dt::F32, Dt::F32>(k, a, p.g, p.vec, grid, st);
        if (in_dt == OSR_F32 && out_dt == OSR_BF16)
            return launch_softmax<Dt::F32, Dt::BF16>(k, a, p.g, p.vec, grid, st);
        if (in_dt == OSR_BF16 && out_dt == OSR_F32)
            return launch_softmax<Dt::BF16, Dt::F32>(k, a, p.g, p.vec, grid, st);
        return launch_softmax<Dt::BF16, Dt::BF16>(k, a, p.g, p.vec, grid, st);
    }
    if (op == Op::LayerNorm)
        return in_dt == OSR_F32 ? launch_layernorm<Dt::F32>(k, a, p.g, p.vec, grid, st)
                                : launch_layernorm<Dt::BF16>(k, a, p.g, p.vec, grid, st);
    const bool fused = op == Op::FusedAddRmsNorm;
    if (in_dt == OSR_F32)
        return fused ? launch_rmsnorm<Dt::F32, true>(k, a, p.g, p.vec, grid, st)
                     : launch_rmsnorm<Dt::F32, false>(k, a, p.g, p.vec, grid, st);
    return fused ? launch_rmsnorm<Dt::BF16, true>(k, a, p.g, p.vec, grid, st)
                 : launch_rmsnorm<Dt::BF16, false>(k, a, p.g, p.vec, grid, st);
}

cudaError_t cluster_occupancy(Op op, osr_dtype in_dt, osr_dtype out_dt, const Plan &p, int *n) {
    if (op == Op::Softmax) {
        if (in_dt == OSR_F32 && out_dt == OSR_F32)
            return softmax_cluster_occupancy<Dt::F32, Dt::F32>(p.g, p.vec, p.cs, n);
        if (in_dt == OSR_F32 && out_dt == OSR_BF16)
            return softmax_cluster_occupancy<Dt::F32, Dt::BF16>(p.g, p.vec, p.cs, n);
        if (in_dt == OSR_BF16 && out_dt == OSR_F32)
            return softmax_cluster_occupancy<Dt::BF16, Dt::F32>(p.g, p.vec, p.cs, n);
        return softmax_cluster_occupancy<Dt::BF16, Dt::BF16>(p.g, p.vec, p.cs, n);
    }
    if (op == Op::LayerNorm)
        return in_dt == OSR_F32 ? layernorm_cluster_occupancy<Dt::F32>(p.g, p.vec, p.cs, n)
                                : layernorm_cluster_occupancy<Dt::BF16>(p.g, p.vec, p.cs, n);
    const bool fused = op == Op::FusedAddRmsNorm;
    if (in_dt == OSR_F32)
        return fused ? rmsnorm_cluster_occupancy<Dt::F32, true>(p.g, p.vec, p.cs, n)
                     : rmsnorm_cluster_occupancy<Dt::F32, false>(p.g, p.vec, p.cs, n);
    return fused ? rmsnorm_cluster_occupancy<Dt::BF16, true>(p.g, p.vec, p.cs, n)
                 : rmsnorm_cluster_occupancy<Dt::BF16, false>(p.g, p.vec, p.cs, n);
}

// A cluster plan whose cluster shape the device cannot schedule becomes a
// split plan (or, if it was forced, an OSR_ERR_UNSUPPORTED).  Results of the
// occupancy query are cached per device and kernel shape.
cudaError_t staged_occupancy(osr_dtype in_dt, osr_dtype out_dt, const Plan &p, int *n) {
    if (in_dt == OSR_F32 && out_dt == OSR_F32)
        return softmax_staged_occupancy<Dt::F32, Dt::F32>(p.cs, p.smem, p.g, p.ru, n);
    if (in_dt == OSR_F32 && out_dt == OSR_BF16)
        return softmax_staged_occupancy<Dt::F32, Dt::BF16>(p.cs, p.smem, p.g, p.ru, n);
    if (in_dt == OSR_BF16 && out_dt == OSR_F32)
        return softmax_staged_occupancy<Dt::BF16, Dt::F32>(p.cs, p.smem, p.g, p.ru, n);
    return softmax_staged_occupancy<Dt::BF16, Dt::BF16>(p.cs, p.smem, p.g, p.ru, n);
}

osr_status check_cluster_plan(Op op, int64_t M, int64_t N, osr_dtype in_dt, osr_dtype out_dt,
                              const DeviceInfo &di, Plan *p) {
    if (p->tier != Tier::Cluster && p->tier != Tier::Staged) return OSR_OK;
    static std::mutex mu;
    static std::map<std::tuple<int, int, int, int, int, int, int, int, size_t, int>, int> cache;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    const auto key = std::make_tuple(dev, (int)op, (int)in_dt, (int)out_dt, (int)p->tier, p->g,
                                     (int)p->vec, p->cs, p->smem, p->ru);
    int n = -1;
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) n = it->second;
    }
    if (n < 0) {
        e = p->tier == Tier::Staged ? staged_occupancy(in_dt, out_dt, *p, &n)
                                    : cluster_occupancy(op, in_dt, out_dt, *p, &n);
        if (e != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
        std::lock_guard<std::mutex> lock(mu);
        cache[key] = n;
    }
    if (n > 0) return OSR_OK;
    if (p->forced) return OSR_ERR_UNSUPPORTED;
    const int64_t nunits = p->vec ? N / p->u : N;
    split_shape(op, M, N, nunits, elem_bytes(in_dt), di.sms, 0, 0, p);
    return OSR_OK;
}

// Top-k geometry: one cluster of cs CTAs per row, each caching a piece of
// the row (at most kTopkMaxPieceBytes) in shared memory.  The fewest CTAs
// that hold the row, raised by the row count (below), but never so far that
// a CTA gets less than one vector per thread.
// A forced spec "topk:cs=<n>" (osr_test_force_kernel) picks cs (tests).
struct TopkPlan {
    int cs = 1;
    int64_t chunk = 0;
    int sort_n = 1;
    uint32_t region0 = 0;
    size_t smem = 0;
    bool forced = false;
};

constexpr size_t kTopkSmemLimit = 227 * 1024 - 256;  // dynamic shared memory per CTA

osr_status topk_plan(int64_t M, int64_t N, int64_t k, osr_dtype dt, bool vec, int sms,
                     int max_cluster, int smem_per_sm, TopkPlan *tp) {
    *tp = TopkPlan();
    const int eb = elem_bytes(dt);
    const int u = vec ? vec_elems(dt) : 1;
    const int64_t cs_min = cdiv(N * eb, kTopkMaxPieceBytes);
    int64_t cs = cs_min;
    const ForceSpec force_spec = forced_spec();
    const char *force = force_spec.get();
    // CTAs of c a row that an SM holds by shared memory (at most 4, the
    // register bound); 0 if a piece of that size does not fit
    auto per_sm = [&](int64_t c) -> int64_t {
        const int64_t ch = cdiv(cdiv(N, c), u) * u;
        if (ch * eb > kTopkMaxPieceBytes) return 0;
        const int64_t cb = ch * eb + (vec ? 0 : 16);
        int64_t r = cb > pow2_at_least(k) * 8 ? cb : pow2_at_least(k) * 8;
        if (r < kTopkMinWords * 8) r = kTopkMinWords * 8;
        const int64_t sm = (int64_t)topk_smem_bytes((uint32_t)cdiv(r, 16) * 16, k);
        if (sm > kTopkSmemLimit) return 0;
        const int64_t per = smem_per_sm / (sm + kTopkStaticSmem + 1024);  // 1 KiB reserved a CTA
        return per > 4 ? 4 : per;
    };
    // c CTAs a row leave at least a vector a thread (or c is the fewest the row needs)
    auto enough_work = [&](int64_t c) { return c == cs_min || cdiv(N, c) >= (int64_t)kTopkThreads * u; };
    const int64_t c_max = kTopkMaxCluster < max_cluster ? kTopkMaxCluster : max_cluster;
    int64_t fcs = 0;
    if (force && strncmp(force, "topk", 4) == 0) {
        if (!parse_kv(force, "cs", &fcs) || fcs < 1) return OSR_ERR_UNSUPPORTED;
        cs = fcs;
        tp->forced = true;
    } else if (M > 96) {
        // many rows: each CTA's time is mostly a chain of short phases, so
        // what counts is how many rows an SM works on at once -- the CTAs an
        // SM holds over the CTAs a row needs; on a tie, the fewest CTAs a row
        // that still puts two on an SM (a lone CTA an SM leaves its copy and
        // phases unoverlapped: 262144 bf16 elements at 3 CTAs a row, one an
        // SM, 0.28 against 0.33 at 6, two an SM).  Measured at 512-2048
        // rows (fraction of the copy peak, against the 6 CTAs a row before):
        // bf16 152064 elements 3 CTAs 0.34 against 0.31, 65536 elements 3
        // 0.33 against 0.20, 32768 elements 2 0.24 against 0.11; fp32 32768
        // elements 3 0.35 against 0.21; fp32 152064 and bf16 262144 stay at 6.
        int64_t best = 0, best_per = 0;
        for (int64_t c = cs_min; c <= c_max; ++c) {
            if (!enough_work(c)) break;
            const int64_t per = per_sm(c);
            if (per == 0) continue;
            if (best == 0 || per * best > best_per * c || (per * best == best_per * c && best_per < 2 && per > best_per)) {
                best = c;
                best_per = per;
            }
        }
        if (best > 0) cs = best;
    } else {
        // measured on 1-96 rows of 152064 elements: 8 CTAs per row while the
        // clusters still spread one CTA an SM (up to 15 rows on 152 SMs;
        // 3-5 % faster than 12, 7-11 % faster than 16, 2-8 % faster than
        // 6), then 6 (16-22 rows: 2-5 % faster than 8 or 4; at 24 rows 4 %
        // slower than 4), then 4 up to 96 rows (64 bf16 rows: 14.2 us
        // against 14.4 at 2, 15.3 at 3, 15.8 at 5, 15.0 at 6, 16.2 at 8);
        // never fewer than the row needs, and never so many that a CTA gets
        // less than one vector per thread
        const int64_t fill = M * 8 <= (int64_t)sms * 4 / 5 ? 8 : M * 6 <= (int64_t)sms * 7 / 8 ? 6 : 4;
        if (fill > cs) cs = fill;
        while (cs > cs_min && cdiv(N, cs) < (int64_t)kTopkThreads * u) cs = cs / 2 > cs_min ? cs / 2 : cs_min;
        // ... as long as the grid stays one wave: past it, the most CTAs a
        // row below that still fit (96 bf16 rows: 4 CTAs a row, 384 CTAs at
        // two an SM, 23.1 us; 3 a row 16.6 us).  Where no size fits (64 fp32
        // rows of 152064 elements), the size with the fewest CTAs per
        // resident slot, the larger on a tie (4 a row, one an SM: 25.9 us;
        // 5, one an SM: 28.7; 6, two an SM: 23.6; 8, two an SM: 24.9).
        auto fits = [&](int64_t c) {
            const int64_t per = per_sm(c);
            return per > 0 && M * c <= per * (int64_t)sms;
        };
        if (!fits(cs)) {
            int64_t c = cs - 1;
            while (c >= cs_min && !fits(c)) --c;
            if (c >= cs_min) {
                cs = c;
            } else {
                int64_t best = 0, best_per = 0;
                for (int64_t c2 = cs_min; c2 <= c_max; ++c2) {
                    if (!enough_work(c2)) break;
                    const int64_t per = per_sm(c2);
                    if (per == 0) continue;
                    if (best == 0 || c2 * best_per <= best * per) {  // c2 / per <= best / best_per
                        best = c2;
                        best_per = per;
                    }
                }
                if (best > 0) cs = best;
            }
        }
    }
    if (cs > max_cluster || cs > kTopkMaxCluster) return OSR_ERR_UNSUPPORTED;
    const int64_t chunk = cdiv(cdiv(N, cs), u) * u;
    if (chunk * eb > kTopkMaxPieceBytes) return OSR_ERR_UNSUPPORTED;
    const int64_t sort_n = pow2_at_least(k);
    // the region holds the piece (element path: shifted by up to 15 bytes,
    // as it lies off the 16-byte grid), and later the gathered lists or the
    // sort
    const int64_t pb = chunk * eb + (vec ? 0 : 16);
    int64_t r0 = pb > sort_n * 8 ? pb : sort_n * 8;
    if (r0 < kTopkMinWords * 8) r0 = kTopkMinWords * 8;
    r0 = cdiv(r0, 16) * 16;
    const size_t smem = topk_smem_bytes((uint32_t)r0, k);
    if (smem > kTopkSmemLimit) return OSR_ERR_UNSUPPORTED;
    tp->cs = (int)cs;
    tp->chunk = chunk;
    tp->sort_n = (int)sort_n;
    tp->region0 = (uint32_t)r0;
    tp->smem = smem;
    return OSR_OK;
}

osr_status execute(Op op, osr_dtype in_dt, osr_dtype out_dt, RowArgs a, const Plan &p,
                   cudaStream_t st) {
    const int64_t M = a.M;
    cudaError_t e = cudaSuccess;
    switch (p.tier) {
    case Tier::Rows: {
        const int64_t grid = p.g <= 32 ? cdiv(M, 128 / p.g) : M;
        if (grid > 0x7fffffffLL) return OSR_ERR_UNSUPPORTED;
        e = launch(op, in_dt, out_dt, Kind::Rows, a, p, grid, st);
        break;
    }
    case Tier::Cluster: {
        const int64_t grid = M * p.cs;
        if (grid > 0x7fffffffLL) return OSR_ERR_UNSUPPORTED;
        a.cs = p.cs;
        a.chunk = p.chunk;
        e = launch(op, in_dt, out_dt, Kind::Cluster, a, p, grid, st);
        break;
    }
    case Tier::Staged: {
        const int64_t grid = M * p.cs;
        if (grid > 0x7fffffffLL) return OSR_ERR_UNSUPPORTED;
        a.cs = p.cs;
        a.chunk = p.chunk;
        if (g_test_flags.load(std::memory_order_relaxed) & OSR_TEST_NO_ARRIVE) a.flags |= kFlagNoArrive;
        if (in_dt == OSR_F32 && out_dt == OSR_F32)
            e = launch_softmax_staged<Dt::F32, Dt::F32>(a, grid, p.smem, p.g, p.ru, st);
        else if (in_dt == OSR_F32 && out_dt == OSR_BF16)
            e = launch_softmax_staged<Dt::F32, Dt::BF16>(a, grid, p.smem, p.g, p.ru, st);
        else if (in_dt == OSR_BF16 && out_dt == OSR_F32)
            e = launch_softmax_staged<Dt::BF16, Dt::F32>(a, grid, p.smem, p.g, p.ru, st);
        else
            e = launch_softmax_staged<Dt::BF16, Dt::BF16>(a, grid, p.smem, p.g, p.ru, st);
        break;
    }
    case Tier::Split: {
        a.cs = p.cs;
        a.chunk = p.chunk;
        const size_t state = op == Op::Softmax     ? sizeof(float2)
                             : op == Op::LayerNorm ? sizeof(float4)
                                                   : sizeof(float);
        void *ws = nullptr;
        if ((e = cudaMallocAsync(&ws, (size_t)M * p.cs * state, st)) != cudaSuccess)
            return cuda_fail(e);
        a.ws = ws;
        for (int64_t r0 = 0; r0 < M && e == cudaSuccess; r0 += p.batch_rows) {
            const int64_t rows = M - r0 < p.batch_rows ? M - r0 : p.batch_rows;
            const int64_t grid = rows * p.cs;
            if (grid > 0x7fffffffLL) {
                e = cudaErrorInvalidConfiguration;
                break;
            }
            a.row0 = r0;
            e = launch(op, in_dt, out_dt, Kind::SplitStats, a, p, grid, st);
            if (e == cudaSuccess) e = launch(op, in_dt, out_dt, Kind::SplitApply, a, p, grid, st);
        }
        cudaError_t f = cudaFreeAsync(ws, st);
        if (e == cudaSuccess) e = f;
        break;
    }
    }
    return e == cudaSuccess ? OSR_OK : cuda_fail(e);
}

// ------------------------------------------------------------ validation

bool overlaps(const void *a, int64_t an, const void *b, int64_t bn) {
    const char *pa = (const char *)a, *pb = (const char *)b;
    return pa < pb + bn && pb < pa + an;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// The buffer must be memory the device can address at that same address:
// device or managed memory, or page-locked host memory that the runtime maps
// into the unified address space (cudaHostAlloc / cudaHostRegister on a
// unified-addressing system: the kernels then read and write it over the
// host link, no staging copy).  Pageable host memory is refused.
bool device_accessible(const void *p) {
    cudaPointerAttributes at;
    cudaError_t e = cudaPointerGetAttributes(&at, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) return true;
    return at.type == cudaMemoryTypeHost && at.devicePointer == p;
}

osr_status check_sizes(int64_t M, int64_t N) {
    if (M < 0 || N <= 0) return OSR_ERR_INVALID;
    if (N > ((int64_t)1 << 40) || M > ((int64_t)1 << 40)) return OSR_ERR_UNSUPPORTED;
    // byte sizes (M x N x up to 8 bytes) must fit int64 arithmetic
    if (M > 0 && N > ((int64_t)1 << 59) / M) return OSR_ERR_UNSUPPORTED;
    return OSR_OK;
}

}  // namespace
}  // namespace osr

using namespace osr;

extern "C" {

const char *osr_status_string(osr_status s) {
    switch (s) {
    case OSR_OK: return "ok";
    case OSR_ERR_INVALID: return "invalid argument (size, null pointer or dtype)";
    case OSR_ERR_ALIGN: return "misaligned buffer";
    case OSR_ERR_ALIAS: return "buffers overlap in a way the call forbids";
    case OSR_ERR_UNSUPPORTED: return "arguments outside what is implemented";
    case OSR_ERR_CUDA: return "CUDA call or kernel launch failed";
    case OSR_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

int osr_last_cuda_error(void) { return g_last_cuda_error; }

int osr_test_set_flags(int flags) { return g_test_flags.exchange(flags); }

osr_status osr_test_force_kernel(const char *spec) {
    if (spec && strlen(spec) >= sizeof g_force) return OSR_ERR_INVALID;
    std::lock_guard<std::mutex> lock(g_force_mu);
    if (spec) {
        strcpy(g_force, spec);
    } else {
        g_force[0] = 0;
    }
    g_force_set.store(g_force[0] != 0, std::memory_order_release);
    return OSR_OK;
}

int osr_version(void) { return 100; }

osr_status osr_plan_describe(int op, int64_t M, int64_t N, osr_dtype in_dt, osr_dtype out_dt,
                             int vec_ok, int sm_count, char *buf, size_t buf_len) {
    if (op < 0 || op > 6 || !dtype_ok(in_dt) || !dtype_ok(out_dt) || !buf || buf_len == 0 ||
        sm_count <= 0)
        return OSR_ERR_INVALID;
    if ((op < 2 || op == 5) && in_dt != out_dt) return OSR_ERR_UNSUPPORTED;
    if (op == 6) {  // top-k: the plan for k = 64 (k changes only the sort buffer)
        const bool tvec = vec_ok && (N % vec_elems(in_dt)) == 0;
        TopkPlan tp;
        const osr_status ts = topk_plan(M, N, N < 64 ? N : 64, in_dt, tvec, sm_count, 16, kSmemPerSmDefault, &tp);
        if (ts != OSR_OK) return ts;
        snprintf(buf, buf_len, "topk cs=%d piece=%lldB %s", tp.cs,
                 (long long)(tp.chunk * elem_bytes(in_dt)), tvec ? "vec" : "scalar");
        return OSR_OK;
    }
    osr_status s = check_sizes(M, N);
    if (s != OSR_OK) return s;
    const bool vec = vec_ok && (N % vec_elems(in_dt)) == 0;
    if (op == 4) {
        const LsePlan lp = lse_plan(M, N, in_dt, vec, !vec && N >= kLsePeelMinN, sm_count,
                                    kSmemPerSmDefault);
        const char *path = lp.peel ? "peel" : vec ? "vec" : "scalar";
        if (lp.staged)
            snprintf(buf, buf_len, "lse-staged g=%d cs=%d piece=%lldB %s", lp.g, lp.cs,
                     (long long)lp.chunk * 16, path);
        else
            snprintf(buf, buf_len, "%s g=%d cs=%d %s", lp.cs > 1 ? "lse-cluster" : "lse-rows", lp.g,
                     lp.cs, path);
        return OSR_OK;
    }
    Plan p;
    const Op o = op == 5 ? Op::LayerNorm : op >= 2 ? Op::Softmax : (Op)op;
    s = make_plan(o, M, N, in_dt, out_dt, vec, sm_count, 16, &p);
    if (s != OSR_OK) return s;
    describe(p, buf, buf_len);
    return OSR_OK;
}

osr_status osr_rmsnorm_fwd(const void *x, const void *gamma, float eps, void *y, int64_t M,
                           int64_t H, osr_dtype dt, void *stream) {
    osr_status s = check_sizes(M, H);
    if (s != OSR_OK) return s;
    if (!dtype_ok(dt)) return OSR_ERR_INVALID;
    if (M == 0) return OSR_OK;
    if (!x || !gamma || !y) return OSR_ERR_INVALID;
    const int64_t bytes = M * H * elem_bytes(dt), gbytes = H * elem_bytes(dt);
    if ((y != x && overlaps(x, bytes, y, bytes)) || overlaps(y, bytes, gamma, gbytes))
        return OSR_ERR_ALIAS;
    if (!device_accessible(x) || !device_accessible(gamma) || !device_accessible(y))
        return OSR_ERR_INVALID;
    DeviceInfo di;
    if ((s = device_info(&di)) != OSR_OK) return s;
    const bool vec = aligned16(x) && aligned16(gamma) && aligned16(y) && H % vec_elems(dt) == 0;
    Plan p;
    if ((s = make_plan(Op::RmsNorm, M, H, dt, dt, vec, di.sms, di.max_cluster, &p)) != OSR_OK)
        return s;
    if ((s = check_cluster_plan(Op::RmsNorm, M, H, dt, dt, di, &p)) != OSR_OK) return s;
    RowArgs a = {};
    a.x = x;
    a.gamma = gamma;
    a.y = y;
    a.M = M;
    a.N = H;
    a.eps = eps;
    return execute(Op::RmsNorm, dt, dt, a, p, (cudaStream_t)stream);
}

osr_status osr_fused_add_rmsnorm(const void *x, void *residual, const void *gamma, float eps,
                                 void *out, int64_t M, int64_t H, osr_dtype dt, void *stream) {
    osr_status s = check_sizes(M, H);
    if (s != OSR_OK) return s;
    if (!dtype_ok(dt)) return OSR_ERR_INVALID;
    if (M == 0) return OSR_OK;
    if (!x || !residual || !gamma || !out) return OSR_ERR_INVALID;
    const int64_t bytes = M * H * elem_bytes(dt), gbytes = H * elem_bytes(dt);
    if (overlaps(residual, bytes, x, bytes) || overlaps(residual, bytes, out, bytes) ||
        overlaps(residual, bytes, gamma, gbytes) || overlaps(out, bytes, gamma, gbytes) ||
        (out != x && overlaps(out, bytes, x, bytes)))
        return OSR_ERR_ALIAS;
    if (!device_accessible(x) || !device_accessible(residual) || !device_accessible(gamma) ||
        !device_accessible(out))
        return OSR_ERR_INVALID;
    DeviceInfo di;
    if ((s = device_info(&di)) != OSR_OK) return s;
    const bool vec = aligned16(x) && aligned16(residual) && aligned16(gamma) && aligned16(out) &&
                     H % vec_elems(dt) == 0;
    Plan p;
    if ((s = make_plan(Op::FusedAddRmsNorm, M, H, dt, dt, vec, di.sms, di.max_cluster, &p)) !=
        OSR_OK)
        return s;
    if ((s = check_cluster_plan(Op::FusedAddRmsNorm, M, H, dt, dt, di, &p)) != OSR_OK) return s;
    RowArgs a = {};
    a.x = x;
    a.res = residual;
    a.gamma = gamma;
    a.y = out;
    a.M = M;
    a.N = H;
    a.eps = eps;
    return execute(Op::FusedAddRmsNorm, dt, dt, a, p, (cudaStream_t)stream);
}

osr_status osr_layernorm_fwd(const void *x, const void *gamma, const void *beta, float eps,
                             void *y, int64_t M, int64_t H, osr_dtype dt, void *stream) {
    osr_status s = check_sizes(M, H);
    if (s != OSR_OK) return s;
    if (!dtype_ok(dt)) return OSR_ERR_INVALID;
    if (M == 0) return OSR_OK;
    if (!x || !gamma || !beta || !y) return OSR_ERR_INVALID;
    const int64_t bytes = M * H * elem_bytes(dt), pbytes = H * elem_bytes(dt);
    if ((y != x && overlaps(x, bytes, y, bytes)) || overlaps(y, bytes, gamma, pbytes) ||
        overlaps(y, bytes, beta, pbytes))
        return OSR_ERR_ALIAS;
    if (!device_accessible(x) || !device_accessible(gamma) || !device_accessible(beta) ||
        !device_accessible(y))
        return OSR_ERR_INVALID;
    DeviceInfo di;
    if ((s = device_info(&di)) != OSR_OK) return s;
    const bool vec = aligned16(x) && aligned16(gamma) && aligned16(beta) && aligned16(y) &&
                     H % vec_elems(dt) == 0;
    Plan p;
    if ((s = make_plan(Op::LayerNorm, M, H, dt, dt, vec, di.sms, di.max_cluster, &p)) != OSR_OK)
        return s;
    if ((s = check_cluster_plan(Op::LayerNorm, M, H, dt, dt, di, &p)) != OSR_OK) return s;
    RowArgs a = {};
    a.x = x;
    a.gamma = gamma;
    a.beta = beta;
    a.y = y;
    a.M = M;
    a.N = H;
    a.eps = eps;
    return execute(Op::LayerNorm, dt, dt, a, p, (cudaStream_t)stream);
}

static osr_status softmax_entry(const void *x, void *y, float *row_max, float *row_sum,
                                int64_t M, int64_t N, osr_dtype in_dt, osr_dtype out_dt, int flags,
                                void *stream) {
    osr_status s = check_sizes(M, N);
    if (s != OSR_OK) return s;
    if (!dtype_ok(in_dt) || !dtype_ok(out_dt)) return OSR_ERR_INVALID;
    if (M == 0) return OSR_OK;
    if (!x || !y) return OSR_ERR_INVALID;
    const int64_t xb = M * N * elem_bytes(in_dt), yb = M * N * elem_bytes(out_dt);
    const bool in_place = x == y && in_dt == out_dt;
    if (!in_place && overlaps(x, xb, y, yb)) return OSR_ERR_ALIAS;
    const void *stats[2] = {row_max, row_sum};
    for (const void *q : stats)
        if (q && (overlaps(q, M * 4, x, xb) || overlaps(q, M * 4, y, yb))) return OSR_ERR_ALIAS;
    if (row_max && row_sum && overlaps(row_max, M * 4, row_sum, M * 4)) return OSR_ERR_ALIAS;
    if (!device_accessible(x) || !device_accessible(y)) return OSR_ERR_INVALID;
    if ((row_max && !device_accessible(row_max)) || (row_sum && !device_accessible(row_sum)))
        return OSR_ERR_INVALID;
    DeviceInfo di;
    if ((s = device_info(&di)) != OSR_OK) return s;
    const bool vec = aligned16(x) && aligned16(y) && N % vec_elems(in_dt) == 0;
    Plan p;
    if ((s = make_plan(Op::Softmax, M, N, in_dt, out_dt, vec, di.sms, di.max_cluster, &p)) !=
        OSR_OK)
        return s;
    if ((s = check_cluster_plan(Op::Softmax, M, N, in_dt, out_dt, di, &p)) != OSR_OK) return s;
    RowArgs a = {};
    a.x = x;
    a.y = y;
    a.row_max = row_max;
    a.row_sum = row_sum;
    a.M = M;
    a.N = N;
    a.flags = flags;
    return execute(Op::Softmax, in_dt, out_dt, a, p, (cudaStream_t)stream);
}

osr_status osr_softmax_rows_stats(const void *x, void *y, float *row_max, float *row_sum,
                                  int64_t M, int64_t N, osr_dtype in_dt, osr_dtype out_dt,
                                  void *stream) {
    return softmax_entry(x, y, row_max, row_sum, M, N, in_dt, out_dt, 0, stream);
}

osr_status osr_log_softmax_rows(const void *x, void *y, int64_t M, int64_t N, osr_dtype in_dt,
                                osr_dtype out_dt, void *stream) {
    return softmax_entry(x, y, nullptr, nullptr, M, N, in_dt, out_dt, kFlagLog, stream);
}

osr_status osr_row_logsumexp(const void *x, float *lse, int64_t *argmax, int64_t M, int64_t N,
                             osr_dtype in_dt, void *stream) {
    osr_status s = check_sizes(M, N);
    if (s != OSR_OK) return s;
    if (!dtype_ok(in_dt)) return OSR_ERR_INVALID;
    if (M == 0) return OSR_OK;
    if (!x || (!lse && !argmax)) return OSR_ERR_INVALID;
    const int64_t xb = M * N * elem_bytes(in_dt);
    if ((lse && overlaps(lse, M * 4, x, xb)) || (argmax && overlaps(argmax, M * 8, x, xb)) ||
        (lse && argmax && overlaps(lse, M * 4, argmax, M * 8)))
        return OSR_ERR_ALIAS;
    if (!device_accessible(x) || (lse && !device_accessible(lse)) ||
        (argmax && !device_accessible(argmax)))
        return OSR_ERR_INVALID;
    DeviceInfo di;
    if ((s = device_info(&di)) != OSR_OK) return s;
    const bool vec = aligned16(x) && N % vec_elems(in_dt) == 0;
    const bool peel = !vec && N >= kLsePeelMinN && (uintptr_t)x % elem_bytes(in_dt) == 0;
    const LsePlan lp = lse_plan(M, N, in_dt, vec, peel, di.sms, di.smem_per_sm);
    if (lp.grid > 0x7fffffffLL) return OSR_ERR_UNSUPPORTED;
    RowArgs a = {};
    a.x = x;
    a.row_sum = lse;
    a.row_arg = argmax;
    a.M = M;
    a.N = N;
    a.cs = lp.cs;
    a.chunk = lp.chunk;
    const cudaError_t e =
        lp.staged ? (in_dt == OSR_F32 ? launch_lse_staged<Dt::F32>(a, lp.grid, lp.smem, (cudaStream_t)stream)
                                      : launch_lse_staged<Dt::BF16>(a, lp.grid, lp.smem, (cudaStream_t)stream))
        : lp.peel ? (in_dt == OSR_F32 ? launch_lse_peel<Dt::F32>(a, lp.g, lp.cs > 1, lp.grid, (cudaStream_t)stream)
                                      : launch_lse_peel<Dt::BF16>(a, lp.g, lp.cs > 1, lp.grid, (cudaStream_t)stream))
        : in_dt == OSR_F32 ? launch_lse<Dt::F32>(a, lp.g, lp.cs > 1, vec, lp.grid, (cudaStream_t)stream)
                           : launch_lse<Dt::BF16>(a, lp.g, lp.cs > 1, vec, lp.grid, (cudaStream_t)stream);
    return e == cudaSuccess ? OSR_OK : cuda_fail(e);
}

osr_status osr_row_topk(const void *x, float *values, int64_t *indices, float *probs, float *lse,
                        int64_t M, int64_t N, int64_t k, osr_dtype in_dt, void *stream) {
    osr_status s = check_sizes(M, N);
    if (s != OSR_OK) return s;
    if (!dtype_ok(in_dt) || k < 1 || k > N) return OSR_ERR_INVALID;
    if (k > kTopkMaxK || N >= ((int64_t)1 << 31)) return OSR_ERR_UNSUPPORTED;
    if (M == 0) return OSR_OK;
    if (!x || !values || !indices) return OSR_ERR_INVALID;
    const int64_t xb = M * N * elem_bytes(in_dt), vb = M * k * 4, ib = M * k * 8, lb = M * 4;
    const void *bufs[4] = {values, indices, probs, lse};
    const int64_t lens[4] = {vb, ib, vb, lb};
    for (int i = 0; i < 4; ++i) {
        if (!bufs[i]) continue;
        if (overlaps(bufs[i], lens[i], x, xb)) return OSR_ERR_ALIAS;
        for (int j = i + 1; j < 4; ++j)
            if (bufs[j] && overlaps(bufs[i], lens[i], bufs[j], lens[j])) return OSR_ERR_ALIAS;
    }
    for (int i = 0; i < 4; ++i)
        if (bufs[i] && !device_accessible(bufs[i])) return OSR_ERR_INVALID;
    if (!device_accessible(x)) return OSR_ERR_INVALID;
    DeviceInfo di;
    if ((s = device_info(&di)) != OSR_OK) return s;
    const bool vec = aligned16(x) && N % vec_elems(in_dt) == 0;
    TopkPlan tp;
    if ((s = topk_plan(M, N, k, in_dt, vec, di.sms, di.max_cluster, di.smem_per_sm, &tp)) != OSR_OK) return s;
    if (M * tp.cs > 0x7fffffffLL) return OSR_ERR_UNSUPPORTED;
    // the cluster shape must be schedulable with this much shared memory
    int n = 0;
    cudaError_t e = in_dt == OSR_F32 ? topk_occupancy<Dt::F32>(vec, tp.cs, tp.smem, &n)
                                     : topk_occupancy<Dt::BF16>(vec, tp.cs, tp.smem, &n);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return OSR_ERR_UNSUPPORTED;
    }
    if (n < 1) return OSR_ERR_UNSUPPORTED;
    TopkArgs a = {};
    a.x = x;
    a.values = values;
    a.indices = indices;
    a.probs = probs;
    a.lse = lse;
    a.M = M;
    a.N = N;
    a.k = k;
    a.chunk = tp.chunk;
    a.cs = tp.cs;
    a.sort_n = tp.sort_n;
    a.region0 = tp.region0;
    e = in_dt == OSR_F32 ? launch_topk<Dt::F32>(a, vec, tp.smem, (cudaStream_t)stream)
                         : launch_topk<Dt::BF16>(a, vec, tp.smem, (cudaStream_t)stream);
    return e == cudaSuccess ? OSR_OK : cuda_fail(e);
}

osr_status osr_softmax_rows(const void *x, void *y, int64_t M, int64_t N, osr_dtype in_dt,
                            osr_dtype out_dt, void *stream) {
    return osr_softmax_rows_stats(x, y, nullptr, nullptr, M, N, in_dt, out_dt, stream);
}

}  // extern "C"
