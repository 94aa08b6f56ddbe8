/*
 * osr.h -- C ABI of the GB300 (sm_103a) row-wise reduce-then-rescale library.
 *
 * Three operations, each applied independently to every row of a row-major
 * matrix:
 *
 *   RMSNorm                y_j = x_j * (mean_j x_j^2 + eps)^(-1/2) * gamma_j
 *   fused residual-add +   h = x + residual (written back to residual),
 *     RMSNorm              out = RMSNorm(h) * gamma
 *   safe softmax           y_i = exp(x_i - m) / d,  m = max_j x_j,
 *                          d = sum_j exp(x_j - m), with (m, d) built by the
 *                          online normaliser and its associative merge
 *                          (m, d) = (max(m1, m2), d1 e^(m1-m) + d2 e^(m2-m)).
 *
 * Pages defining these operations (cited by title and section):
 *   "RMSNorm、Softmax 与在线归约" (notes.kuangjux.top): "RMSNorm 归约什么",
 *       "稳定 Softmax：归一化之前先减最大值", "Online Softmax 为什么要重缩放旧的和",
 *       "从逐元素更新到合并两个 tile".
 *   "GPU Kernel 工程（04）：共享内存与 reduction——softmax、LayerNorm 与 online
 *       softmax" (arganzheng.life): 七 "softmax：safe、三遍、两遍、online",
 *       八.1 "RMSNorm：均方在 FP32 累加", 八.3 "fused residual + RMSNorm".
 *   "两个融合算子：RMSNorm 与 online softmax" (daleiyang.github.io): §5
 *       "递推式怎么来的", "结合律：为什么能做树形归约".
 *   "Softmax 与归一化", CUDA 进阶手册 (anrans.github.io): "Online softmax",
 *       "按行长度选择并行方式" (row-length dispatch table).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers named x, y, residual, gamma, beta, out, row_max, row_sum, lse,
 *   values, ... are pointers the current CUDA device can read/write at that
 *   address: device memory (cudaMalloc, cudaMallocAsync, a torch CUDA
 *   tensor's data_ptr()), managed memory, or page-locked host memory mapped
 *   into the unified address space (cudaHostAlloc, cudaHostRegister, a
 *   pinned torch CPU tensor's data_ptr()): the kernels then read and write
 *   host memory over the host link, with no staging copy.  Pageable host
 *   memory returns OSR_ERR_INVALID.  The caller owns every buffer; the
 *   library keeps no pointer after the call returns.
 * - Matrices are row-major and dense: row i starts at element i * (row
 *   length).  Rows of length H (norms) or N (softmax).
 * - Arithmetic is binary32 for every dtype (bfloat16 inputs are widened
 *   exactly, sums and maxima accumulate in binary32); results are rounded
 *   once to the output dtype, round-to-nearest-even.
 * - Any alignment is accepted: 16-byte aligned buffers whose row length in
 *   bytes is a multiple of 16 take 128-bit loads/stores, anything else takes
 *   an element-wise path with the same arithmetic.
 * - `stream` is a cudaStream_t (NULL = the legacy default stream).  All
 *   device work is enqueued on it asynchronously; no entry point
 *   synchronises the device or the stream.  The split-row path draws a small
 *   workspace (rows x pieces x 8 bytes) from the stream-ordered allocator
 *   (cudaMallocAsync / cudaFreeAsync on `stream`).
 * - M == 0 is a no-op returning OSR_OK.  Row length <= 0, M < 0, a NULL
 *   required pointer, or a dtype value outside osr_dtype return
 *   OSR_ERR_INVALID before any device work.  M and the row length may each
 *   be up to 2^40 and their product up to 2^59; beyond that the call returns
 *   OSR_ERR_UNSUPPORTED before any device work.  Errors are reported only by
 *   return value: nothing is printed and the process is never terminated.
 * - Entry points are thread-safe; calls on the same stream execute in order.
 */
#ifndef OSR_H
#define OSR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum osr_dtype {
    OSR_F32 = 0,  /* IEEE binary32 */
    OSR_BF16 = 1  /* bfloat16: the upper 16 bits of a binary32 */
} osr_dtype;

typedef enum osr_status {
    OSR_OK = 0,
    OSR_ERR_INVALID = 1,        /* bad size, NULL pointer or dtype value */
    OSR_ERR_ALIGN = 2,          /* reserved: misalignment is never an error */
    OSR_ERR_ALIAS = 3,          /* buffers overlap in a way the call forbids */
    OSR_ERR_UNSUPPORTED = 4,    /* valid arguments outside what is implemented */
    OSR_ERR_CUDA = 5,           /* a CUDA call or launch failed: osr_last_cuda_error() */
    OSR_ERR_DEVICE_TIMEOUT = 6  /* a kernel's bounded wait ran out (see osr_device_fault) */
} osr_status;

/*
 * RMSNorm forward: y[i, j] = x[i, j] * r_i * gamma[j],
 * r_i = 1 / sqrt(sum_j x[i, j]^2 / H + eps).
 *   x      [M, H] of dtype dt, read only (may equal y: in place)
 *   gamma  [H] of dtype dt
 *   eps    added to the mean square inside the square root
 *   y      [M, H] of dtype dt, written
 * y == x is allowed; any other overlap of y with x or gamma -> OSR_ERR_ALIAS.
 */
osr_status osr_rmsnorm_fwd(const void *x, const void *gamma, float eps, void *y,
                           int64_t M, int64_t H, osr_dtype dt, void *stream);

/*
 * Fused residual-add + RMSNorm:
 *   residual[i, j] <- round_dt(x[i, j] + residual[i, j])
 *   out[i, j]      <- residual[i, j] * r_i * gamma[j]   (of the rounded sum)
 *   x        [M, H] dtype dt, read only (may equal out: in place)
 *   residual [M, H] dtype dt, read and overwritten
 *   gamma    [H] dtype dt
 *   out      [M, H] dtype dt, written
 * out == x is allowed.  residual must not overlap x, out or gamma, and out
 * must not overlap gamma -> otherwise OSR_ERR_ALIAS.
 */
osr_status osr_fused_add_rmsnorm(const void *x, void *residual, const void *gamma, float eps,
                                 void *out, int64_t M, int64_t H, osr_dtype dt, void *stream);

/*
 * LayerNorm forward: y[i, j] = (x[i, j] - mu_i) / sqrt(var_i + eps) * gamma[j]
 * + beta[j], mu_i = (1/H) sum_j x[i, j], var_i = (1/H) sum_j (x[i, j] - mu_i)^2
 * ("Softmax 与归一化" (anrans.github.io), "LayerNorm 与 RMSNorm"; "GPU Kernel
 * 工程（04）" 八.2).  Two passes over the row held on chip, on values shifted
 * by the row's first element; rows split over CTAs merge their (n, mean, M2)
 * with Chan's formula.
 *   x, y [M, H], gamma, beta [H], all of dtype dt; y == x is allowed, any
 *   other overlap of y with x, gamma or beta -> OSR_ERR_ALIAS.
 */
osr_status osr_layernorm_fwd(const void *x, const void *gamma, const void *beta, float eps,
                             void *y, int64_t M, int64_t H, osr_dtype dt, void *stream);

/*
 * Row softmax: y[i, :] = softmax(x[i, :]).
 *   x  [M, N] dtype in_dt, read only
 *   y  [M, N] dtype out_dt, written
 * Any in_dt/out_dt pair of OSR_F32/OSR_BF16.  y == x is allowed when
 * in_dt == out_dt (in place); any other overlap -> OSR_ERR_ALIAS.
 * Entries equal to -inf give 0; a row of only -inf gives NaN; a NaN or +inf
 * entry makes its row NaN.
 */
osr_status osr_softmax_rows(const void *x, void *y, int64_t M, int64_t N,
                            osr_dtype in_dt, osr_dtype out_dt, void *stream);

/*
 * Row softmax that also returns each row's normaliser statistics:
 *   row_max [M] binary32: m_i = max_j x[i, j] (exact), may be NULL
 *   row_sum [M] binary32: d_i = sum_j exp(x[i, j] - m_i), may be NULL
 * so that log(sum_j exp(x[i, j])) = m_i + log(d_i).  Other arguments and
 * rules as osr_softmax_rows; row_max/row_sum must not overlap x or y.
 */
osr_status osr_softmax_rows_stats(const void *x, void *y, float *row_max, float *row_sum,
                                  int64_t M, int64_t N, osr_dtype in_dt, osr_dtype out_dt,
                                  void *stream);

/*
 * Device-side fault report.  The staged softmax tier (16-byte rows longer
 * than one CTA holds) waits for its bulk copies into shared memory (bound:
 * 1 s) and for the other CTAs' (m, d) states (bound: 2 s); if a wait ever
 * runs out, the kernel records the fault in a device word (bit 0: copies,
 * bit 1: states), skips its stores and exits normally, so the context stays
 * usable.  The other cluster kernels (the register cluster tier of every
 * row op, log-sum-exp, top-k) bound their state exchanges the same way and
 * report a time-out in their outputs instead: NaN values, -1 indices.
 * This call synchronises `stream`, copies the word to *fault (0 = none),
 * clears it, and returns OSR_ERR_DEVICE_TIMEOUT if it was set, OSR_OK if not
 * (OSR_ERR_INVALID for a NULL fault pointer, OSR_ERR_CUDA on a CUDA error).
 * The word is per device and shared by all streams of the process.
 */
osr_status osr_device_fault(void *stream, int *fault);

/*
 * Row log-softmax: y[i, j] = (x[i, j] - m_i) - log d_i with m_i and d_i the
 * row's normaliser statistics, computed by the same kernels (and dispatcher)
 * as osr_softmax_rows.  Arguments, dtypes, in-place and alias rules as
 * osr_softmax_rows.  -inf entries give -inf; a NaN entry makes its row NaN.
 * The logarithm of the safe softmax of "RMSNorm、Softmax 与在线归约",
 * "稳定 Softmax：归一化之前先减最大值", written so that every intermediate is as
 * small as the result.
 */
osr_status osr_log_softmax_rows(const void *x, void *y, int64_t M, int64_t N, osr_dtype in_dt,
                                osr_dtype out_dt, void *stream);

/*
 * Per-row sampling statistics without writing the probabilities:
 *   lse    [M] binary32: log(sum_j exp(x[i, j])) = m_i + log d_i, may be NULL
 *   argmax [M] int64:    the first j with x[i, j] = m_i, may be NULL
 * (at least one of the two non-NULL).  Reads each row once; nothing else is
 * written.  "Softmax 与归一化" (anrans.github.io), exercise 2 "大词表采样":
 * greedy sampling needs only the argmax, so the softmax row need not be
 * produced.  NaN entries are skipped by the maximum (and make lse NaN); a
 * row of only -inf gives lse = -inf and argmax = -1.  x may have any dtype
 * of osr_dtype; lse/argmax must not overlap x or each other.
 */
osr_status osr_row_logsumexp(const void *x, float *lse, int64_t *argmax, int64_t M, int64_t N,
                             osr_dtype in_dt, void *stream);

/*
 * Top-k sampling prologue of each row, from one read of the row
 * ("Softmax 与归一化" (anrans.github.io), exercise 2 "大词表采样": top-k
 * sampling takes the k largest logits first and the softmax of only those):
 *   values  [M][k] binary32: the k largest x[i, :], largest first; equal
 *                            values in increasing column order; a NaN ranks
 *                            above every number, -0 and +0 are equal
 *   indices [M][k] int64:    their column indices
 *   probs   [M][k] binary32: exp(values[t] - values[0]) / sum_s exp(values[s] -
 *                            values[0]) over the k, may be NULL
 *   lse     [M] binary32:    log(sum_j exp(x[i, j])) of the whole row, as
 *                            osr_row_logsumexp, may be NULL
 * x: [M][N] row-major, dtype in_dt (any of osr_dtype), any alignment (16-byte
 * aligned rows with N a multiple of 16 bytes take the vector loads).  Values
 * are the row's own values converted exactly to binary32; the selection is
 * exact (no rounding decides it), so values and indices are unique.
 * Limits: 1 <= k <= min(N, 1024) (k > N: OSR_ERR_INVALID, k > 1024:
 * OSR_ERR_UNSUPPORTED); a row must fit 16 CTAs' shared memory (192 KiB of
 * elements each: N <= 1.5 Mi bfloat16 or 786 Ki binary32) and N < 2^31,
 * else OSR_ERR_UNSUPPORTED.  Outputs must not overlap x or each other
 * (OSR_ERR_ALIAS).  All buffers are caller-owned (see the conventions);
 * the call is asynchronous on `stream` and allocates nothing.
 */
osr_status osr_row_topk(const void *x, float *values, int64_t *indices, float *probs, float *lse,
                        int64_t M, int64_t N, int64_t k, osr_dtype in_dt, void *stream);

/* Static description of a status code (never NULL). */
const char *osr_status_string(osr_status s);

/* cudaError_t value recorded by the most recent OSR_ERR_CUDA on the calling
 * thread (0 if none). */
int osr_last_cuda_error(void);

/*
 * Which kernel the length-based dispatcher picks, without touching a GPU.
 *   op        0 = RMSNorm, 1 = fused residual-add + RMSNorm, 2 = softmax,
 *             3 = log-softmax, 4 = log-sum-exp / argmax, 5 = LayerNorm,
 *             6 = top-k (the geometry for k = 64; k sizes only the sort)
 *   vec_ok    1 if every buffer is 16-byte aligned (the 128-bit path)
 *   sm_count  streaming multiprocessors of the target device (152 on GB300);
 *             the plan assumes 228 KiB of shared memory per SM (GB300), where
 *             the compute entry points read the current device's figure
 *   buf       receives a NUL-terminated description, e.g.
 *             "rows g=256 ept=16 vec" or "cluster cs=10 g=1024 ept=16 vec"
 * Honours a plan forced with osr_test_force_kernel (osr_test.h) exactly as
 * the compute entry points do.  Returns OSR_ERR_INVALID on bad arguments.
 */
osr_status osr_plan_describe(int op, int64_t M, int64_t N, osr_dtype in_dt, osr_dtype out_dt,
                             int vec_ok, int sm_count, char *buf, size_t buf_len);

/*
 * Row softmax that allocates nothing.
 *
 * No page this library follows has a counterpart of this call; it exists for
 * callers that cannot allocate device memory while they run: serving loops
 * that freeze their memory footprint after start-up, programs on devices or
 * drivers without stream-ordered memory pools
 * (cudaDevAttrMemoryPoolsSupported == 0), and code running inside another
 * allocator's callbacks, where calling an allocator again can deadlock.
 * osr_softmax_rows may take a small workspace from cudaMallocAsync; this call
 * never calls cudaMalloc*, cudaFree* or any allocating routine.
 *
 * It computes what osr_softmax_rows computes (same arguments, dtypes,
 * in-place and alias rules, same results within rounding) with the two-pass
 * split-row kernels, keeping each row's per-piece (m, d) partials in one
 * fixed device array of OSR_NOALLOC_MAX_PARTIALS pairs (8 bytes each,
 * 512 KiB) compiled into the library.  Every GPU that loads the library holds
 * that array until the process exits.
 *   - M may be at most OSR_NOALLOC_MAX_PARTIALS; larger M returns
 *     OSR_ERR_UNSUPPORTED before any device work.  Rows are cut into fewer
 *     pieces when needed so that M x pieces fits the array (only for very
 *     large inputs: more than 32768 rows, each longer than 165 KB); each
 *     launch then takes more rows, whose second read may partly miss L2.
 *   - Buffers: device, managed or mapped page-locked host memory, exactly
 *     as osr_softmax_rows accepts them.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  The address is kept for the life of the
 *     process: it does not survive cudaDeviceReset or a switch to another
 *     primary context on that device, after which this call must not be
 *     used.
 *   - All calls share the one array and it keeps whatever the last call
 *     wrote.  Nothing in it needs to start at zero: every slot a call reads
 *     is written earlier in the same call.  Calls whose work overlaps on the
 *     GPU (different streams, or different host threads on one device
 *     without ordering between them) race on the array and may return wrong
 *     results; order them on one stream or with events.
 *   - A CUDA failure returns OSR_ERR_CUDA; osr_last_cuda_error() does not
 *     report the code for this call.
 */
#define OSR_NOALLOC_MAX_PARTIALS 65536
osr_status osr_softmax_rows_noalloc(const void *x, void *y, int64_t M, int64_t N,
                                    osr_dtype in_dt, osr_dtype out_dt, void *stream);

/* Library version, major * 10000 + minor * 100 + patch. */
int osr_version(void);

#ifdef __cplusplus
}
#endif

#endif /* OSR_H */
