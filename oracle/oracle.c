/*
 * oracle.c -- plain, slow, fp64 CPU oracle for the row-wise
 * reduce-then-rescale operations: RMSNorm, fused residual-add + RMSNorm and
 * safe softmax.
 *
 * TEST INFRASTRUCTURE. Only the test-suite, the smoke check and the timed
 * CPU-baseline leg of the benchmark load the library built from this file.
 * The CUDA library never calls it, and the two share no source, header,
 * table or helper.  Every function here is a direct restatement of a
 * definition printed on the pages cited beside it; nothing is blocked, fused
 * or reordered beyond what that definition states.  All arithmetic is IEEE
 * binary64; the only narrowing is the explicit, single rounding of a binary64
 * result to the storage type (binary32 or bfloat16), round-to-nearest-even.
 *
 * Pages cited (by title and section):
 *   [KJ]  "RMSNorm、Softmax 与在线归约" (notes.kuangjux.top)
 *   [DY]  "两个融合算子：RMSNorm 与 online softmax" (daleiyang.github.io)
 *   [AZ]  "GPU Kernel 工程（04）：共享内存与 reduction——softmax、LayerNorm
 *          与 online softmax" (arganzheng.life)
 *   [AR]  "Softmax 与归一化", CUDA 进阶手册 (anrans.github.io)
 *   [LL]  "第23讲：为什么Attention必须先算Max？" (lilinji.mintlify.site)
 *
 * Storage types: 0 = binary32, 1 = bfloat16 (the upper 16 bits of a binary32).
 * Every function takes rows stored contiguously, row-major, row stride equal
 * to the row length, and writes binary64 results.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_F32 0
#define ORC_BF16 1

static int g_threads = 1;

/* Number of host threads used over rows (rows are independent, so this does
 * not change any result). */
void orc_set_threads(int n) { g_threads = n > 0 ? n : 1; }
int orc_get_threads(void) { return g_threads; }

/* Value of element i of a binary32 or bfloat16 array, exactly, as binary64. */
static double elem(const void *p, int dt, int64_t i) {
    if (dt == ORC_F32) return (double)((const float *)p)[i];
    uint32_t u = (uint32_t)((const uint16_t *)p)[i] << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a binary64 value once, to nearest with ties to even, to bfloat16
 * (8 significant bits, exponent range of binary32).  Returns the 16-bit
 * pattern.  Near v the bfloat16 values are spaced 2^(e-8), where
 * v = f * 2^e with 0.5 <= |f| < 1; below the normal range (e < -125) the
 * spacing stays at the subnormal quantum 2^-133. */
uint16_t orc_round_bf16(double v) {
    if (isnan(v)) return 0x7FC0;
    if (isinf(v)) return v < 0 ? 0xFF80 : 0x7F80;
    if (v == 0.0) return signbit(v) ? 0x8000 : 0x0000;
    int e;
    frexp(v, &e);
    if (e < -125) e = -125;
    double q = ldexp(1.0, e - 8);
    double r = nearbyint(v / q) * q; /* default rounding mode: ties to even */
    if (fabs(r) >= 0x1p128) return v < 0 ? 0xFF80 : 0x7F80;
    float f = (float)r; /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* Round a binary64 value once to the storage type and return that stored
 * value as binary64. */
static double round_to(double v, int dt) {
    if (dt == ORC_F32) return (double)(float)v;
    uint32_t u = (uint32_t)orc_round_bf16(v) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Store n binary64 values into a binary32 or bfloat16 array, each rounded
 * once to nearest-even. */
void orc_round_array(const double *v, int64_t n, int dt, void *out) {
    for (int64_t i = 0; i < n; ++i) {
        if (dt == ORC_F32)
            ((float *)out)[i] = (float)v[i];
        else
            ((uint16_t *)out)[i] = orc_round_bf16(v[i]);
    }
}

/* RMSNorm of one row, definition of [KJ] "RMSNorm 归约什么" and [AZ] 八.1:
 *   r = (mean_j x_j^2 + eps)^(-1/2),   y_j = x_j * r * gamma_j
 * eps sits inside the square root; the mean divides by H.  `h` holds the row
 * as binary64. */
static void rmsnorm_row(const double *h, const void *gamma, int dt, double eps,
                        int64_t H, double *y, double *rstd) {
    double ss = 0.0;
    for (int64_t j = 0; j < H; ++j) ss += h[j] * h[j];
    double r = 1.0 / sqrt(ss / (double)H + eps);
    for (int64_t j = 0; j < H; ++j) y[j] = h[j] * r * elem(gamma, dt, j);
    if (rstd) *rstd = r;
}

/* y[M][H] = RMSNorm(x) * gamma; rstd[M] (optional) = r of each row. */
void orc_rmsnorm(const void *x, const void *gamma, int dt, double eps, int64_t M,
                 int64_t H, double *y, double *rstd) {
#pragma omp parallel for schedule(static) num_threads(g_threads)
    for (int64_t i = 0; i < M; ++i) {
        double *h = y + i * H; /* the row is widened into its output slot */
        for (int64_t j = 0; j < H; ++j) h[j] = elem(x, dt, i * H + j);
        rmsnorm_row(h, gamma, dt, eps, H, h, rstd ? rstd + i : 0);
    }
}

/* Fused residual-add + RMSNorm, [AZ] 八.3 and [AR] "RMSNorm" fused variant:
 *   h = x + residual          (stored back as the new residual, rounded once
 *                              to the storage type)
 *   out = RMSNorm(h) * gamma  (of the stored, rounded h)
 * h_out[M][H] receives the new residual (values exactly representable in the
 * storage type), y[M][H] the normalised output before its final rounding. */
void orc_fused_add_rmsnorm(const void *x, const void *residual, const void *gamma,
                           int dt, double eps, int64_t M, int64_t H, double *h_out,
                           double *y, double *rstd) {
#pragma omp parallel for schedule(static) num_threads(g_threads)
    for (int64_t i = 0; i < M; ++i) {
        double *h = h_out + i * H;
        for (int64_t j = 0; j < H; ++j)
            h[j] = round_to(elem(x, dt, i * H + j) + elem(residual, dt, i * H + j), dt);
        rmsnorm_row(h, gamma, dt, eps, H, y + i * H, rstd ? rstd + i : 0);
    }
}

/* LayerNorm, two-pass definition of [AR] "LayerNorm 与 RMSNorm" and [AZ] 八.2:
 *   mu = (1/H) sum_j x_j,  var = (1/H) sum_j (x_j - mu)^2,
 *   y_j = (x_j - mu) / sqrt(var + eps) * gamma_j + beta_j.
 * mean_out/rstd_out (optional) receive mu and 1/sqrt(var + eps) per row. */
void orc_layernorm(const void *x, const void *gamma, const void *beta, int dt, double eps,
                   int64_t M, int64_t H, double *y, double *mean_out, double *rstd_out) {
#pragma omp parallel for schedule(static) num_threads(g_threads)
    for (int64_t i = 0; i < M; ++i) {
        double mu = 0.0;
        for (int64_t j = 0; j < H; ++j) mu += elem(x, dt, i * H + j);
        mu /= (double)H;
        double var = 0.0;
        for (int64_t j = 0; j < H; ++j) {
            const double c = elem(x, dt, i * H + j) - mu;
            var += c * c;
        }
        var /= (double)H;
        const double r = 1.0 / sqrt(var + eps);
        for (int64_t j = 0; j < H; ++j)
            y[i * H + j] = (elem(x, dt, i * H + j) - mu) * r * elem(gamma, dt, j) + elem(beta, dt, j);
        if (mean_out) mean_out[i] = mu;
        if (rstd_out) rstd_out[i] = r;
    }
}

/* Welford's running (n, mean, M2), one element at a time ([AZ] 八.2):
 *   n <- n + 1,  delta = x - mean,  mean <- mean + delta / n,
 *   M2 <- M2 + delta * (x - mean)   (with the updated mean).
 * Returns the state after all N elements of row i, M2 = sum (x - mean)^2. */
void orc_welford(const void *x, int dt, int64_t M, int64_t N, double *n_out, double *mean_out,
                 double *m2_out) {
    for (int64_t i = 0; i < M; ++i) {
        double n = 0.0, mean = 0.0, m2 = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            const double v = elem(x, dt, i * N + j);
            n += 1.0;
            const double delta = v - mean;
            mean += delta / n;
            m2 += delta * (v - mean);
        }
        n_out[i] = n;
        mean_out[i] = mean;
        m2_out[i] = m2;
    }
}

/* Chan et al.'s merge of two (n, mean, M2) states ([AZ] 八.2):
 *   n = na + nb,  delta = mean_b - mean_a,  mean = mean_a + delta nb / n,
 *   M2 = M2_a + M2_b + delta^2 na nb / n. */
void orc_chan_merge(double na, double ma, double qa, double nb, double mb, double qb, double *n,
                    double *mean, double *m2) {
    const double nn = na + nb;
    const double delta = mb - ma;
    *n = nn;
    *mean = ma + delta * nb / nn;
    *m2 = qa + qb + delta * delta * na * nb / nn;
}

/* Passes 1 and 2 of the three-pass safe softmax of [KJ] "稳定 Softmax" and
 * [AZ] 七.2 for row i: m = max_j x_j (and the first j where it occurs),
 * d = sum_j exp(x_j - m). */
static void row_max_sum(const void *x, int dt, int64_t i, int64_t N, double *m_out,
                        double *d_out, int64_t *at_out) {
    double m = -INFINITY;
    int64_t at = -1;
    for (int64_t j = 0; j < N; ++j) {
        double v = elem(x, dt, i * N + j);
        if (v > m) {
            m = v;
            at = j;
        }
    }
    double d = 0.0;
    for (int64_t j = 0; j < N; ++j) d += exp(elem(x, dt, i * N + j) - m);
    *m_out = m;
    *d_out = d;
    if (at_out) *at_out = at;
}

/* Safe softmax, three passes, [KJ] "稳定 Softmax" and [AZ] 七.2:
 *   m = max_j x_j,  d = sum_j exp(x_j - m),  y_i = exp(x_i - m) / d.
 * m_out/d_out (optional) receive m and d of each row. */
void orc_softmax(const void *x, int dt, int64_t M, int64_t N, double *y,
                 double *m_out, double *d_out) {
#pragma omp parallel for schedule(static) num_threads(g_threads)
    for (int64_t i = 0; i < M; ++i) {
        double m, d;
        row_max_sum(x, dt, i, N, &m, &d, 0);
        for (int64_t j = 0; j < N; ++j) y[i * N + j] = exp(elem(x, dt, i * N + j) - m) / d;
        if (m_out) m_out[i] = m;
        if (d_out) d_out[i] = d;
    }
}

/* Log-softmax: log y_i = (x_i - m) - log d with m and d of the three-pass
 * definition (the logarithm of [KJ] "稳定 Softmax"; [AR] "Online softmax"
 * notes that consumers such as samplers need only the statistics).  Written
 * as (x_i - m) - log d so every intermediate is as small as the result. */
void orc_log_softmax(const void *x, int dt, int64_t M, int64_t N, double *y) {
#pragma omp parallel for schedule(static) num_threads(g_threads)
    for (int64_t i = 0; i < M; ++i) {
        double m, d;
        row_max_sum(x, dt, i, N, &m, &d, 0);
        const double ld = log(d);
        for (int64_t j = 0; j < N; ++j) y[i * N + j] = (elem(x, dt, i * N + j) - m) - ld;
    }
}

/* Row statistics a sampler needs without the probabilities: the
 * log-sum-exp m + log d and the index of the row maximum (the first one on
 * ties).  [AR] exercise 2 "大词表采样": greedy sampling needs only the
 * argmax, so the full row of probabilities need not be written. */
void orc_logsumexp_argmax(const void *x, int dt, int64_t M, int64_t N, double *lse,
                          int64_t *argmax) {
#pragma omp parallel for schedule(static) num_threads(g_threads)
    for (int64_t i = 0; i < M; ++i) {
        double m, d;
        int64_t at;
        row_max_sum(x, dt, i, N, &m, &d, &at);
        if (lse) lse[i] = m + log(d);
        if (argmax) argmax[i] = at;
    }
}

/* Online normaliser, one element at a time, [KJ] "Online Softmax 为什么要重缩放
 * 旧的和" and [AR] "Online softmax": start from the first element as (x_1, 1);
 * for each further x:  m' = max(m, x),  d <- d * exp(m - m') + exp(x - m'),
 * m <- m'.  Then y_i = exp(x_i - m) / d.  Defined for non-empty finite rows. */
void orc_softmax_online(const void *x, int dt, int64_t M, int64_t N, double *y,
                        double *m_out, double *d_out) {
#pragma omp parallel for schedule(static) num_threads(g_threads)
    for (int64_t i = 0; i < M; ++i) {
        double m = elem(x, dt, i * N), d = 1.0;
        for (int64_t j = 1; j < N; ++j) {
            double v = elem(x, dt, i * N + j);
            double mn = v > m ? v : m;
            d = d * exp(m - mn) + exp(v - mn);
            m = mn;
        }
        for (int64_t j = 0; j < N; ++j) y[i * N + j] = exp(elem(x, dt, i * N + j) - m) / d;
        if (m_out) m_out[i] = m;
        if (d_out) d_out[i] = d;
    }
}

/* Merge of two (m, d) summaries, [DY] §5·三 "结合律" and [KJ] "从逐元素更新到
 * 合并两个 tile":  m = max(m1, m2),  d = d1 * exp(m1 - m) + d2 * exp(m2 - m). */
void orc_md_merge(double m1, double d1, double m2, double d2, double *m, double *d) {
    double mm = m1 > m2 ? m1 : m2;
    *m = mm;
    *d = d1 * exp(m1 - mm) + d2 * exp(m2 - mm);
}

/* Row statistics by chunk summaries, [DY] §4·四 "S4": each run of `chunk`
 * consecutive elements is summarised on its own (its max, then the sum of
 * exp(x - that max)), and the summaries are merged left to right with the
 * (m, d) merge above.  Used only to check that chunking does not change the
 * statistics. */
void orc_softmax_chunked_stats(const void *x, int dt, int64_t M, int64_t N,
                               int64_t chunk, double *m_out, double *d_out) {
#pragma omp parallel for schedule(static) num_threads(g_threads)
    for (int64_t i = 0; i < M; ++i) {
        double m = -INFINITY, d = 0.0;
        int first = 1;
        for (int64_t c0 = 0; c0 < N; c0 += chunk) {
            int64_t c1 = c0 + chunk < N ? c0 + chunk : N;
            double cm = -INFINITY;
            for (int64_t j = c0; j < c1; ++j) {
                double v = elem(x, dt, i * N + j);
                if (v > cm) cm = v;
            }
            double cd = 0.0;
            for (int64_t j = c0; j < c1; ++j) cd += exp(elem(x, dt, i * N + j) - cm);
            if (first) {
                m = cm;
                d = cd;
                first = 0;
            } else {
                orc_md_merge(m, d, cm, cd, &m, &d);
            }
        }
        m_out[i] = m;
        d_out[i] = d;
    }
}

/* Top-k sampling prologue of a row, [AR] exercise 2 ("大词表采样": sampling
 * needs no full softmax -- greedy needs the argmax, top-k picks the k largest
 * logits first and takes the softmax of those):
 *   order: element a precedes b when x_a > x_b, or x_a == x_b and a < b
 *          (-0 and +0 are equal; a NaN ranks above every number);
 *   values[t], indices[t]: the t-th element of the row in that order, t < k;
 *   probs[t] = exp(values[t] - values[0]) / sum_{s<k} exp(values[s] - values[0]);
 *   lse (optional) = log sum_j exp(x_j) of the whole row, m + log d with the
 *   m and d of the three-pass softmax.
 * The order is the plain definition: the whole row is sorted (qsort) and the
 * first k taken. */
struct topk_item {
    double v;
    int64_t i;
};

static int topk_cmp(const void *pa, const void *pb) {
    const struct topk_item *a = (const struct topk_item *)pa, *b = (const struct topk_item *)pb;
    const int an = isnan(a->v), bn = isnan(b->v);
    if (an != bn) return an ? -1 : 1;
    if (!an && a->v != b->v) return a->v > b->v ? -1 : 1;
    return a->i < b->i ? -1 : (a->i > b->i ? 1 : 0);
}

void orc_topk(const void *x, int dt, int64_t M, int64_t N, int64_t k, double *values,
              int64_t *indices, double *probs, double *lse) {
#pragma omp parallel for schedule(dynamic) num_threads(g_threads)
    for (int64_t i = 0; i < M; ++i) {
        struct topk_item *it = (struct topk_item *)malloc((size_t)N * sizeof(struct topk_item));
        for (int64_t j = 0; j < N; ++j) {
            it[j].v = elem(x, dt, i * N + j);
            it[j].i = j;
        }
        qsort(it, (size_t)N, sizeof(struct topk_item), topk_cmp);
        double z = 0.0;
        for (int64_t t = 0; t < k; ++t) z += exp(it[t].v - it[0].v);
        for (int64_t t = 0; t < k; ++t) {
            values[i * k + t] = it[t].v;
            indices[i * k + t] = it[t].i;
            if (probs) probs[i * k + t] = exp(it[t].v - it[0].v) / z;
        }
        free(it);
        if (lse) {
            double m, d;
            row_max_sum(x, dt, i, N, &m, &d, 0);
            lse[i] = m + log(d);
        }
    }
}
