/*
 * Oracle for MFA decode attention -- TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline leg (and its
 * reference arm) may load or call this file.  It shares no code, header, table
 * or constant with the CUDA path.
 *
 * What it computes (Step-3, paperlayer.ai/abs/2507.19427v1, section 2 "Step-3
 * Model Card": MFA keeps many query heads over a factorised QK circuit; section
 * 5 "Model-System Co-design": 8-bit KV, intensity 128, rank 16,384, which fix
 * H=64 heads of width d=256 over ONE shared K head and ONE shared V head).
 * For every sequence b and query head h, over the tokens t of the paged cache:
 *
 *     k_t = K_pool[block_table[b][t / page]][t % page][:]      (V likewise)
 *     s_t = scale * sum_i q[b,h,i] * k_t[i]
 *     m   = max_t s_t,  p_t = exp(s_t - m),  l = sum_t p_t
 *     O[b,h,:] = sum_t p_t v_t / l,          lse[b,h] = m + ln(l)
 *
 * i.e. softmax(q K^T * scale) V written out plainly, in double precision, two
 * passes over the tokens, no splitting and no blocking.  Inputs are converted
 * exactly: bf16 -> double by bit placement; an FP8 e4m3 code -> double from the
 * OCP FP8 format definition (1 sign, 4 exponent bits with bias 7, 3 mantissa
 * bits, subnormals at exponent 0, NaN at S.1111.111, no infinities), times its
 * per-token fp32 scale (an exact product in double).
 *
 * A token range [t_begin, t_end) per sequence may be given (NULL = [0, len)):
 * this yields the partial results (O over the range, lse over the range) that
 * the split-KV step produces.  An empty range gives O = 0 and lse = -inf.
 *
 * mfa_oracle_combine() merges partials with the log-sum-exp rule:
 *     lse* = M + ln sum_s exp(lse_s - M),  M = max_s lse_s
 *     O    = sum_s exp(lse_s - lse*) O_s
 * (all partials -inf -> O = 0, lse = -inf).
 *
 * Threads split the independent (b, h) pairs; no arithmetic is reordered.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

static double bf16_to_double(uint16_t bits) {
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* OCP FP8 E4M3 ("fn" variant): value = (-1)^s * 2^(e-7) * (1 + m/8) for e > 0,
 * (-1)^s * 2^(-6) * (m/8) for e == 0; e == 15 && m == 7 is NaN. */
double mfa_oracle_e4m3_to_double(uint8_t code) {
    int s = (code >> 7) & 1;
    int e = (code >> 3) & 15;
    int m = code & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

typedef struct {
    int B, H, d, page, max_pages, kv_fp8;
    const uint16_t *q;
    const void *k_cache, *v_cache;
    const float *k_scale, *v_scale;
    const int32_t *block_table, *seq_lens, *t_begin, *t_end;
    double scale;
    double *out, *lse;
    int nthreads;
} job_t;

typedef struct {
    const job_t *job;
    int tid;
} worker_t;

/* Element i of the key (or value) row of token t of sequence b, as a double. */
static double kv_elem(const job_t *J, int which_v, int b, int t, int i) {
    int32_t blk = J->block_table[(size_t)b * J->max_pages + t / J->page];
    size_t row = (size_t)blk * J->page + (size_t)(t % J->page);
    if (J->kv_fp8) {
        const uint8_t *pool = (const uint8_t *)(which_v ? J->v_cache : J->k_cache);
        const float *sc = which_v ? J->v_scale : J->k_scale;
        return mfa_oracle_e4m3_to_double(pool[row * J->d + i]) * (double)sc[row];
    } else {
        const uint16_t *pool = (const uint16_t *)(which_v ? J->v_cache : J->k_cache);
        return bf16_to_double(pool[row * J->d + i]);
    }
}

static void one_head(const job_t *J, int b, int h, double *s) {
    int L = J->seq_lens[b];
    int t0 = J->t_begin ? J->t_begin[b] : 0;
    int t1 = J->t_end ? J->t_end[b] : L;
    double *o = J->out + ((size_t)b * J->H + h) * J->d;
    const uint16_t *qh = J->q + ((size_t)b * J->H + h) * J->d;
    for (int i = 0; i < J->d; ++i) o[i] = 0.0;
    if (t1 <= t0) {
        J->lse[(size_t)b * J->H + h] = -INFINITY;
        return;
    }
    /* pass 1: scores and their maximum */
    double m = -INFINITY;
    for (int t = t0; t < t1; ++t) {
        double acc = 0.0;
        for (int i = 0; i < J->d; ++i) acc += bf16_to_double(qh[i]) * kv_elem(J, 0, b, t, i);
        s[t - t0] = J->scale * acc;
        if (s[t - t0] > m) m = s[t - t0];
    }
    /* pass 2: exponentials, their sum, and the weighted sum of values */
    double l = 0.0;
    for (int t = t0; t < t1; ++t) {
        double p = exp(s[t - t0] - m);
        l += p;
        for (int i = 0; i < J->d; ++i) o[i] += p * kv_elem(J, 1, b, t, i);
    }
    for (int i = 0; i < J->d; ++i) o[i] /= l;
    J->lse[(size_t)b * J->H + h] = m + log(l);
}

static void *worker(void *arg) {
    const worker_t *W = (const worker_t *)arg;
    const job_t *J = W->job;
    int maxlen = 1;
    for (int b = 0; b < J->B; ++b) {
        int t0 = J->t_begin ? J->t_begin[b] : 0;
        int t1 = J->t_end ? J->t_end[b] : J->seq_lens[b];
        if (t1 - t0 > maxlen) maxlen = t1 - t0;
    }
    double *s = (double *)malloc(sizeof(double) * (size_t)maxlen);
    if (!s) return (void *)1;
    long npairs = (long)J->B * J->H;
    for (long pidx = W->tid; pidx < npairs; pidx += J->nthreads)
        one_head(J, (int)(pidx / J->H), (int)(pidx % J->H), s);
    free(s);
    return NULL;
}

int mfa_oracle_num_cpus(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/*
 * Returns 0 on success, -1 on a bad argument, -2 on allocation failure.
 * q: bf16 bits [B,H,d]; k_cache/v_cache: bf16 bits or e4m3 codes [num_blocks,page,d];
 * k_scale/v_scale: fp32 [num_blocks,page] (FP8 only); block_table: int32 [B,max_pages];
 * seq_lens: int32 [B]; t_begin/t_end: int32 [B] or NULL; out: double [B,H,d]; lse: double [B,H].
 * nthreads <= 0 uses every online CPU.
 */
int mfa_oracle_decode(int B, int H, int d, int page, int max_pages, int kv_fp8,
                      const uint16_t *q, const void *k_cache, const void *v_cache,
                      const float *k_scale, const float *v_scale,
                      const int32_t *block_table, const int32_t *seq_lens,
                      const int32_t *t_begin, const int32_t *t_end,
                      double scale, double *out, double *lse, int nthreads) {
    if (B < 0 || H <= 0 || d <= 0 || page <= 0 || max_pages <= 0) return -1;
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !out || !lse) return -1;
    if (kv_fp8 && (!k_scale || !v_scale)) return -1;
    for (int b = 0; b < B; ++b) {
        int L = seq_lens[b];
        int t0 = t_begin ? t_begin[b] : 0;
        int t1 = t_end ? t_end[b] : L;
        if (L < 0 || L > max_pages * page || t0 < 0 || t1 > L) return -1;
    }
    job_t J = {B, H, d, page, max_pages, kv_fp8, q, k_cache, v_cache, k_scale, v_scale,
               block_table, seq_lens, t_begin, t_end, scale, out, lse, 0};
    if (nthreads <= 0) nthreads = mfa_oracle_num_cpus();
    long npairs = (long)B * H;
    if (npairs == 0) return 0;
    if (nthreads > npairs) nthreads = (int)npairs;
    J.nthreads = nthreads;
    worker_t *ws = (worker_t *)calloc((size_t)nthreads, sizeof(worker_t));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!ws || !th) {
        free(ws);
        free(th);
        return -2;
    }
    int rc = 0;
    for (int k = 0; k < nthreads; ++k) {
        ws[k].job = &J;
        ws[k].tid = k;
    }
    for (int k = 1; k < nthreads; ++k)
        if (pthread_create(&th[k], NULL, worker, &ws[k]) != 0) rc = -2;
    if (worker(&ws[0]) != NULL) rc = -2;
    for (int k = 1; k < nthreads; ++k) {
        void *r = NULL;
        pthread_join(th[k], &r);
        if (r != NULL) rc = -2;
    }
    free(ws);
    free(th);
    return rc;
}

/*
 * Log-sum-exp merge of S partial results per (row, head).
 * part_o: double [S, R, d]; part_lse: double [S, R]; out: double [R, d]; lse: double [R].
 * R counts (sequence, head) rows.
 */
int mfa_oracle_combine(int S, long R, int d, const double *part_o, const double *part_lse,
                       double *out, double *lse) {
    if (S < 0 || R < 0 || d <= 0 || !part_o || !part_lse || !out || !lse) return -1;
    for (long r = 0; r < R; ++r) {
        double M = -INFINITY;
        for (int s = 0; s < S; ++s)
            if (part_lse[(size_t)s * R + r] > M) M = part_lse[(size_t)s * R + r];
        double *o = out + (size_t)r * d;
        for (int i = 0; i < d; ++i) o[i] = 0.0;
        if (M == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double tot = 0.0;
        for (int s = 0; s < S; ++s) tot += exp(part_lse[(size_t)s * R + r] - M);
        double L = M + log(tot);
        for (int s = 0; s < S; ++s) {
            double w = exp(part_lse[(size_t)s * R + r] - L);
            const double *os = part_o + ((size_t)s * R + r) * d;
            for (int i = 0; i < d; ++i) o[i] += w * os[i];
        }
        lse[r] = L;
    }
    return 0;
}
