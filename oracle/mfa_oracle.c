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
 * Threads split independent (sequence, group of heads) units; each head's
 * arithmetic runs in the order written above.
 *
 * The attention designs the Step-3 page compares MFA with (section 5 "Model-System
 * Co-design", the "Attention Design" items; section 7's attention ablation) are the same
 * definition over other cache layouts, handled here by two more parameters:
 *   - G key/value heads per cache row (grouped-query attention): a cache row holds G heads
 *     of width d side by side, and query head h reads head g(h) = h / (H / G), columns
 *     [g(h) d, (g(h) + 1) d) of the row, of both pools;
 *   - one latent shared by keys and values (MLA-style): v_cache NULL means every value row
 *     is the key row itself.
 * MFA is G = 1 with separate pools.
 *
 * 4-bit caches (MXFP4, the OCP Microscaling format): two E2M1 codes a byte and one E8M0
 * power-of-two scale per 32 consecutive elements of a row; decoded exactly, code value times
 * scale.
 *
 * mfa_oracle_kv_append() (end of file) writes a decode step's new key and value rows into
 * the paged cache, quantising them to e4m3 with per-row scales for an FP8 cache, or to MXFP4.
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
/* OCP MX FP4 E2M1 (low nibble of code): value = (-1)^s * 2^(e-1) * (1 + m/2) for e > 0,
 * (-1)^s * m/2 for e == 0 (1 sign, 2 exponent bits with bias 1, 1 mantissa bit; no
 * infinities or NaN): magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double mfa_oracle_e2m1_to_double(uint8_t code) {
    int s = (code >> 3) & 1;
    int e = (code >> 1) & 3;
    int m = code & 1;
    double v = (e == 0) ? (double)m / 2.0 : ldexp(1.0 + (double)m / 2.0, e - 1);
    return s ? -v : v;
}

/* OCP MX E8M0 scale: 2^(e - 127), e = 255 is NaN. */
double mfa_oracle_e8m0_to_double(uint8_t e) {
    if (e == 255) return NAN;
    return ldexp(1.0, (int)e - 127);
}

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
    int B, H, G, d, page, max_pages, kv_fmt;   /* kv_fmt: 0 bf16, 1 e4m3, 2 MXFP4 */
    const uint16_t *q;
    const void *k_cache, *v_cache;
    const void *k_scale, *v_scale;
    const int32_t *block_table, *seq_lens, *t_begin, *t_end;
    double scale;
    double *out, *lse;
    int nthreads;
} job_t;

typedef struct {
    const job_t *job;
    int tid;
} worker_t;

/* Head groups: the heads of a sequence are split into groups of HEAD_GROUP so
 * that the threads have independent work; a group decodes each key and value row
 * once and uses it for its heads (all of which read the same key/value head). */
#define HEAD_GROUP 8

/* Key/value head g of the row of token t of sequence b (row width G d), decoded to
 * doubles; a shared latent (v_cache NULL) gives the key row for values too. */
static void kv_row(const job_t *J, int which_v, int b, int t, int g, double *dst) {
    int32_t blk = J->block_table[(size_t)b * J->max_pages + t / J->page];
    size_t row = (size_t)blk * J->page + (size_t)(t % J->page);
    size_t base = row * (size_t)J->G * (size_t)J->d + (size_t)g * (size_t)J->d;
    const void *vpool = J->v_cache ? J->v_cache : J->k_cache;
    if (J->kv_fmt == 1) {
        const uint8_t *pool = (const uint8_t *)(which_v ? vpool : J->k_cache);
        const float *sc = (const float *)(which_v && J->v_cache ? J->v_scale : J->k_scale);
        for (int i = 0; i < J->d; ++i)
            dst[i] = mfa_oracle_e4m3_to_double(pool[base + i]) * (double)sc[row];
    } else if (J->kv_fmt == 2) {
        /* MXFP4: element e of the row is E2M1 code (byte e / 2, low nibble for even e) times
         * the E8M0 scale of its block of 32, scale byte e / 32 of the row */
        const uint8_t *pool = (const uint8_t *)(which_v ? vpool : J->k_cache);
        const uint8_t *sc = (const uint8_t *)(which_v && J->v_cache ? J->v_scale : J->k_scale);
        const size_t rowlen = (size_t)J->G * (size_t)J->d;
        for (int i = 0; i < J->d; ++i) {
            const size_t e = (size_t)g * (size_t)J->d + (size_t)i;
            const uint8_t byte = pool[row * (rowlen / 2) + e / 2];
            const uint8_t code = (e & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
            dst[i] = mfa_oracle_e2m1_to_double(code) * mfa_oracle_e8m0_to_double(sc[row * (rowlen / 32) + e / 32]);
        }
    } else {
        const uint16_t *pool = (const uint16_t *)(which_v ? vpool : J->k_cache);
        for (int i = 0; i < J->d; ++i) dst[i] = bf16_to_double(pool[base + i]);
    }
}

typedef struct {
    double *s;    /* [HEAD_GROUP][maxlen] scores */
    double *q;    /* [HEAD_GROUP][d] */
    double *row;  /* [d] */
} scratch_t;

/* Heads [h0, h1) of sequence b over the token range of b. */
static void head_group(const job_t *J, int b, int h0, int h1, size_t maxlen, scratch_t *W) {
    int L = J->seq_lens[b];
    int t0 = J->t_begin ? J->t_begin[b] : 0;
    int t1 = J->t_end ? J->t_end[b] : L;
    int d = J->d;
    int g = h0 / (J->H / J->G);   /* the key/value head of every query head in [h0, h1) */
    for (int h = h0; h < h1; ++h) {
        double *o = J->out + ((size_t)b * J->H + h) * d;
        const uint16_t *qh = J->q + ((size_t)b * J->H + h) * d;
        for (int i = 0; i < d; ++i) {
            o[i] = 0.0;
            W->q[(size_t)(h - h0) * d + i] = bf16_to_double(qh[i]);
        }
        if (t1 <= t0) J->lse[(size_t)b * J->H + h] = -INFINITY;
    }
    if (t1 <= t0) return;
    /* pass 1: scores s_t = scale * q.k_t and their maximum per head */
    double m[HEAD_GROUP];
    for (int h = h0; h < h1; ++h) m[h - h0] = -INFINITY;
    for (int t = t0; t < t1; ++t) {
        kv_row(J, 0, b, t, g, W->row);
        for (int h = h0; h < h1; ++h) {
            const double *qv = W->q + (size_t)(h - h0) * d;
            double acc = 0.0;
            for (int i = 0; i < d; ++i) acc += qv[i] * W->row[i];
            double st = J->scale * acc;
            W->s[(size_t)(h - h0) * maxlen + (size_t)(t - t0)] = st;
            if (st > m[h - h0]) m[h - h0] = st;
        }
    }
    /* pass 2: p_t = exp(s_t - m), l = sum p_t, O = sum p_t v_t / l, lse = m + ln l */
    double l[HEAD_GROUP];
    for (int h = h0; h < h1; ++h) l[h - h0] = 0.0;
    for (int t = t0; t < t1; ++t) {
        kv_row(J, 1, b, t, g, W->row);
        for (int h = h0; h < h1; ++h) {
            double p = exp(W->s[(size_t)(h - h0) * maxlen + (size_t)(t - t0)] - m[h - h0]);
            l[h - h0] += p;
            double *o = J->out + ((size_t)b * J->H + h) * d;
            for (int i = 0; i < d; ++i) o[i] += p * W->row[i];
        }
    }
    for (int h = h0; h < h1; ++h) {
        double *o = J->out + ((size_t)b * J->H + h) * d;
        for (int i = 0; i < d; ++i) o[i] /= l[h - h0];
        J->lse[(size_t)b * J->H + h] = m[h - h0] + log(l[h - h0]);
    }
}

static void *worker(void *arg) {
    const worker_t *Wk = (const worker_t *)arg;
    const job_t *J = Wk->job;
    size_t maxlen = 1;
    for (int b = 0; b < J->B; ++b) {
        int t0 = J->t_begin ? J->t_begin[b] : 0;
        int t1 = J->t_end ? J->t_end[b] : J->seq_lens[b];
        if (t1 - t0 > (int)maxlen) maxlen = (size_t)(t1 - t0);
    }
    scratch_t W;
    W.s = (double *)malloc(sizeof(double) * maxlen * HEAD_GROUP);
    W.q = (double *)malloc(sizeof(double) * (size_t)J->d * HEAD_GROUP);
    W.row = (double *)malloc(sizeof(double) * (size_t)J->d);
    if (!W.s || !W.q || !W.row) {
        free(W.s);
        free(W.q);
        free(W.row);
        return (void *)1;
    }
    int per = J->H / J->G;                           /* query heads per key/value head */
    int hg = per < HEAD_GROUP ? per : HEAD_GROUP;     /* divides per (checked by the caller) */
    int groups = J->H / hg;
    long nunits = (long)J->B * groups;
    for (long u = Wk->tid; u < nunits; u += J->nthreads) {
        int b = (int)(u / groups), gi = (int)(u % groups);
        int h0 = gi * hg, h1 = h0 + hg;
        head_group(J, b, h0, h1, maxlen, &W);
    }
    free(W.s);
    free(W.q);
    free(W.row);
    return NULL;
}

int mfa_oracle_num_cpus(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/*
 * Returns 0 on success, -1 on a bad argument, -2 on allocation failure.
 * q: bf16 bits [B,H,d]; k_cache/v_cache by kv_fmt: 0 bf16 bits [num_blocks,page,G*d],
 * 1 e4m3 codes [num_blocks,page,G*d] with fp32 scales k_scale/v_scale [num_blocks,page],
 * 2 MXFP4 codes [num_blocks,page,G*d/2] (two a byte) with E8M0 scales [num_blocks,page,
 * G*d/32] (v_cache NULL: values are the key rows, v_scale unused); G divides H, and H / G is at most HEAD_GROUP
 * or a multiple of it; block_table: int32 [B,max_pages]; seq_lens: int32 [B];
 * t_begin/t_end: int32 [B] or NULL; out: double [B,H,d]; lse: double [B,H].
 * nthreads <= 0 uses every online CPU.
 */
int mfa_oracle_decode(int B, int H, int G, int d, int page, int max_pages, int kv_fmt,
                      const uint16_t *q, const void *k_cache, const void *v_cache,
                      const void *k_scale, const void *v_scale,
                      const int32_t *block_table, const int32_t *seq_lens,
                      const int32_t *t_begin, const int32_t *t_end,
                      double scale, double *out, double *lse, int nthreads) {
    if (B < 0 || H <= 0 || G <= 0 || H % G != 0 || d <= 0 || page <= 0 || max_pages <= 0) return -1;
    if (H / G > HEAD_GROUP && (H / G) % HEAD_GROUP != 0) return -1;
    if (!q || !k_cache || !block_table || !seq_lens || !out || !lse) return -1;
    if (kv_fmt < 0 || kv_fmt > 2) return -1;
    if (kv_fmt == 2 && (G * d) % 32 != 0) return -1;
    if (kv_fmt != 0 && (!k_scale || (v_cache && !v_scale))) return -1;
    for (int b = 0; b < B; ++b) {
        int L = seq_lens[b];
        int t0 = t_begin ? t_begin[b] : 0;
        int t1 = t_end ? t_end[b] : L;
        if (L < 0 || L > max_pages * page || t0 < 0 || t1 > L) return -1;
    }
    job_t J = {B, H, G, d, page, max_pages, kv_fmt, q, k_cache, v_cache, k_scale, v_scale,
               block_table, seq_lens, t_begin, t_end, scale, out, lse, 0};
    if (nthreads <= 0) nthreads = mfa_oracle_num_cpus();
    int hg = H / G < HEAD_GROUP ? H / G : HEAD_GROUP;
    long nunits = (long)B * (H / hg);
    if (nunits == 0) return 0;
    if (nthreads > nunits) nthreads = (int)nunits;
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

/* ------------------------------------------------------------------------------------------
 * KV-cache append with FP8 quantisation (the step before attention in a decode step: the
 * attention instances own and fill their KV caches, Step-3 page section 7 "Implementation
 * and Results"; the cache holds 8-bit KV, section 5 "Model-System Co-design").
 *
 * For every sequence b with positions[b] = t0 >= 0, its T new tokens' key rows
 * k_new[b*T + i][:] and value rows v_new[b*T + i][:] (bf16), i < T, go to position
 * t = t0 + i: slot t % page of page block_table[b][t / page]:
 *   - bf16 cache: the bf16 bits unchanged;
 *   - e4m3 cache: one fp32 scale per row, s = absmax / 448 (s = 1 for an all-zero row), and
 *     codes e4m3(x_i / s), x_i the row's bf16 values; both divisions are fp32 divisions
 *     rounded to nearest, and the e4m3 rounding is to the nearest value, ties to the even
 *     code, with magnitudes above 448 saturating to 448.
 * positions[b] < 0: no token for b (nothing written).  t >= max_pages * page, or a page id
 * outside [0, num_blocks): nothing written for that token, and bit 1 (position) or bit 0
 * (page id) of the return mask is set.
 */

static float bf16_to_float(uint16_t bits) {
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return f;
}

/* Nearest e4m3 value to y, found by trying every non-negative finite code (0x00..0x7E,
 * whose values increase with the code); of two equally near codes the even one wins.
 * |y| >= 448 gives 448.  The sign bit of y is kept, so a negative y that rounds to zero
 * gives 0x80.  y must not be NaN. */
uint8_t mfa_oracle_e4m3_from_float(float y) {
    const int neg = signbit(y) != 0;
    const double a = fabs((double)y);
    int best = 0x7E;
    if (a < 448.0) {
        double bd = a;   /* distance to code 0 (value 0) */
        best = 0;
        for (int c = 1; c <= 0x7E; ++c) {
            const double dist = fabs(mfa_oracle_e4m3_to_double((uint8_t)c) - a);
            if (dist < bd || (dist == bd && (c & 1) == 0)) {
                best = c;
                bd = dist;
            }
        }
    }
    return (uint8_t)(neg ? (0x80 | best) : best);
}

/* mfa_oracle_e4m3_from_float over an array (for the encoder's pins). */
void mfa_oracle_e4m3_from_float_array(const float *y, long n, uint8_t *codes) {
    for (long i = 0; i < n; ++i) codes[i] = mfa_oracle_e4m3_from_float(y[i]);
}

static void quantise_row(const uint16_t *x, int d, uint8_t *codes, float *scale) {
    float absmax = 0.0f;
    for (int i = 0; i < d; ++i) {
        const float a = fabsf(bf16_to_float(x[i]));
        if (a > absmax) absmax = a;
    }
    const float s = (absmax > 0.0f) ? absmax / 448.0f : 1.0f;
    for (int i = 0; i < d; ++i) codes[i] = mfa_oracle_e4m3_from_float(bf16_to_float(x[i]) / s);
    *scale = s;
}

/* Nearest E2M1 value to y (codes 0..7 increase in value); of two equally near codes the one
 * with an even code wins; |y| >= 6 gives 6.  The sign bit of y is kept (a negative y that
 * rounds to zero gives code 8).  y must not be NaN. */
uint8_t mfa_oracle_e2m1_from_double(double y) {
    const int neg = signbit(y) != 0;
    const double a = fabs(y);
    int best = 7;
    if (a < 6.0) {
        double bd = a;
        best = 0;
        for (int c = 1; c <= 7; ++c) {
            const double dist = fabs(mfa_oracle_e2m1_to_double((uint8_t)c) - a);
            if (dist < bd || (dist == bd && (c & 1) == 0)) {
                best = c;
                bd = dist;
            }
        }
    }
    return (uint8_t)(neg ? (8 | best) : best);
}

/* The OCP MX shared exponent of a block: floor(log2(amax)) minus E2M1's largest exponent
 * (2), clamped to E8M0's [-127, 127]; an all-zero block takes -127. */
int mfa_oracle_mx_block_exponent(const float *x, int n) {
    float amax = 0.0f;
    for (int i = 0; i < n; ++i)
        if (fabsf(x[i]) > amax) amax = fabsf(x[i]);
    if (amax == 0.0f) return -127;
    int E = 0;
    frexpf(amax, &E);               /* amax = f 2^E, f in [0.5, 1): floor(log2 amax) = E - 1 */
    int e = (E - 1) - 2;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

/* MXFP4 row: per block of 32, scale 2^e with e the shared exponent, codes E2M1(x / 2^e)
 * (an exact power-of-two scaling, then rounding to nearest even, saturating at 6). */
static void quantise_row_mx(const uint16_t *x, int d, uint8_t *codes, uint8_t *scales) {
    float blk[32];
    for (int b = 0; b < d / 32; ++b) {
        for (int i = 0; i < 32; ++i) blk[i] = bf16_to_float(x[32 * b + i]);
        const int e = mfa_oracle_mx_block_exponent(blk, 32);
        scales[b] = (uint8_t)(e + 127);
        for (int i = 0; i < 32; ++i) {
            const int j = 32 * b + i;
            const uint8_t c = mfa_oracle_e2m1_from_double(ldexp((double)blk[i], -e));
            if (j & 1)
                codes[j / 2] = (uint8_t)((codes[j / 2] & 0x0F) | (c << 4));
            else
                codes[j / 2] = (uint8_t)((codes[j / 2] & 0xF0) | c);
        }
    }
}

/*
 * k_new/v_new: bf16 bits [B*T,d]; positions: int32 [B]; block_table: int32 [B,max_pages];
 * k_cache/v_cache by kv_fmt (0 bf16, 1 e4m3, 2 MXFP4, layouts as mfa_oracle_decode's with
 * G = 1), updated in place; k_scale/v_scale: fp32 [num_blocks,page] (e4m3) or E8M0 bytes
 * [num_blocks,page,d/32] (MXFP4), updated in place.
 * Returns the error mask described above (0 = every row written or skipped by choice),
 * or -1 on a bad argument.
 */
int mfa_oracle_kv_append(int B, int T, int d, int page, int max_pages, int num_blocks, int kv_fmt,
                         const uint16_t *k_new, const uint16_t *v_new, const int32_t *positions,
                         const int32_t *block_table, void *k_cache, void *v_cache,
                         void *k_scale, void *v_scale) {
    if (B < 0 || T < 1 || d <= 0 || page <= 0 || max_pages <= 0 || num_blocks <= 0) return -1;
    if (!k_new || !v_new || !positions || !block_table || !k_cache || !v_cache) return -1;
    if (kv_fmt < 0 || kv_fmt > 2 || (kv_fmt == 2 && d % 32 != 0)) return -1;
    if (kv_fmt != 0 && (!k_scale || !v_scale)) return -1;
    int mask = 0;
    for (int x = 0; x < B * T; ++x) {
        const int b = x / T;
        if (positions[b] < 0) continue;
        const int t = positions[b] + x % T;
        if (t >= max_pages * page) {
            mask |= 2;
            continue;
        }
        const int blk = block_table[(size_t)b * max_pages + t / page];
        if (blk < 0 || blk >= num_blocks) {
            mask |= 1;
            continue;
        }
        const size_t row = (size_t)blk * page + (size_t)(t % page);
        if (kv_fmt == 1) {
            quantise_row(k_new + (size_t)x * d, d, (uint8_t *)k_cache + row * d, (float *)k_scale + row);
            quantise_row(v_new + (size_t)x * d, d, (uint8_t *)v_cache + row * d, (float *)v_scale + row);
        } else if (kv_fmt == 2) {
            quantise_row_mx(k_new + (size_t)x * d, d, (uint8_t *)k_cache + row * (d / 2),
                            (uint8_t *)k_scale + row * (d / 32));
            quantise_row_mx(v_new + (size_t)x * d, d, (uint8_t *)v_cache + row * (d / 2),
                            (uint8_t *)v_scale + row * (d / 32));
        } else {
            memcpy((uint16_t *)k_cache + row * d, k_new + (size_t)x * d, (size_t)d * sizeof(uint16_t));
            memcpy((uint16_t *)v_cache + row * d, v_new + (size_t)x * d, (size_t)d * sizeof(uint16_t));
        }
    }
    return mask;
}
