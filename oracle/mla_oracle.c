/*
 * mla_oracle.c -- FP64 CPU oracle for MLA decode attention over a paged FP8
 * latent-KV cache, and for the log-sum-exp merge of partial answers.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant
 * with the CUDA library.  It is deliberately plain and slow: every result is
 * the textbook definition written out in double precision, with no blocking,
 * fusion, splitting or reordering beyond what the definition states.
 *
 * Source of the method: the blog post "Kimi K3 on AMD Instinct MI355X: vLLM
 * serving ..." (three language editions of the same post).
 *   - Model section: each MLA layer keeps a compressed KV history that grows
 *     with the conversation, and every new query attends over all of it.
 *   - Section 1 "Cache" (DCP paragraph): a history may be cut into shards;
 *     each partial answer carries normalisation information and the partials
 *     are merged with softmax weights.  Worked figure: 24 layers x 142,000
 *     positions x 576 FP8 bytes ~ 1.96 GB per GPU, ~245 MB under DCP8.
 *   - Section 4 "MLA": every query head attends to the cached positions
 *     independently, so adding (padding) heads does not change another
 *     head's softmax; history partitions are work split inside one GPU and
 *     leave the KV storage unchanged.
 *   - Benchmark configuration section: the KV cache is FP8.
 *
 * Conventions the post leaves open, as read by this library (each one is also
 * listed in the design notes):
 *   - One cached position is 576 FP8 (OCP E4M3FN) codes: the first 512 are the
 *     compressed latent (which is also the value vector) and the last 64 the
 *     already-rotated positional part.  The query arrives absorbed: 576 bf16
 *     values per head.
 *   - One fp32 scale per tensor: x = decode(code) * kv_scale.
 *   - Pages of 64 positions; logical position p of request b lives in page
 *     block_table[b][p / 64], row p % 64.
 *   - seq_lens[b] counts the T new positions; query t (0-based) of request b
 *     sees positions p < seq_lens[b] - T + 1 + t (causal inside the draft).
 *   - lse is the natural logarithm of sum_p exp(score_p), with score_p
 *     already multiplied by sm_scale and built from scaled latents.
 *
 * Build:  gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared -pthread \
 *             -o libmla_oracle.so mla_oracle.c -lm
 * (-ffp-contract=off keeps x86-64 and aarch64 results bit-identical.)
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_PAGE 64
#define ORACLE_DQK 576
#define ORACLE_DV 512

/* ------------------------------------------------------------------ */
/* Number formats                                                       */
/* ------------------------------------------------------------------ */

/* OCP 8-bit floating point, E4M3FN variant: 1 sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits, no infinities; exponent 15 with mantissa 7 is NaN
 * (so the largest finite magnitude is 1.75 * 2^8 = 448).  Exponent 0 encodes
 * subnormals m/8 * 2^(1-7). */
double oracle_e4m3fn_to_double(uint8_t code)
{
    int sign = code >> 7;
    int e = (code >> 3) & 15;
    int m = code & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, 1 - 7);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32; widening is exact. */
static double bf16_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------ */
/* Decode attention                                                     */
/* ------------------------------------------------------------------ */

typedef struct {
    const uint16_t *q;          /* bf16 bits [B][T][H][576]                  */
    const uint8_t *kv;          /* e4m3fn codes [num_pages][64][576]          */
    int64_t num_pages;
    double kv_scale;
    const int32_t *block_table; /* [B][bt_stride]                             */
    int64_t bt_stride;
    const int32_t *seq_lens;    /* [B]                                        */
    int B, T, H;
    double sm_scale;
    const uint8_t *pos_mask;    /* optional [pos_mask_len]: 1 keeps position  */
    int64_t pos_mask_len;
    const uint8_t *row_mask;    /* optional [B][T][H]: 1 computes that row    */
    double *out;                /* [B][T][H][512]                             */
    double *lse;                /* [B][T][H]                                  */
    double lut[256];            /* decoded code values times kv_scale         */
    volatile int64_t next_unit; /* work counter over (b, t)                   */
    volatile int error;
} decode_job;

static int keep_position(const decode_job *J, int64_t p)
{
    if (!J->pos_mask)
        return 1;
    if (p >= J->pos_mask_len)
        return 0;
    return J->pos_mask[p] != 0;
}

static int row_wanted(const decode_job *J, int b, int t, int h)
{
    if (!J->row_mask)
        return 1;
    return J->row_mask[((int64_t)b * J->T + t) * J->H + h] != 0;
}

/* Address of the 576 codes of logical position p of request b. */
static const uint8_t *position_codes(const decode_job *J, int b, int64_t p, int *err)
{
    int32_t page = J->block_table[(int64_t)b * J->bt_stride + p / ORACLE_PAGE];
    if (page < 0 || page >= J->num_pages) {
        *err = 1;
        return NULL;
    }
    return J->kv + ((int64_t)page * ORACLE_PAGE + p % ORACLE_PAGE) * ORACLE_DQK;
}

/* One (request b, query position t) unit: all wanted heads.
 * Two passes over the visible positions (textbook two-pass softmax):
 *   pass 1: s_h(p) = sm_scale * sum_{d<576} q_h[d] * x_p[d], kept for all p;
 *   pass 2: M_h = max_p s_h(p), Z_h = sum_p exp(s_h(p) - M_h),
 *           out_h[d] = sum_p exp(s_h(p) - M_h) * x_p[d] / Z_h   (d < 512),
 *           lse_h = M_h + ln Z_h. */
static int decode_unit(decode_job *J, int b, int t)
{
    const int H = J->H;
    int64_t L = J->seq_lens[b];
    /* visible prefix for query t; an empty history (L == 0) has none */
    int64_t n = (L == 0) ? 0 : L - J->T + 1 + t;
    double *x = NULL, *score = NULL, *qd = NULL, *mx = NULL, *z = NULL;
    int64_t *pos = NULL;
    int err = 0;
    int64_t cnt = 0;

    if (L > 0 && L < J->T)
        return 2; /* the T new positions must already be in the history */

    qd = (double *)malloc(sizeof(double) * H * ORACLE_DQK);
    x = (double *)malloc(sizeof(double) * ORACLE_DQK);
    mx = (double *)malloc(sizeof(double) * H);
    z = (double *)malloc(sizeof(double) * H);
    pos = (int64_t *)malloc(sizeof(int64_t) * (n > 0 ? n : 1));
    score = (double *)malloc(sizeof(double) * H * (n > 0 ? n : 1));
    if (!qd || !x || !mx || !z || !pos || !score) {
        err = 3;
        goto done;
    }
    for (int h = 0; h < H; ++h)
        for (int d = 0; d < ORACLE_DQK; ++d)
            qd[h * ORACLE_DQK + d] =
                bf16_to_double(J->q[(((int64_t)b * J->T + t) * H + h) * ORACLE_DQK + d]);

    /* pass 1: scores of every kept visible position */
    for (int64_t p = 0; p < n; ++p) {
        if (!keep_position(J, p))
            continue;
        const uint8_t *codes = position_codes(J, b, p, &err);
        if (err)
            goto done;
        for (int d = 0; d < ORACLE_DQK; ++d)
            x[d] = J->lut[codes[d]];
        for (int h = 0; h < H; ++h) {
            if (!row_wanted(J, b, t, h))
                continue;
            double acc = 0.0;
            for (int d = 0; d < ORACLE_DQK; ++d)
                acc += qd[h * ORACLE_DQK + d] * x[d];
            score[(int64_t)h * n + cnt] = J->sm_scale * acc;
        }
        pos[cnt++] = p;
    }

    for (int h = 0; h < H; ++h) {
        if (!row_wanted(J, b, t, h))
            continue;
        double *o = J->out + (((int64_t)b * J->T + t) * H + h) * ORACLE_DV;
        double *l = J->lse + ((int64_t)b * J->T + t) * H + h;
        memset(o, 0, sizeof(double) * ORACLE_DV);
        if (cnt == 0) {
            *l = -INFINITY; /* nothing visible: empty partial answer */
            mx[h] = -INFINITY;
            continue;
        }
        double m = -INFINITY;
        for (int64_t i = 0; i < cnt; ++i)
            if (score[(int64_t)h * n + i] > m)
                m = score[(int64_t)h * n + i];
        mx[h] = m;
        z[h] = 0.0;
    }

    /* pass 2: weights and the weighted sum of the first 512 dims */
    for (int64_t i = 0; i < cnt; ++i) {
        const uint8_t *codes = position_codes(J, b, pos[i], &err);
        if (err)
            goto done;
        for (int d = 0; d < ORACLE_DV; ++d)
            x[d] = J->lut[codes[d]];
        for (int h = 0; h < H; ++h) {
            if (!row_wanted(J, b, t, h))
                continue;
            double w = exp(score[(int64_t)h * n + i] - mx[h]);
            double *o = J->out + (((int64_t)b * J->T + t) * H + h) * ORACLE_DV;
            z[h] += w;
            for (int d = 0; d < ORACLE_DV; ++d)
                o[d] += w * x[d];
        }
    }
    if (cnt > 0) {
        for (int h = 0; h < H; ++h) {
            if (!row_wanted(J, b, t, h))
                continue;
            double *o = J->out + (((int64_t)b * J->T + t) * H + h) * ORACLE_DV;
            for (int d = 0; d < ORACLE_DV; ++d)
                o[d] /= z[h];
            J->lse[((int64_t)b * J->T + t) * H + h] = mx[h] + log(z[h]);
        }
    }
done:
    free(qd);
    free(x);
    free(mx);
    free(z);
    free(pos);
    free(score);
    return err;
}

static void *decode_worker(void *arg)
{
    decode_job *J = (decode_job *)arg;
    const int64_t units = (int64_t)J->B * J->T;
    for (;;) {
        int64_t u = __sync_fetch_and_add(&J->next_unit, 1);
        if (u >= units || J->error)
            break;
        int rc = decode_unit(J, (int)(u / J->T), (int)(u % J->T));
        if (rc)
            J->error = rc;
    }
    return NULL;
}

static int resolve_threads(int n_threads, int64_t units)
{
    if (n_threads <= 0) {
        long c = sysconf(_SC_NPROCESSORS_ONLN);
        n_threads = c > 0 ? (int)c : 1;
    }
    if (n_threads > units)
        n_threads = (int)(units > 0 ? units : 1);
    return n_threads;
}

/* Returns the number of worker threads actually used (>0), or a negative
 * code: -1 bad arguments, -2 a request has seq_len < T, -3 out of memory,
 * -4 a block-table entry is not a valid page id. */
int oracle_mla_decode(const uint16_t *q, const uint8_t *kv, int64_t num_pages,
                      float kv_scale, const int32_t *block_table, int64_t bt_stride,
                      const int32_t *seq_lens, int B, int T, int H, double sm_scale,
                      const uint8_t *pos_mask, int64_t pos_mask_len,
                      const uint8_t *row_mask, double *out, double *lse, int n_threads)
{
    if (!q || !kv || !block_table || !seq_lens || !out || !lse || B < 0 || T < 1 || H < 1)
        return -1;
    for (int b = 0; b < B; ++b)
        if (seq_lens[b] < 0 || (int64_t)(seq_lens[b] + ORACLE_PAGE - 1) / ORACLE_PAGE > bt_stride)
            return -1;

    decode_job *J = (decode_job *)calloc(1, sizeof(decode_job));
    if (!J)
        return -3;
    J->q = q;
    J->kv = kv;
    J->num_pages = num_pages;
    J->kv_scale = (double)kv_scale;
    J->block_table = block_table;
    J->bt_stride = bt_stride;
    J->seq_lens = seq_lens;
    J->B = B;
    J->T = T;
    J->H = H;
    J->sm_scale = sm_scale;
    J->pos_mask = pos_mask;
    J->pos_mask_len = pos_mask_len;
    J->row_mask = row_mask;
    J->out = out;
    J->lse = lse;
    for (int c = 0; c < 256; ++c)
        J->lut[c] = oracle_e4m3fn_to_double((uint8_t)c) * J->kv_scale;

    const int64_t units = (int64_t)B * T;
    int nt = resolve_threads(n_threads, units);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * nt);
    int started = 0;
    if (th) {
        for (int i = 0; i < nt; ++i) {
            if (pthread_create(&th[i], NULL, decode_worker, J) != 0)
                break;
            ++started;
        }
    }
    if (started == 0)
        decode_worker(J); /* no threads available: run inline */
    for (int i = 0; i < started; ++i)
        pthread_join(th[i], NULL);
    free(th);

    int rc = J->error;
    free(J);
    if (rc == 1)
        return -4;
    if (rc == 2)
        return -2;
    if (rc == 3)
        return -3;
    return started > 0 ? started : 1;
}

/* ------------------------------------------------------------------ */
/* Merge of partial answers by their normalisers                         */
/* ------------------------------------------------------------------ */

/* Section 1 "Cache" (DCP): each partial answer o_s over a part of the history
 * carries lse_s = ln sum_{p in part s} exp(score_p).  For any partition of the
 * positions:  lse = M' + ln sum_s exp(lse_s - M'),  M' = max_s lse_s,
 *             out = sum_s exp(lse_s - lse) * o_s.
 * Parts with lse_s = -inf weigh 0; if every part is empty the result is
 * out = 0, lse = -inf.  part_out is [S][rows][D], part_lse is [S][rows]. */
int oracle_lse_merge(int S, int64_t rows, int D, const double *part_out,
                     const double *part_lse, double *out, double *lse)
{
    if (S < 1 || rows < 0 || D < 1 || !part_out || !part_lse || !out || !lse)
        return -1;
    for (int64_t r = 0; r < rows; ++r) {
        double m = -INFINITY;
        for (int s = 0; s < S; ++s)
            if (part_lse[(int64_t)s * rows + r] > m)
                m = part_lse[(int64_t)s * rows + r];
        double *o = out + r * D;
        for (int d = 0; d < D; ++d)
            o[d] = 0.0;
        if (m == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double sum = 0.0;
        for (int s = 0; s < S; ++s) {
            double ls = part_lse[(int64_t)s * rows + r];
            if (ls != -INFINITY)
                sum += exp(ls - m);
        }
        double total = m + log(sum);
        lse[r] = total;
        for (int s = 0; s < S; ++s) {
            double ls = part_lse[(int64_t)s * rows + r];
            if (ls == -INFINITY)
                continue;
            double w = exp(ls - total);
            const double *os = part_out + ((int64_t)s * rows + r) * D;
            for (int d = 0; d < D; ++d)
                o[d] += w * os[d];
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Appending new positions to the cache                                 */
/* ------------------------------------------------------------------ */

/* Encode a binary32 value as an E4M3FN byte, written out from the format
 * definition above: magnitudes of 448 and more (the largest finite value)
 * take 448; otherwise the nearest of the 127 non-negative finite values is
 * chosen, a tie going to the code whose mantissa is even; the sign bit is the
 * input's (so -0 and small negative values encode as 0x80).  NaN encodes as
 * 0x7F. */
uint8_t oracle_e4m3fn_encode(float x)
{
    if (isnan(x))
        return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0)
        return sign | 0x7E;
    /* the non-negative finite codes 0x00..0x7E have increasing values */
    int c = 0;
    while (c + 1 <= 0x7E && oracle_e4m3fn_to_double((uint8_t)(c + 1)) <= a)
        ++c;
    double lo = oracle_e4m3fn_to_double((uint8_t)c);
    if (lo == a)
        return sign | (uint8_t)c;
    double hi = oracle_e4m3fn_to_double((uint8_t)(c + 1));
    double dl = a - lo, dh = hi - a;
    int pick;
    if (dl < dh)
        pick = c;
    else if (dh < dl)
        pick = c + 1;
    else
        pick = (c & 1) == 0 ? c : c + 1;  /* tie: even mantissa */
    return sign | (uint8_t)pick;
}

void oracle_e4m3fn_encode_array(const float *x, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3fn_encode(x[i]);
}

/* The step before the decode in every decode step (the post's model section:
 * the compressed history grows by one latent per new position): the new
 * latent of request b at draft position t -- 576 bf16 values, the 512 latent
 * dims followed by the 64 rotated positional dims -- is divided by kv_scale
 * in binary32 (one correctly rounded division per value), encoded as E4M3FN
 * and written to page block_table[b][p / 64], row p % 64, with
 * p = start_pos[b] + t.  Nothing else in the cache changes.  A row whose
 * position lies outside [0, max_pages * 64) or whose page id lies outside
 * [0, num_pages) is not written, and the call returns -2. */
int oracle_append_latent(const uint16_t *latent, int B, int T, float kv_scale,
                         const int32_t *block_table, int64_t bt_stride, int max_pages,
                         const int32_t *start_pos, uint8_t *kv, int64_t num_pages)
{
    if (B < 0 || T < 0 || (B > 0 && T > 0 && (!latent || !block_table || !start_pos || !kv)))
        return -1;
    int rc = 0;
    for (int b = 0; b < B; ++b) {
        for (int t = 0; t < T; ++t) {
            int64_t p = (int64_t)start_pos[b] + t;
            if (p < 0 || p >= (int64_t)max_pages * ORACLE_PAGE) {
                rc = -2;
                continue;
            }
            int32_t page = block_table[(int64_t)b * bt_stride + p / ORACLE_PAGE];
            if (page < 0 || page >= num_pages) {
                rc = -2;
                continue;
            }
            uint8_t *dst = kv + ((int64_t)page * ORACLE_PAGE + p % ORACLE_PAGE) * ORACLE_DQK;
            const uint16_t *src = latent + ((int64_t)b * T + t) * ORACLE_DQK;
            for (int d = 0; d < ORACLE_DQK; ++d) {
                uint32_t u = (uint32_t)src[d] << 16;
                float f;
                memcpy(&f, &u, sizeof f);
                float v = f / kv_scale;
                dst[d] = oracle_e4m3fn_encode(v);
            }
        }
    }
    return rc;
}
