/*
 * oracle.c -- plain, slow, fp64 CPU oracle of the paged-attention decode path.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library. The CUDA path never calls it,
 * shares no code with it and must not fall back to it.
 *
 * What it computes, step by step, and where each step is defined:
 *
 *  cache write   Each new token's K and V vectors go to their slot: block
 *                slot / block_size, offset slot % block_size. Raw 16-bit words
 *                are copied; nothing is converted. (yangyu.win blog #54,
 *                section 5 question 2: a sequence that grows past a block
 *                boundary takes one new block from the free pool; itimpress.au
 *                "PagedAttention, ...", section 1: K and V of every previous
 *                token are kept so they are not recomputed.)
 *  copy-on-write A shared block about to be written is first copied whole to a
 *                fresh block (yangyu.win blog #54, section 5 question 2).
 *  gather        Logical token t of a sequence lives in physical block
 *                block_table[t / block_size] at offset t % block_size.
 *                (yangyu.win blog #54, section 2.2 figure: tokens 0-15 -> page 7,
 *                16-31 -> page 2, 32-47 -> page 19; learn.tanhdev.com part 8,
 *                block-table diagram: virtual 0 -> #42, 1 -> #108, 2 -> #19.)
 *  attention     A_i = softmax(q_i K^T / sqrt(d_k)), o_i = sum over blocks j and
 *                slots t of a_{i,j,t} v_{(j,t)}. (learn.tanhdev.com part 8,
 *                section "Thuc thi kernel toan hoc trong CUDA", equations for A_i,
 *                A_{i,j} and o_i.) GQA: query head h reads KV head h / (Hq / Hkv)
 *                (contiguous groups; the pages name GQA, not the mapping).
 *                With q_len > 1 (verifying draft tokens in one pass:
 *                itimpress.au section 1, yangyu.win section 2.4) query row qi sits
 *                at position L - q_len + qi and sees tokens 0 .. L - q_len + qi.
 *  verify-accept Speculative rejection sampling over the target's verify pass
 *                (yangyu.win blog #54, section 5 question 3; maths.nthquan ch. 17
 *                "Speculative decoding", algorithm steps 3-4): draft token x_i is
 *                kept with probability min(1, p_i(x_i) / q_i(x_i)); the first
 *                rejected position is resampled from max(0, p_i - q_i)
 *                renormalised and later drafts are dropped; if every draft is
 *                kept, one more token is drawn from the target's next
 *                distribution. The uniform draws are inputs.
 *  partitions    The context is cut into fixed partitions; each yields its own
 *                (max, sum of exponentials, unnormalised weighted V), and a
 *                reduction combines them (maths.nthquan ch. 17 "Scaling and
 *                deployment", section "Sequence parallelism": local attention
 *                per cached segment, then a reduction). The combination is the
 *                log-sum-exp merge written out from the softmax definition.
 *
 * All arithmetic is fp64. fp16/bf16 inputs are decoded exactly from their bit
 * patterns. The softmax subtracts the maximum score first (the same value,
 * written to avoid overflow). Nothing is blocked, fused or reordered beyond
 * these definitions.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define OR_OK 0
#define OR_ERR_ARG 1
#define OR_ERR_BOUNDS 2
#define OR_ERR_OOM 3

#define OR_FP16 0
#define OR_BF16 1

/* ---------------------------------------------------------------- decoding */

/* IEEE binary16: sign, 5-bit exponent (bias 15), 10-bit fraction. */
double oracle_f16_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);    /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
double oracle_bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double dec(uint16_t w, int dtype) {
    return dtype == OR_BF16 ? oracle_bf16_to_double(w) : oracle_f16_to_double(w);
}

/* ------------------------------------------------------------- cache write */

/* k, v: [num_tokens, Hkv, d]; pools: [num_blocks, Hkv, bs, d]. slot < 0 is skipped. */
int oracle_cache_write(uint16_t *k_pool, uint16_t *v_pool, const uint16_t *k, const uint16_t *v,
                       const int64_t *slot_mapping, int64_t num_tokens, int64_t num_blocks,
                       int bs, int Hkv, int d) {
    if (!k_pool || !v_pool || !k || !v || !slot_mapping || bs <= 0 || Hkv <= 0 || d <= 0)
        return OR_ERR_ARG;
    for (int64_t i = 0; i < num_tokens; ++i) {
        int64_t s = slot_mapping[i];
        if (s < 0) continue;
        int64_t blk = s / bs, off = s % bs;
        if (blk >= num_blocks) return OR_ERR_BOUNDS;
        for (int h = 0; h < Hkv; ++h) {
            int64_t src = (i * Hkv + h) * (int64_t)d;
            int64_t dst = ((blk * Hkv + h) * bs + off) * (int64_t)d;
            memcpy(k_pool + dst, k + src, (size_t)d * sizeof(uint16_t));
            memcpy(v_pool + dst, v + src, (size_t)d * sizeof(uint16_t));
        }
    }
    return OR_OK;
}

/*
 * Copy-on-write copy: block pairs[2i] -> block pairs[2i+1] of both pools, every KV head, raw
 * words (yangyu.win blog #54, section 5 question 2: a diverging sequence gets its own copy of
 * the shared block it is about to write).
 */
int oracle_copy_blocks(uint16_t *k_pool, uint16_t *v_pool, const int32_t *pairs, int64_t n, int64_t num_blocks,
                       int bs, int Hkv, int d) {
    if (!k_pool || !v_pool || (n > 0 && !pairs) || bs <= 0 || Hkv <= 0 || d <= 0) return OR_ERR_ARG;
    const int64_t words = (int64_t)Hkv * bs * d;
    for (int64_t i = 0; i < n; ++i) {
        int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) return OR_ERR_BOUNDS;
        memcpy(k_pool + dst * words, k_pool + src * words, (size_t)words * sizeof(uint16_t));
        memcpy(v_pool + dst * words, v_pool + src * words, (size_t)words * sizeof(uint16_t));
    }
    return OR_OK;
}

/* ------------------------------------------------------------------ gather */

/* Contiguous [L, Hkv, d] copy of one sequence's K (or V) through its block-table row. */
int oracle_gather(const uint16_t *pool, const int32_t *table_row, int64_t L, int64_t num_blocks,
                  int bs, int Hkv, int d, uint16_t *out) {
    if (!pool || !table_row || !out || L < 0 || bs <= 0) return OR_ERR_ARG;
    for (int64_t t = 0; t < L; ++t) {
        int64_t phys = table_row[t / bs];
        int64_t off = t % bs;
        if (phys < 0 || phys >= num_blocks) return OR_ERR_BOUNDS;
        for (int h = 0; h < Hkv; ++h)
            memcpy(out + (t * Hkv + h) * (int64_t)d, pool + ((phys * Hkv + h) * bs + off) * (int64_t)d,
                   (size_t)d * sizeof(uint16_t));
    }
    return OR_OK;
}

/* --------------------------------------------------------------- attention */

/*
 * The attention of one sequence on contiguous K/V given as fp64 values.
 *   qd  [q_len, Hq, d]     kd, vd  [L, Hkv, d]     out  [q_len, Hq, d]
 *   weights (optional) [q_len, Hq, L]: the softmax weights, 0 for masked tokens.
 */
static int attention_f64(const double *qd, const double *kd, const double *vd, int64_t L, int q_len, int Hq,
                         int Hkv, int d, float scale, double *out, double *weights) {
    if (q_len < 1 || L < q_len || Hkv <= 0 || Hq % Hkv != 0 || d <= 0) return OR_ERR_ARG;
    int G = Hq / Hkv;
    double *s = (double *)malloc((size_t)L * sizeof(double));
    if (!s) return OR_ERR_OOM;
    for (int qi = 0; qi < q_len; ++qi) {
        int64_t last = L - q_len + qi;                     /* inclusive causal limit */
        for (int h = 0; h < Hq; ++h) {
            int g = h / G;
            const double *qr = qd + ((int64_t)qi * Hq + h) * d;
            double mx = -INFINITY;
            for (int64_t t = 0; t <= last; ++t) {
                double dot = 0.0;
                const double *kr = kd + (t * Hkv + g) * (int64_t)d;
                for (int k = 0; k < d; ++k) dot += qr[k] * kr[k];
                s[t] = (double)scale * dot;
                if (s[t] > mx) mx = s[t];
            }
            double l = 0.0;
            for (int64_t t = 0; t <= last; ++t) { s[t] = exp(s[t] - mx); l += s[t]; }
            double *o = out + ((int64_t)qi * Hq + h) * d;
            for (int k = 0; k < d; ++k) o[k] = 0.0;
            for (int64_t t = 0; t <= last; ++t) {
                double p = s[t] / l;
                const double *vr = vd + (t * Hkv + g) * (int64_t)d;
                for (int k = 0; k < d; ++k) o[k] += p * vr[k];
            }
            if (weights) {
                double *w = weights + ((int64_t)qi * Hq + h) * L;
                for (int64_t t = 0; t < L; ++t) w[t] = t <= last ? s[t] / l : 0.0;
            }
        }
    }
    free(s);
    return OR_OK;
}

static double *decode_all(const uint16_t *w, int64_t n, int dtype) {
    double *x = (double *)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
    if (x)
        for (int64_t i = 0; i < n; ++i) x[i] = dec(w[i], dtype);
    return x;
}

/*
 * One sequence on contiguous K/V (16-bit words, decoded exactly).
 *   q   [q_len, Hq, d]     kc, vc  [L, Hkv, d]     out  [q_len, Hq, d] (double)
 *   weights (optional) [q_len, Hq, L]: the softmax weights, 0 for masked tokens.
 */
int oracle_attention(const uint16_t *q, const uint16_t *kc, const uint16_t *vc, int64_t L, int q_len,
                     int Hq, int Hkv, int d, int dtype, float scale, double *out, double *weights) {
    if (!q || !kc || !vc || !out || q_len < 1 || L < q_len || Hkv <= 0 || Hq % Hkv != 0 || d <= 0)
        return OR_ERR_ARG;
    double *qd = decode_all(q, (int64_t)q_len * Hq * d, dtype);
    double *kd = decode_all(kc, L * Hkv * d, dtype);
    double *vd = decode_all(vc, L * Hkv * d, dtype);
    int rc = (!qd || !kd || !vd) ? OR_ERR_OOM
                                 : attention_f64(qd, kd, vd, L, q_len, Hq, Hkv, d, scale, out, weights);
    free(qd);
    free(kd);
    free(vd);
    return rc;
}

/* --------------------------------------------------------- paged attention */

/* Contiguous [L, d] copy of KV head g of one sequence through its block-table row. */
static int gather_head(const uint16_t *pool, const int32_t *table_row, int64_t L, int64_t num_blocks, int bs,
                       int Hkv, int d, int g, uint16_t *out) {
    for (int64_t t = 0; t < L; ++t) {
        int64_t phys = table_row[t / bs];
        int64_t off = t % bs;
        if (phys < 0 || phys >= num_blocks) return OR_ERR_BOUNDS;
        memcpy(out + t * (int64_t)d, pool + ((phys * Hkv + g) * bs + off) * (int64_t)d, (size_t)d * sizeof(uint16_t));
    }
    return OR_OK;
}

typedef struct {
    const uint16_t *q, *k_pool, *v_pool;
    const int32_t *tables;
    const int32_t *lens;
    const int32_t *seqs;         /* which sequences to compute (rows of q / out follow this list) */
    int64_t stride, num_blocks;
    int nseq, q_len, Hq, Hkv, d, bs, dtype;
    float scale;
    double *out;
    int next;                    /* work counter over (listed sequence, KV head) items */
    int err;
    pthread_mutex_t mu;
} paged_job;

/*
 * One work item = one sequence and one KV head g: gather that head's K and V through the
 * block table, then run attention for the G query heads of group g (the same computation
 * as the whole-sequence call, restricted to one group: Hkv = 1, Hq = G).
 */
static void *paged_worker(void *arg) {
    paged_job *J = (paged_job *)arg;
    const int G = J->Hq / J->Hkv;
    for (;;) {
        pthread_mutex_lock(&J->mu);
        int item = J->next++;
        pthread_mutex_unlock(&J->mu);
        if (item >= J->nseq * J->Hkv) break;
        int i = item / J->Hkv, g = item % J->Hkv;
        int b = J->seqs ? J->seqs[i] : i;
        int64_t L = J->lens[b];
        int rc = OR_OK;
        if (L < J->q_len || (L + J->bs - 1) / J->bs > J->stride) rc = OR_ERR_BOUNDS;
        uint16_t *kc = NULL, *vc = NULL, *qs = NULL;
        double *os = NULL;
        if (rc == OR_OK) {
            kc = (uint16_t *)malloc((size_t)L * J->d * sizeof(uint16_t));
            vc = (uint16_t *)malloc((size_t)L * J->d * sizeof(uint16_t));
            qs = (uint16_t *)malloc((size_t)J->q_len * G * J->d * sizeof(uint16_t));
            os = (double *)malloc((size_t)J->q_len * G * J->d * sizeof(double));
            if (!kc || !vc || !qs || !os) rc = OR_ERR_OOM;
        }
        const int32_t *row = J->tables + (int64_t)b * J->stride;
        if (rc == OR_OK) rc = gather_head(J->k_pool, row, L, J->num_blocks, J->bs, J->Hkv, J->d, g, kc);
        if (rc == OR_OK) rc = gather_head(J->v_pool, row, L, J->num_blocks, J->bs, J->Hkv, J->d, g, vc);
        const uint16_t *qb = J->q + (int64_t)i * J->q_len * J->Hq * J->d;
        double *ob = J->out + (int64_t)i * J->q_len * J->Hq * J->d;
        if (rc == OR_OK) {
            for (int qi = 0; qi < J->q_len; ++qi)
                for (int hh = 0; hh < G; ++hh)
                    memcpy(qs + ((int64_t)qi * G + hh) * J->d, qb + ((int64_t)qi * J->Hq + g * G + hh) * J->d,
                           (size_t)J->d * sizeof(uint16_t));
            rc = oracle_attention(qs, kc, vc, L, J->q_len, G, 1, J->d, J->dtype, J->scale, os, NULL);
        }
        if (rc == OR_OK)
            for (int qi = 0; qi < J->q_len; ++qi)
                for (int hh = 0; hh < G; ++hh)
                    memcpy(ob + ((int64_t)qi * J->Hq + g * G + hh) * J->d, os + ((int64_t)qi * G + hh) * J->d,
                           (size_t)J->d * sizeof(double));
        free(kc);
        free(vc);
        free(qs);
        free(os);
        if (rc != OR_OK) {
            pthread_mutex_lock(&J->mu);
            if (!J->err) J->err = rc;
            pthread_mutex_unlock(&J->mu);
        }
    }
    return NULL;
}

int oracle_num_cpus(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/*
 * Paged decode for the sequences listed in seqs (or all num_seqs when seqs is NULL):
 * gather each sequence through its block-table row, then attention.
 *   q, out: one [q_len, Hq, d] row per listed sequence, in list order.
 *   *threads_used (may be NULL) receives the number of threads used.
 */
int oracle_paged_attention(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                           const int32_t *block_tables, int64_t stride, const int32_t *context_lens,
                           const int32_t *seqs, int nseq, int64_t num_blocks, int bs, int q_len, int Hq,
                           int Hkv, int d, int dtype, float scale, double *out, int num_threads,
                           int *threads_used) {
    if (!q || !k_pool || !v_pool || !block_tables || !context_lens || !out || nseq < 0 || Hkv <= 0 ||
        Hq % Hkv != 0 || bs <= 0)
        return OR_ERR_ARG;
    paged_job J;
    memset(&J, 0, sizeof J);
    J.q = q; J.k_pool = k_pool; J.v_pool = v_pool; J.tables = block_tables; J.lens = context_lens;
    J.seqs = seqs; J.stride = stride; J.num_blocks = num_blocks; J.nseq = nseq; J.q_len = q_len;
    J.Hq = Hq; J.Hkv = Hkv; J.d = d; J.bs = bs; J.dtype = dtype; J.scale = scale; J.out = out;
    pthread_mutex_init(&J.mu, NULL);
    int items = nseq * Hkv;
    int nt = num_threads > 0 ? num_threads : oracle_num_cpus();
    if (nt > items) nt = items > 0 ? items : 1;
    pthread_t *th = (pthread_t *)malloc((size_t)nt * sizeof(pthread_t));
    if (!th) return OR_ERR_OOM;
    for (int i = 0; i < nt; ++i) pthread_create(&th[i], NULL, paged_worker, &J);
    for (int i = 0; i < nt; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.mu);
    if (threads_used) *threads_used = nt;
    return J.err;
}

/* ------------------------------------------------ partitions and the merge */

/*
 * One sequence on contiguous K/V, context cut into partitions of P tokens.
 * For partition p (tokens [pP, min((p+1)P, L)) that row qi may see):
 *   m[p]  = max score            (-inf when the row sees none of them)
 *   l[p]  = sum exp(s_t - m[p])  (0 when empty)
 *   o[p]  = sum exp(s_t - m[p]) v_t   (unnormalised; 0 when empty)
 * Layouts: m, l [q_len, Hq, np]; o [q_len, Hq, np, d], np = ceil(L / P).
 */
int oracle_attention_partitions(const uint16_t *q, const uint16_t *kc, const uint16_t *vc, int64_t L,
                                int q_len, int Hq, int Hkv, int d, int dtype, float scale, int64_t P,
                                double *m, double *l, double *o) {
    if (!q || !kc || !vc || !m || !l || !o || P <= 0 || q_len < 1 || L < q_len || Hq % Hkv != 0)
        return OR_ERR_ARG;
    int G = Hq / Hkv;
    int64_t np_ = (L + P - 1) / P;
    double *s = (double *)malloc((size_t)P * sizeof(double));
    if (!s) return OR_ERR_OOM;
    for (int qi = 0; qi < q_len; ++qi) {
        int64_t last = L - q_len + qi;
        for (int h = 0; h < Hq; ++h) {
            int g = h / G;
            const uint16_t *qr = q + ((int64_t)qi * Hq + h) * d;
            for (int64_t p = 0; p < np_; ++p) {
                int64_t row = ((int64_t)qi * Hq + h) * np_ + p;
                int64_t t0 = p * P, t1 = (p + 1) * P < L ? (p + 1) * P : L;
                if (t1 > last + 1) t1 = last + 1;
                double mx = -INFINITY, sum = 0.0;
                double *op = o + row * d;
                for (int k = 0; k < d; ++k) op[k] = 0.0;
                for (int64_t t = t0; t < t1; ++t) {
                    double dot = 0.0;
                    const uint16_t *kr = kc + (t * Hkv + g) * (int64_t)d;
                    for (int k = 0; k < d; ++k) dot += dec(qr[k], dtype) * dec(kr[k], dtype);
                    s[t - t0] = (double)scale * dot;
                    if (s[t - t0] > mx) mx = s[t - t0];
                }
                for (int64_t t = t0; t < t1; ++t) {
                    double e = exp(s[t - t0] - mx);
                    sum += e;
                    const uint16_t *vr = vc + (t * Hkv + g) * (int64_t)d;
                    for (int k = 0; k < d; ++k) op[k] += e * dec(vr[k], dtype);
                }
                m[row] = mx;
                l[row] = sum;
            }
        }
    }
    free(s);
    return OR_OK;
}

/*
 * Log-sum-exp merge of np partitions of one output row:
 *   M = max over non-empty partitions of m[p]
 *   out = sum_p exp(m[p] - M) o[p] / sum_p exp(m[p] - M) l[p]
 * m, l: [np]; o: [np, d]; out: [d].
 */
int oracle_lse_merge(int64_t np_, const double *m, const double *l, const double *o, int d, double *out) {
    if (!m || !l || !o || !out || np_ < 1) return OR_ERR_ARG;
    double M = -INFINITY;
    for (int64_t p = 0; p < np_; ++p)
        if (l[p] > 0.0 && m[p] > M) M = m[p];
    double den = 0.0;
    for (int k = 0; k < d; ++k) out[k] = 0.0;
    for (int64_t p = 0; p < np_; ++p) {
        if (!(l[p] > 0.0)) continue;
        double w = exp(m[p] - M);
        den += w * l[p];
        for (int k = 0; k < d; ++k) out[k] += w * o[p * d + k];
    }
    for (int k = 0; k < d; ++k) out[k] /= den;
    return OR_OK;
}

/* ------------------------------------------------ speculative rejection sampling */

/*
 * Index of the first j with sum_{t <= j} w_t > v * sum_t w_t (serial fp64 sums). When the total
 * is 0 the result is -1.
 */
static int64_t inverse_cdf(const double *w, int64_t V, double v) {
    double total = 0.0;
    for (int64_t t = 0; t < V; ++t) total += w[t];
    if (!(total > 0.0)) return -1;
    const double target = v * total;
    double c = 0.0;
    for (int64_t t = 0; t < V; ++t) {
        c += w[t];
        if (c > target) return t;
    }
    for (int64_t t = V - 1; t >= 0; --t)       /* v * total rounded up to total: the last token with mass */
        if (w[t] > 0.0) return t;
    return -1;
}

/*
 * One batch of verifications.
 *   p      fp32 [B, K+1, V]  target distributions at the K draft positions and the next one
 *   q      fp32 [B, K, V]    draft distributions
 *   draft  int32 [B, K]      draft tokens
 *   u      fp32 [B, K]       uniforms in [0, 1) for the accept tests
 *   v      fp32 [B]          uniform in [0, 1) for the one token drawn at the end
 *   out    int32 [B, K+1]    emitted tokens (kept drafts, then the drawn token), -1 after them
 *   n_out  int32 [B]         number of emitted tokens (kept drafts + 1)
 * The accept test is evaluated in fp32 as u * q < p (the same comparison as
 * u < p / q for q > 0, without a division). The drawn token is the inverse CDF
 * of max(0, p_i - q_i) (or of p_K when all drafts are kept) at v, in fp64;
 * when the residual has no mass, p_i itself is used.
 */
int oracle_spec_verify(const float *p, const float *q, const int32_t *draft, const float *u, const float *v,
                       int64_t B, int K, int64_t V, int32_t *out, int32_t *n_out) {
    if (!p || !q || !draft || !u || !v || !out || !n_out || B < 0 || K < 0 || V <= 0) return OR_ERR_ARG;
    double *w = (double *)malloc((size_t)V * sizeof(double));
    if (!w) return OR_ERR_OOM;
    int rc = OR_OK;
    for (int64_t b = 0; b < B && rc == OR_OK; ++b) {
        int32_t *o = out + b * (K + 1);
        for (int i = 0; i <= K; ++i) o[i] = -1;
        int n = 0;
        int rejected = -1;
        for (int i = 0; i < K; ++i) {
            const int32_t x = draft[b * K + i];
            if (x < 0 || x >= V) { rc = OR_ERR_BOUNDS; break; }
            const float pi = p[(b * (K + 1) + i) * V + x];
            const float qi = q[(b * K + i) * V + x];
            const float uq = u[b * K + i] * qi;       /* one fp32 rounding */
            if (uq < pi) {
                o[n++] = x;
            } else {
                rejected = i;
                break;
            }
        }
        if (rc != OR_OK) break;
        int64_t tok;
        if (rejected >= 0) {
            const float *pr = p + (b * (K + 1) + rejected) * V;
            const float *qr = q + (b * K + rejected) * V;
            for (int64_t t = 0; t < V; ++t) {
                const double r = (double)pr[t] - (double)qr[t];
                w[t] = r > 0.0 ? r : 0.0;
            }
            tok = inverse_cdf(w, V, (double)v[b]);
            if (tok < 0) {
                for (int64_t t = 0; t < V; ++t) w[t] = pr[t] > 0.0f ? (double)pr[t] : 0.0;
                tok = inverse_cdf(w, V, (double)v[b]);
            }
        } else {
            const float *pr = p + (b * (K + 1) + K) * V;
            for (int64_t t = 0; t < V; ++t) w[t] = pr[t] > 0.0f ? (double)pr[t] : 0.0;
            tok = inverse_cdf(w, V, (double)v[b]);
        }
        o[n++] = (int32_t)tok;
        n_out[b] = n;
    }
    free(w);
    return rc;
}

/* ---------------------------------------------------------------- FP8 KV */

/*
 * FP8 E4M3 (1 sign bit, 4 exponent bits with bias 7, 3 fraction bits; no
 * infinities; S.1111.111 is NaN; largest finite 448): the code's value.
 */
double oracle_e4m3_to_double(uint8_t c) {
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 7;
    double v;
    if (e == 15 && m == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)m, -9);                  /* subnormal: m/8 * 2^(1-7) */
    else
        v = ldexp((double)(8 + m), e - 10);        /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

/* Round a float to the nearest E4M3 value (ties to even), saturating to +-448; NaN -> NaN code. */
uint8_t oracle_f32_to_e4m3(float x) {
    if (x != x) return 0x7F;
    uint8_t sign = (x < 0.0f || (x == 0.0f && 1.0f / x < 0.0f)) ? 0x80 : 0;
    double a = fabs((double)x);
    if (a >= 448.0) return sign | 0x7E;
    /* quantum of the binade (normals: 2^(e-3); subnormals: 2^-9) */
    int e;
    frexp(a, &e);                                   /* a = f * 2^e, f in [0.5, 1) -> binade exponent e-1 */
    int be = e - 1;
    if (be < -6) be = -6;
    double quantum = ldexp(1.0, be - 3);
    double n = nearbyint(a / quantum);              /* exact division by a power of two; ties to even */
    double r = n * quantum;
    if (r >= 448.0) return sign | 0x7E;
    if (r == 0.0) return sign;
    int re;
    frexp(r, &re);
    int rbe = re - 1;                               /* binade of the rounded value */
    if (rbe < -6) {                                 /* subnormal: r = m * 2^-9 */
        int m = (int)nearbyint(r / ldexp(1.0, -9));
        return sign | (uint8_t)m;
    }
    int m = (int)nearbyint(r / ldexp(1.0, rbe - 3)) - 8;
    return sign | (uint8_t)(((rbe + 7) << 3) | m);
}

/*
 * Quantising cache write. A pool in FP8 layout holds, in one buffer, the codes
 * [num_blocks, Hkv, bs, d] (bytes) followed by one float32 scale per slot and
 * head [num_blocks, Hkv, bs]. Each new (token, head) row of d 16-bit values x
 * is stored as scale = amax|x| / 448 (float32; 1 when amax is 0) and codes
 * e4m3(x / scale) (the division in float32), so the row's largest magnitude
 * maps to the largest finite code and nothing overflows (the quantisation
 * section of learn.tanhdev.com part 8: FP8 E4M3 KV halves the cache, with care
 * against outliers; yangyu.win blog #54 section 4: quantise the KV cache to
 * FP8). slot < 0 is skipped.
 */
int oracle_cache_write_fp8(uint8_t *k_pool, uint8_t *v_pool, const uint16_t *k, const uint16_t *v,
                           const int64_t *slot_mapping, int64_t num_tokens, int64_t num_blocks, int bs, int Hkv,
                           int d, int dtype) {
    if (!k_pool || !v_pool || !k || !v || !slot_mapping || bs <= 0 || Hkv <= 0 || d <= 0) return OR_ERR_ARG;
    const int64_t codes = num_blocks * Hkv * bs * (int64_t)d;
    for (int64_t i = 0; i < num_tokens; ++i) {
        int64_t s = slot_mapping[i];
        if (s < 0) continue;
        int64_t blk = s / bs, off = s % bs;
        if (blk >= num_blocks) return OR_ERR_BOUNDS;
        for (int which = 0; which < 2; ++which) {
            uint8_t *pool = which ? v_pool : k_pool;
            const uint16_t *src = which ? v : k;
            float *scales = (float *)(pool + codes);
            for (int h = 0; h < Hkv; ++h) {
                const uint16_t *row = src + (i * Hkv + h) * (int64_t)d;
                float amax = 0.0f;
                for (int c = 0; c < d; ++c) {
                    float a = fabsf((float)dec(row[c], dtype));
                    if (a > amax) amax = a;
                }
                float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
                int64_t slot_row = (blk * Hkv + h) * bs + off;
                scales[slot_row] = scale;
                for (int c = 0; c < d; ++c) pool[slot_row * d + c] = oracle_f32_to_e4m3((float)dec(row[c], dtype) / scale);
            }
        }
    }
    return OR_OK;
}

/*
 * Paged decode over FP8 pools: each (sequence, KV head) item gathers its codes
 * and scales through the block table, dequantises (code value * scale, fp64)
 * and runs the same attention as the 16-bit path. q and out as in
 * oracle_paged_attention.
 */
int oracle_paged_attention_fp8(const uint16_t *q, const uint8_t *k_pool, const uint8_t *v_pool,
                               const int32_t *block_tables, int64_t stride, const int32_t *context_lens,
                               const int32_t *seqs, int nseq, int64_t num_blocks, int bs, int q_len, int Hq,
                               int Hkv, int d, int dtype, float scale, double *out) {
    if (!q || !k_pool || !v_pool || !block_tables || !context_lens || !out || nseq < 0 || Hkv <= 0 ||
        Hq % Hkv != 0)
        return OR_ERR_ARG;
    const int G = Hq / Hkv;
    const int64_t codes = num_blocks * Hkv * bs * (int64_t)d;
    const float *ks = (const float *)(k_pool + codes);
    const float *vs = (const float *)(v_pool + codes);
    for (int i = 0; i < nseq; ++i) {
        const int b = seqs ? seqs[i] : i;
        const int64_t L = context_lens[b];
        if (L < q_len || (L + bs - 1) / bs > stride) return OR_ERR_BOUNDS;
        const int32_t *row = block_tables + (int64_t)b * stride;
        double *qd = (double *)malloc((size_t)q_len * G * d * sizeof(double));
        double *kd = (double *)malloc((size_t)L * d * sizeof(double));
        double *vd = (double *)malloc((size_t)L * d * sizeof(double));
        double *od = (double *)malloc((size_t)q_len * G * d * sizeof(double));
        int rc = (!qd || !kd || !vd || !od) ? OR_ERR_OOM : OR_OK;
        for (int g = 0; g < Hkv && rc == OR_OK; ++g) {
            for (int64_t t = 0; t < L && rc == OR_OK; ++t) {
                int64_t phys = row[t / bs];
                if (phys < 0 || phys >= num_blocks) { rc = OR_ERR_BOUNDS; break; }
                int64_t sr = (phys * Hkv + g) * bs + t % bs;
                for (int c = 0; c < d; ++c) {
                    kd[t * d + c] = oracle_e4m3_to_double(k_pool[sr * d + c]) * (double)ks[sr];
                    vd[t * d + c] = oracle_e4m3_to_double(v_pool[sr * d + c]) * (double)vs[sr];
                }
            }
            if (rc != OR_OK) break;
            const uint16_t *qb = q + (int64_t)i * q_len * Hq * d;
            for (int qi = 0; qi < q_len; ++qi)
                for (int hh = 0; hh < G; ++hh)
                    for (int c = 0; c < d; ++c)
                        qd[((int64_t)qi * G + hh) * d + c] = dec(qb[((int64_t)qi * Hq + g * G + hh) * d + c], dtype);
            rc = attention_f64(qd, kd, vd, L, q_len, G, 1, d, scale, od, NULL);
            double *ob = out + (int64_t)i * q_len * Hq * d;
            for (int qi = 0; qi < q_len && rc == OR_OK; ++qi)
                for (int hh = 0; hh < G; ++hh)
                    memcpy(ob + ((int64_t)qi * Hq + g * G + hh) * d, od + ((int64_t)qi * G + hh) * d,
                           (size_t)d * sizeof(double));
        }
        free(qd);
        free(kd);
        free(vd);
        free(od);
        if (rc != OR_OK) return rc;
    }
    return OR_OK;
}
