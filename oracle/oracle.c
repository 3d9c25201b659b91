/*
 * oracle.c -- plain, slow, fp64 CPU oracle for one decode-maximal hybrid batch
 * run through a LLaMA-style decoder layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark use it.  It shares no code, header, table or helper with the
 * CUDA library; both sides see the same seeded input bytes and nothing else.
 *
 * What it computes (sources are the four public web pages on SARATHI /
 * Sarathi-Serve):
 *
 *  - Row order of the hybrid batch: the chunk's C prefill rows first, then the
 *    D decode rows (SARATHI summary, section 3.4 "Decode-Maximal Batching",
 *    "How fusion works").  Every linear op is applied to every row with the
 *    same weights; rows never mix in a linear op.
 *  - Chunked causal attention: chunk row i sits at absolute position
 *    offset+i and attends to every key at positions 0..offset+i of its own
 *    request -- the cached prefix plus the causal triangle inside the chunk
 *    (SARATHI summary, section 3.4 "Chunked-Prefills", Figure 6, which
 *    states this makes chunked prefill equal to full prefill).
 *  - Decode attention: a decode with S cached tokens attends to S+1 keys, its
 *    cache plus its own new key (Sarathi-Serve Guide, "Deep Dive:
 *    Mathematical Formulation and Attention Mechanics", K_decode of size
 *    (S_i+1) x d_k), i.e. positions 0..S.
 *  - Block-diagonal masking: a query never sees keys of another request, nor
 *    a later key of its own (same Guide section, the unified hybrid mask M,
 *    read as softmax(QK^T/sqrt(d) + M) since M only takes 0 or -inf).
 *  - Paged KV: 16-token blocks (Sarathi-Serve Guide, production checklist,
 *    "Paged KV-Cache Page Sizing"); the physical slot of position p is
 *    block_table[p / bs] * bs + p % bs.  New K/V are written in place
 *    ("committed to the page cache", Guide, "Chunked-Prefills").
 *  - The layer itself (RMSNorm, RoPE rotate-half with theta, SwiGLU) is not
 *    on the pages; it is the LLaMA layer the workloads name (hidden, heads,
 *    FFN, theta 1e4, eps 1e-6), written out here from its textbook
 *    definition.
 *
 * Precision: every accumulation is fp64, bf16 inputs are widened exactly.
 * Two modes:
 *   exact  (mirror = 0): no intermediate rounding at all;
 *   mirror (mirror = 1): round to bf16 (round-to-nearest-even, once, from the
 *          fp64 value) at the points where the GPU stores bf16 tensors:
 *          n1, q and k after RoPE, v, o, h, n2, a, y.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fPIC -shared (no fast-math).
 * OpenMP only splits independent rows / heads across threads; each output
 * value is still a single sequential fp64 sum in index order.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Planted-mistake switch for the mutation tests.  The default build has
 * OR_MUTATE == 0 and no mutation is compiled in. */
#ifndef OR_MUTATE
#define OR_MUTATE 0
#endif

#define OR_OK 0
#define OR_EINVAL -1
#define OR_ERANGE -2

/* ------------------------------------------------------------------ bf16 */

double or_bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round an fp64 value to the nearest bf16 (ties to even) in one step. */
uint16_t or_f64_to_bf16(double d)
{
    float f;
    uint32_t u;
    if (isnan(d))
        return (uint16_t)(signbit(d) ? 0xFFC0u : 0x7FC0u);
    if (fabs(d) >= 0x1p-126 || d == 0.0 || isinf(d)) {
        /* keep 8 significant bits of the fp64 significand */
        uint64_t b;
        memcpy(&b, &d, sizeof b);
        if (!isinf(d)) {
            uint64_t lsb = (b >> 45) & 1u;
            b += (((uint64_t)1 << 44) - 1u) + lsb;
            b &= ~(((uint64_t)1 << 45) - 1u);
        }
        double r;
        memcpy(&r, &b, sizeof r);
        f = (float)r; /* exact, or +-inf past the bf16 range */
    } else {
        /* bf16 subnormals are multiples of 2^-133 */
        double q = nearbyint(d * 0x1p133);
        f = (float)(q * 0x1p-133);
    }
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

static double rbf(double x, int mirror)
{
    return mirror ? or_bf16_to_f64(or_f64_to_bf16(x)) : x;
}

/* ------------------------------------------------------------- layer ops */

/* y[o] = sum_k W[o][k] * x[k], W bf16 row-major [out][in]. */
void or_matvec(const uint16_t *W, int out_dim, int in_dim, const double *x, double *y)
{
    for (int o = 0; o < out_dim; ++o) {
        const uint16_t *w = W + (size_t)o * in_dim;
        double s = 0.0;
        for (int k = 0; k < in_dim; ++k) {
#if OR_MUTATE == 7
            /* planted: transposed operand (reads column o instead of row o) */
            s += or_bf16_to_f64(W[(size_t)k * out_dim + o]) * x[k];
#else
            s += or_bf16_to_f64(w[k]) * x[k];
#endif
        }
        y[o] = s;
    }
}

/* RMSNorm: out = x / sqrt(mean(x^2) + eps) * gamma. */
void or_rmsnorm(const double *x, const uint16_t *gamma, int n, double eps, double *out)
{
    double ss = 0.0;
    for (int i = 0; i < n; ++i)
        ss += x[i] * x[i];
#if OR_MUTATE == 5
    double r = 1.0 / sqrt(ss + eps); /* planted: sum instead of mean */
#else
    double r = 1.0 / sqrt(ss / (double)n + eps);
#endif
    for (int i = 0; i < n; ++i)
        out[i] = x[i] * r * (gamma ? or_bf16_to_f64(gamma[i]) : 1.0);
}

/* RoPE, rotate-half convention: pair (j, j + d/2) rotated by pos * theta^(-2j/d). */
void or_rope(double *v, int d, int pos, double theta)
{
    int half = d / 2;
    for (int j = 0; j < half; ++j) {
        double inv = pow(theta, -2.0 * (double)j / (double)d);
        double a = (double)pos * inv;
        double c = cos(a), s = sin(a);
#if OR_MUTATE == 1
        /* planted: interleaved pairs (2j, 2j+1) */
        double x0 = v[2 * j], x1 = v[2 * j + 1];
        v[2 * j] = x0 * c - x1 * s;
        v[2 * j + 1] = x1 * c + x0 * s;
#elif OR_MUTATE == 2
        /* planted: rotation sign flipped */
        double x0 = v[j], x1 = v[j + half];
        v[j] = x0 * c + x1 * s;
        v[j + half] = x1 * c - x0 * s;
#else
        double x0 = v[j], x1 = v[j + half];
        v[j] = x0 * c - x1 * s;
        v[j + half] = x1 * c + x0 * s;
#endif
    }
}

double or_silu(double z)
{
#if OR_MUTATE == 6
    return 1.0 / (1.0 + exp(-z)); /* planted: sigmoid without the factor z */
#else
    return z / (1.0 + exp(-z));
#endif
}

/* Physical slot of absolute position pos through a block table. */
int or_slot(const int32_t *bt, int n_blocks, int block_size, int num_blocks, int pos)
{
    if (pos < 0)
        return OR_ERANGE;
    int b = pos / block_size;
    if (b >= n_blocks)
        return OR_ERANGE;
    int blk = bt[b];
    if (blk < 0 || blk >= num_blocks)
        return OR_ERANGE;
#if OR_MUTATE == 10
    return blk * block_size + (block_size - 1 - pos % block_size); /* planted: wrong in-block index */
#else
    return blk * block_size + pos % block_size;
#endif
}

/*
 * Attention of one query head over keys at positions 0..last_pos of one
 * request.  q: [d]; k_pool/v_pool: [num_blocks*bs][n_kv][d]; out: [d].
 * scores s_t = q.k_t / sqrt(d); p = softmax(s) (max subtracted); o = sum p_t v_t.
 */
int or_attention_head(const double *q, int d, int kv_head, int n_kv,
                      const double *k_pool, const double *v_pool,
                      const int32_t *bt, int n_blocks, int block_size, int num_blocks,
                      int last_pos, double *out)
{
#if OR_MUTATE == 3
    int n_keys = last_pos; /* planted: the query misses its own key */
#else
    int n_keys = last_pos + 1;
#endif
    if (n_keys <= 0) {
        for (int i = 0; i < d; ++i)
            out[i] = 0.0;
        return OR_OK;
    }
    double *s = (double *)malloc(sizeof(double) * (size_t)n_keys);
    if (!s)
        return OR_EINVAL;
#if OR_MUTATE == 4
    double scale = 1.0; /* planted: missing 1/sqrt(d) */
#else
    double scale = 1.0 / sqrt((double)d);
#endif
    double m = -INFINITY;
    for (int t = 0; t < n_keys; ++t) {
        int slot = or_slot(bt, n_blocks, block_size, num_blocks, t);
        if (slot < 0) {
            free(s);
            return OR_ERANGE;
        }
        const double *k = k_pool + ((size_t)slot * n_kv + kv_head) * d;
        double dot = 0.0;
        for (int i = 0; i < d; ++i)
            dot += q[i] * k[i];
        s[t] = dot * scale;
        if (s[t] > m)
            m = s[t];
    }
    double l = 0.0;
    for (int t = 0; t < n_keys; ++t) {
        s[t] = exp(s[t] - m);
        l += s[t];
    }
    for (int i = 0; i < d; ++i)
        out[i] = 0.0;
    for (int t = 0; t < n_keys; ++t) {
        int slot = or_slot(bt, n_blocks, block_size, num_blocks, t);
        const double *v = v_pool + ((size_t)slot * n_kv + kv_head) * d;
        double p = s[t] / l;
        for (int i = 0; i < d; ++i)
            out[i] += p * v[i];
    }
    free(s);
    return OR_OK;
}

/* ---------------------------------------------------------- layer forward */

typedef struct {
    int hidden, n_heads, n_kv_heads, head_dim, ffn, block_size, num_blocks;
    double rms_eps, rope_theta;
} or_dims;

typedef struct {
    const uint16_t *w_qkv;     /* [(n_heads + 2 n_kv) d][hidden]: q rows, k rows, v rows */
    const uint16_t *w_o;       /* [hidden][n_heads d] */
    const uint16_t *w_gate_up; /* [2 ffn][hidden]: gate rows then up rows */
    const uint16_t *w_down;    /* [hidden][ffn] */
    const uint16_t *norm1;     /* [hidden] */
    const uint16_t *norm2;     /* [hidden] */
} or_layer;

typedef struct {
    int chunk_offset, chunk_len;
    const int32_t *chunk_bt;
    int chunk_n_blocks;
    int n_decodes;
    const int32_t *decode_ctx;   /* [n_decodes] tokens already cached */
    const int32_t *decode_bt;    /* [n_decodes][max_blocks_per_seq] */
    int max_blocks_per_seq;
} or_batch;

/* Optional intermediates, each [T][...] fp64, any may be NULL. */
typedef struct {
    double *q; /* [T][n_heads d], after RoPE */
    double *k; /* [T][n_kv d], after RoPE */
    double *v; /* [T][n_kv d] */
    double *o; /* [T][n_heads d] attention output */
    double *h; /* [T][hidden] after the first residual */
    double *a; /* [T][ffn] silu(g) * u */
    double *n1; /* [T][hidden] RMSNorm-1 output */
    double *n2; /* [T][hidden] RMSNorm-2 output */
} or_aux;

static void row_info(const or_batch *b, int r, int *pos, const int32_t **bt, int *nb)
{
    if (r < b->chunk_len) {
        *pos = b->chunk_offset + r;
        *bt = b->chunk_bt;
        *nb = b->chunk_n_blocks;
    } else {
        int j = r - b->chunk_len;
        *pos = b->decode_ctx[j];
        *bt = b->decode_bt + (size_t)j * b->max_blocks_per_seq;
        *nb = b->max_blocks_per_seq;
    }
}

/*
 * One decoder layer over the rows of one hybrid batch.
 *   x_in, y_out: [T][hidden] fp64, T = chunk_len + n_decodes.
 *   k_pool, v_pool: the oracle's own paged pool, [num_blocks*bs][n_kv][d];
 *     rows' new K/V are written at their slots before any attention reads.
 *   row_sel: NULL for all rows, else a [T] 0/1 mask.  Selecting chunk row i
 *     requires chunk rows 0..i-1 selected too (causality).
 * Returns 0, or a negative error code with nothing guaranteed about outputs.
 */
int oracle_layer_forward(const or_dims *dm, const or_layer *w, int mirror,
                         double *k_pool, double *v_pool, const or_batch *b,
                         const double *x_in, double *y_out, const uint8_t *row_sel,
                         or_aux *aux)
{
    const int H = dm->hidden, nh = dm->n_heads, nkv = dm->n_kv_heads, d = dm->head_dim;
    const int F = dm->ffn, bs = dm->block_size;
    const int T = b->chunk_len + b->n_decodes;
    const int qd = nh * d, kvd = nkv * d, nqkv = qd + 2 * kvd;
    if (H <= 0 || nh <= 0 || nkv <= 0 || d <= 0 || (d & 1) || F <= 0 || bs <= 0 || nh % nkv)
        return OR_EINVAL;
    if (b->chunk_len < 0 || b->n_decodes < 0 || T <= 0 || b->chunk_offset < 0)
        return OR_EINVAL;
    if (row_sel) {
        int seen_gap = 0;
        for (int r = 0; r < b->chunk_len; ++r) {
            if (!row_sel[r])
                seen_gap = 1;
            else if (seen_gap)
                return OR_EINVAL;
        }
    }
    /* validate every row's slot before touching the pool; no two rows of a
     * batch may write the same slot */
    int *slots = (int *)malloc(sizeof(int) * (size_t)T);
    if (!slots)
        return OR_EINVAL;
    for (int r = 0; r < T; ++r) {
        int pos, nb;
        const int32_t *bt;
        row_info(b, r, &pos, &bt, &nb);
        slots[r] = or_slot(bt, nb, bs, dm->num_blocks, pos);
        if (slots[r] < 0) {
            free(slots);
            return OR_ERANGE;
        }
        for (int r2 = 0; r2 < r; ++r2) {
            if (slots[r2] == slots[r]) {
                free(slots);
                return OR_EINVAL;
            }
        }
    }
    free(slots);

    double *q = (double *)calloc((size_t)T * qd, sizeof(double));
    double *o = (double *)calloc((size_t)T * qd, sizeof(double));
    double *hbuf = (double *)calloc((size_t)T * H, sizeof(double));
    if (!q || !o || !hbuf) {
        free(q);
        free(o);
        free(hbuf);
        return OR_EINVAL;
    }

    /* phase 1: norm-1, QKV projection, RoPE, KV append */
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < T; ++r) {
        if (row_sel && !row_sel[r])
            continue;
        int pos, nb;
        const int32_t *bt;
        row_info(b, r, &pos, &bt, &nb);
        double *n1 = (double *)malloc(sizeof(double) * (size_t)H);
        double *qkv = (double *)malloc(sizeof(double) * (size_t)nqkv);
        if (!n1 || !qkv) {
            free(n1);
            free(qkv);
#pragma omp atomic write
            err = 1;
            continue;
        }
        or_rmsnorm(x_in + (size_t)r * H, w->norm1, H, dm->rms_eps, n1);
        for (int i = 0; i < H; ++i)
            n1[i] = rbf(n1[i], mirror);
        if (aux && aux->n1)
            memcpy(aux->n1 + (size_t)r * H, n1, sizeof(double) * (size_t)H);
        or_matvec(w->w_qkv, nqkv, H, n1, qkv);
        for (int hq = 0; hq < nh; ++hq)
            or_rope(qkv + (size_t)hq * d, d, pos, dm->rope_theta);
        for (int hk = 0; hk < nkv; ++hk)
            or_rope(qkv + qd + (size_t)hk * d, d, pos, dm->rope_theta);
        for (int i = 0; i < nqkv; ++i)
            qkv[i] = rbf(qkv[i], mirror);
        memcpy(q + (size_t)r * qd, qkv, sizeof(double) * (size_t)qd);
        int slot = or_slot(bt, nb, bs, dm->num_blocks, pos);
        memcpy(k_pool + (size_t)slot * kvd, qkv + qd, sizeof(double) * (size_t)kvd);
        memcpy(v_pool + (size_t)slot * kvd, qkv + qd + kvd, sizeof(double) * (size_t)kvd);
        if (aux && aux->q)
            memcpy(aux->q + (size_t)r * qd, qkv, sizeof(double) * (size_t)qd);
        if (aux && aux->k)
            memcpy(aux->k + (size_t)r * kvd, qkv + qd, sizeof(double) * (size_t)kvd);
        if (aux && aux->v)
            memcpy(aux->v + (size_t)r * kvd, qkv + qd + kvd, sizeof(double) * (size_t)kvd);
        free(n1);
        free(qkv);
    }
    if (err) {
        free(q);
        free(o);
        free(hbuf);
        return OR_EINVAL;
    }

    /* phase 2: attention, one (row, head) at a time */
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
    for (int r = 0; r < T; ++r) {
        for (int hq = 0; hq < nh; ++hq) {
            if (row_sel && !row_sel[r])
                continue;
            int pos, nb;
            const int32_t *bt;
            row_info(b, r, &pos, &bt, &nb);
            int kvh = hq / (nh / nkv);
            int rc = or_attention_head(q + (size_t)r * qd + (size_t)hq * d, d, kvh, nkv,
                                       k_pool, v_pool, bt, nb, bs, dm->num_blocks, pos,
                                       o + (size_t)r * qd + (size_t)hq * d);
            if (rc) {
#pragma omp atomic write
                err = 1;
            }
#if OR_MUTATE != 12
            for (int i = 0; i < d; ++i)
                o[(size_t)r * qd + (size_t)hq * d + i] =
                    rbf(o[(size_t)r * qd + (size_t)hq * d + i], mirror);
#endif /* planted (12): the mirror keeps o unrounded */
        }
    }
    if (err) {
        free(q);
        free(o);
        free(hbuf);
        return OR_ERANGE;
    }

    /* phase 3: O-proj + residual, norm-2, gate/up + SwiGLU, down + residual */
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < T; ++r) {
        if (row_sel && !row_sel[r])
            continue;
        const double *x = x_in + (size_t)r * H;
        double *hr = hbuf + (size_t)r * H;
        double *tmp = (double *)malloc(sizeof(double) * (size_t)H);
        double *n2 = (double *)malloc(sizeof(double) * (size_t)H);
        double *gu = (double *)malloc(sizeof(double) * (size_t)2 * F);
        double *act = (double *)malloc(sizeof(double) * (size_t)F);
        if (!tmp || !n2 || !gu || !act) {
            free(tmp);
            free(n2);
            free(gu);
            free(act);
#pragma omp atomic write
            err = 1;
            continue;
        }
        or_matvec(w->w_o, H, qd, o + (size_t)r * qd, tmp);
        for (int i = 0; i < H; ++i) {
#if OR_MUTATE == 8
            hr[i] = rbf(tmp[i], mirror); /* planted: residual dropped */
#else
            hr[i] = rbf(x[i] + tmp[i], mirror);
#endif
        }
        or_rmsnorm(hr, w->norm2, H, dm->rms_eps, n2);
#if OR_MUTATE != 11
        for (int i = 0; i < H; ++i)
            n2[i] = rbf(n2[i], mirror);
#endif /* planted (11): the mirror keeps n2 unrounded */
        if (aux && aux->n2)
            memcpy(aux->n2 + (size_t)r * H, n2, sizeof(double) * (size_t)H);
        or_matvec(w->w_gate_up, 2 * F, H, n2, gu);
        for (int j = 0; j < F; ++j) {
#if OR_MUTATE == 9
            act[j] = rbf(or_silu(gu[F + j]) * gu[j], mirror); /* planted: gate/up swapped */
#else
            act[j] = rbf(or_silu(gu[j]) * gu[F + j], mirror);
#endif
        }
        or_matvec(w->w_down, H, F, act, tmp);
        for (int i = 0; i < H; ++i)
            y_out[(size_t)r * H + i] = rbf(hr[i] + tmp[i], mirror);
        if (aux && aux->a)
            memcpy(aux->a + (size_t)r * F, act, sizeof(double) * (size_t)F);
        free(tmp);
        free(n2);
        free(gu);
        free(act);
    }
    if (aux && aux->o)
        memcpy(aux->o, o, sizeof(double) * (size_t)T * qd);
    if (aux && aux->h)
        memcpy(aux->h, hbuf, sizeof(double) * (size_t)T * H);
    free(q);
    free(o);
    free(hbuf);
    return err ? OR_EINVAL : OR_OK;
}

/* Threads OpenMP will use (1 when built without OpenMP). */
int or_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void or_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}
