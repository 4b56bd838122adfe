/*
 * dsa_oracle.c -- plain, slow, single-threaded CPU oracle for the DSA
 * "score, select, sparse read" path (lightweight indexer -> Top-K -> sparse
 * MLA attention).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library links, includes or calls
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline
 * leg load it.  It shares no header, helper, table or constant with the CUDA
 * path: every codec below is written out from the format definitions.
 *
 * What it computes, and where the pages define it:
 *
 *  - Indexer score ("Day-0 Inference Adaptation and Optimization for Hybrid
 *    Attention Architectures", §1 sparse attention branch and §3 Optimization 1;
 *    "Optimizing Inference for Hybrid Attention LLMs: A Practical Guide to Day-0
 *    Adaptation", §3.1 Indexer Fusion; "Day0 Inference Support and Performance
 *    Optimization for New-Architecture LLMs", §4 item 1): every causal history
 *    position s of query t gets
 *        score[t][s] = sum_j w[t][j] * ReLU( q[t][j] . k[s] )
 *    i.e. a per-head dot product, a per-head activation and a learnable
 *    cross-head weighting.  Operands are decoded exactly, products and sums are
 *    accumulated in double, and the result is rounded to float once.
 *  - Top-K selection (same passages): the K highest scores among positions
 *    0..pos(t); equal scores are ordered by lower position first; fewer than K
 *    valid positions return all of them, the rest of the row is -1.
 *  - Sparse MLA attention ("Day0 Inference Support and Performance
 *    Optimization for New-Architecture LLMs", §2 item 2 and §4 "Sparse
 *    attention reads by index"; "Day0 Inference Optimization for a New Hybrid
 *    Attention Architecture: A Full-Stack Deep Dive", operator fusion item 1):
 *    softmax attention of every query head over the selected latent KV rows
 *    only; logits scale*(q . kv[0:D]), values kv[0:Dv].  Computed in double.
 *  - Quantisation codecs ("Day-0 Inference Adaptation and Optimization for
 *    Hybrid Attention Architectures", §4 Optimization 2; "Day0 Inference
 *    Adaptation and Performance Optimization for a Sparse Hybrid Architecture
 *    LLM", §3.1): MXFP8 with one power-of-two scale per 32 elements for the
 *    index Q/K, and FP8 E4M3 for the main KV cache (per-row fp32 scale on the
 *    512 latent dims, rope dims kept bf16).  Element and scale encodings follow
 *    the OCP 8-bit floating point and OCP Microscaling v1.0 definitions.
 *  - FP8 KV at the pages' per-token-head-tile granularity ("Day-0 Inference
 *    Adaptation and Optimization for Hybrid Attention Architectures", §4
 *    Optimization 2; "Optimizing Inference for Hybrid Attention LLMs: A
 *    Practical Guide to Day-0 Adaptation", §4 Hierarchical Quantization;
 *    "Day0 Inference Support and Performance Optimization for New-Architecture
 *    LLMs", §5 Tiered Quantization, item 2): within each token's
 *    latent row every tile of 128 consecutive elements has its own scale, so
 *    the 512 latent dims carry four fp32 scales; each tile uses the row rule
 *    above on its own amax.  The rope dims stay bf16.
 *  - Cache append ("Optimizing Inference for Hybrid Attention LLMs: A
 *    Practical Guide to Day-0 Adaptation", §4 key points 1-2): new tokens'
 *    index keys and latent rows quantised by the codecs above straight into
 *    their page slots.
 *
 * Every function here is pinned by a CPU test against something other than
 * itself (brute force, closed forms, library routines on special cases,
 * invariants); see tests/test_oracle_*.py.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

#define ORC_IDX_BF16 0
#define ORC_IDX_MXFP8 1
#define ORC_KV_BF16 0
#define ORC_KV_FP8_ROWSCALE 1
#define ORC_KV_FP8_TILE128 2

/* ------------------------------------------------------------------------ */
/* Scalar codecs, from the format definitions.                              */
/* ------------------------------------------------------------------------ */

/* bfloat16 is the upper half of an IEEE-754 binary32: widen exactly. */
double orc_bf16_to_f64(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP FP8 E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits.  No infinities;
 * S.1111.111 is NaN.  Exponent field 0 holds subnormals m/8 * 2^-6. */
double orc_e4m3_to_f64(uint8_t c)
{
    int s = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* Round-half-to-even of a non-negative double to an integer-valued double. */
static double orc_rne(double a)
{
    double f = floor(a);
    double r = a - f;
    if (r > 0.5)
        return f + 1.0;
    if (r < 0.5)
        return f;
    return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* Encode to E4M3 with round-to-nearest-even, saturating to +-448 (the largest
 * finite E4M3 magnitude, 1.75 * 2^8).  NaN maps to the positive NaN code. */
uint8_t orc_f64_to_e4m3_sat(double x)
{
    uint8_t sign;
    double a;
    int e, q;
    if (isnan(x))
        return 0x7F;
    sign = (x < 0.0 || (x == 0.0 && signbit(x))) ? 0x80 : 0x00;
    a = fabs(x);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: units of 2^-9; q == 8 is the smallest normal,
         * whose code (exponent 1, mantissa 0) is numerically 8 as well */
        q = (int)orc_rne(ldexp(a, 9));
        return (uint8_t)(sign | q);
    }
    (void)frexp(a, &e); /* a = f * 2^e, f in [0.5, 1) */
    e -= 1;             /* a = (1 + t) * 2^e, t in [0, 1) */
    q = (int)orc_rne((ldexp(a, -e) - 1.0) * 8.0);
    if (q == 8) {
        q = 0;
        e += 1;
    }
    /* a < 448 guarantees e + 7 <= 15 and never the NaN code */
    return (uint8_t)(sign | ((e + 7) << 3) | q);
}

/* OCP MX E8M0 scale: 2^(byte-127); byte 255 is NaN. */
double orc_e8m0_to_f64(uint8_t b)
{
    if (b == 0xFF)
        return NAN;
    return ldexp(1.0, (int)b - 127);
}

/* ------------------------------------------------------------------------ */
/* Quantisers.                                                              */
/* ------------------------------------------------------------------------ */

/* MXFP8 (OCP Microscaling v1.0, E4M3 elements, block of 32): for each block
 * of 32 consecutive elements, X = floor(log2(amax)) - 8 (8 is the exponent of
 * E4M3's largest normal), scale byte = X + 127 clamped to [0, 254], element =
 * E4M3_rne_sat(x / 2^X).  A block whose amax is 0 gets scale byte 127 and zero
 * elements.  n must be a multiple of 32. */
void orc_quant_mxfp8(const uint16_t *x, int64_t n, uint8_t *q, uint8_t *e8m0)
{
    int64_t b, i;
    for (b = 0; b < n / 32; ++b) {
        double amax = 0.0;
        int X, byte, e;
        for (i = 0; i < 32; ++i) {
            double v = fabs(orc_bf16_to_f64(x[b * 32 + i]));
            if (v > amax)
                amax = v;
        }
        if (amax == 0.0) {
            e8m0[b] = 127;
            for (i = 0; i < 32; ++i)
                q[b * 32 + i] = 0;
            continue;
        }
        (void)frexp(amax, &e);
        X = (e - 1) - 8;
        byte = X + 127;
        if (byte < 0)
            byte = 0;
        if (byte > 254)
            byte = 254;
        X = byte - 127;
        e8m0[b] = (uint8_t)byte;
        for (i = 0; i < 32; ++i)
            q[b * 32 + i] = orc_f64_to_e4m3_sat(ldexp(orc_bf16_to_f64(x[b * 32 + i]), -X));
    }
}

/* FP8 KV row quantiser: a 576-wide bf16 latent row is split into 512 "nope"
 * dims stored as E4M3 with one fp32 scale per row and 64 rope dims kept bf16.
 * s = fl32(amax / 448) (amax over the 512 dims; s = 1 when amax is 0) and
 * element = E4M3_rne_sat(fl32(x / s)), both divisions in binary32. */
void orc_quant_fp8_rows(const uint16_t *kv, int64_t rows, uint8_t *nope, uint16_t *rope, float *scale)
{
    int64_t r;
    int d;
    for (r = 0; r < rows; ++r) {
        const uint16_t *row = kv + r * 576;
        float amax = 0.0f, s;
        for (d = 0; d < 512; ++d) {
            float v = (float)fabs(orc_bf16_to_f64(row[d]));
            if (v > amax)
                amax = v;
        }
        s = (amax == 0.0f) ? 1.0f : amax / 448.0f;
        scale[r] = s;
        for (d = 0; d < 512; ++d) {
            float xv = (float)orc_bf16_to_f64(row[d]);
            float y = xv / s;
            nope[r * 512 + d] = orc_f64_to_e4m3_sat((double)y);
        }
        for (d = 0; d < 64; ++d)
            rope[r * 64 + d] = row[512 + d];
    }
}

/* ------------------------------------------------------------------------ */
/* Paged cache addressing.                                                  */
/* ------------------------------------------------------------------------ */

/* Logical position s of a sequence lives in physical row
 * page_table_row[s / page_size] * page_size + s % page_size.
 * Returns -1 if the page id is outside [0, num_pages). */
static int64_t orc_phys_row(const int32_t *pt_row, int32_t page_size, int64_t num_pages, int64_t s)
{
    int64_t page = pt_row[s / page_size];
    if (page < 0 || page >= num_pages)
        return -1;
    return page * (int64_t)page_size + s % page_size;
}

/* Absolute position of query i of sequence b: the queries of a sequence are
 * its last (cu_q[b+1]-cu_q[b]) positions. */
static int64_t orc_query_pos(const int32_t *seq_lens, const int32_t *cu_q, int b, int64_t t)
{
    int64_t nq = cu_q[b + 1] - cu_q[b];
    return (int64_t)seq_lens[b] - nq + (t - cu_q[b]);
}

static int orc_seq_of(const int32_t *cu_q, int B, int64_t t)
{
    int b;
    for (b = 0; b < B; ++b)
        if (t >= cu_q[b] && t < cu_q[b + 1])
            return b;
    return -1;
}

/* ------------------------------------------------------------------------ */
/* Indexer scores.                                                          */
/* ------------------------------------------------------------------------ */

static double orc_idx_elem(int dtype, const void *base, const uint8_t *scales, int64_t row, int d_I, int d)
{
    if (dtype == ORC_IDX_BF16)
        return orc_bf16_to_f64(((const uint16_t *)base)[row * d_I + d]);
    return orc_e4m3_to_f64(((const uint8_t *)base)[row * d_I + d]) *
           orc_e8m0_to_f64(scales[row * (d_I / 32) + d / 32]);
}

/* Scores of one query against positions 0..n_pos-1 of its sequence.
 * q and q_scale point at the query's [H_I, d_I] block (and [H_I, d_I/32]
 * scale bytes for MXFP8); w at its [H_I] head weights.  Returns 0, or -1 if a
 * page id is out of range. */
int orc_index_scores_row(int dtype, int H_I, int d_I, const void *q, const uint8_t *q_scale, const float *w,
                         const void *k_cache, const uint8_t *k_scale, int64_t num_pages, const int32_t *pt_row,
                         int32_t page_size, int64_t n_pos, float *scores)
{
    int64_t s;
    int j, d;
    double *qd = (double *)malloc(sizeof(double) * (size_t)H_I * (size_t)d_I);
    double *kd = (double *)malloc(sizeof(double) * (size_t)d_I);
    if (!qd || !kd) {
        free(qd);
        free(kd);
        return -2;
    }
    for (j = 0; j < H_I; ++j)
        for (d = 0; d < d_I; ++d)
            qd[j * d_I + d] = orc_idx_elem(dtype, q, q_scale, j, d_I, d);
    for (s = 0; s < n_pos; ++s) {
        int64_t row = orc_phys_row(pt_row, page_size, num_pages, s);
        double acc = 0.0;
        if (row < 0) {
            free(qd);
            free(kd);
            return -1;
        }
        for (d = 0; d < d_I; ++d)
            kd[d] = orc_idx_elem(dtype, k_cache, k_scale, row, d_I, d);
        for (j = 0; j < H_I; ++j) {
            double dot = 0.0;
            for (d = 0; d < d_I; ++d)
                dot += qd[j * d_I + d] * kd[d];
            if (dot > 0.0)
                acc += (double)w[j] * dot;
        }
        scores[s] = (float)acc;
    }
    free(qd);
    free(kd);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Top-K by full sort.                                                      */
/* ------------------------------------------------------------------------ */

typedef struct {
    float v;
    int32_t i;
} orc_pair;

/* Higher score first; equal scores (including -0 == +0) by lower position. */
static int orc_pair_cmp(const void *a, const void *b)
{
    const orc_pair *x = (const orc_pair *)a, *y = (const orc_pair *)b;
    if (x->v > y->v)
        return -1;
    if (x->v < y->v)
        return 1;
    return (x->i < y->i) ? -1 : (x->i > y->i);
}

/* Top-K of scores[0..n-1]: writes min(K, n) positions, sorted ascending, to
 * out[0..], pads out[min(K,n)..K-1] with -1 and returns min(K, n). */
static int orc_int_cmp(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

int orc_topk_row(const float *scores, int64_t n, int32_t K, int32_t *out)
{
    int64_t i, m = n < K ? n : K;
    orc_pair *p = (orc_pair *)malloc(sizeof(orc_pair) * (size_t)(n > 0 ? n : 1));
    if (!p)
        return -2;
    for (i = 0; i < n; ++i) {
        p[i].v = scores[i];
        p[i].i = (int32_t)i;
    }
    qsort(p, (size_t)n, sizeof(orc_pair), orc_pair_cmp);
    for (i = 0; i < m; ++i)
        out[i] = p[i].i;
    qsort(out, (size_t)m, sizeof(int32_t), orc_int_cmp);
    for (i = m; i < K; ++i)
        out[i] = -1;
    free(p);
    return (int)m;
}

/* Top-K over R rows of a score matrix with row stride ld; row r is valid up to
 * lens[r] entries.  out is [R, K]. */
int orc_topk_rows(const float *scores, int64_t ld, const int32_t *lens, int32_t R, int32_t K, int32_t *out)
{
    int32_t r;
    for (r = 0; r < R; ++r)
        if (orc_topk_row(scores + (int64_t)r * ld, lens[r], K, out + (int64_t)r * K) < 0)
            return -2;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Fused indexer + Top-K over a batch of queries.                           */
/* ------------------------------------------------------------------------ */

/* For each requested query row t (rows == NULL means all T rows, else the
 * n_rows listed), compute the scores of positions 0..pos(t) and select the
 * top K.  indices is [n_rows, K] (or [T, K]); scores_out, if not NULL, is
 * [n_rows, ld_scores] and receives the raw scores.  Returns 0, -1 on a bad
 * page id, -3 on a bad query layout. */
int orc_index_topk(int dtype, int H_I, int d_I, const void *q_idx, const uint8_t *q_scale, const float *head_w,
                   const void *k_cache, const uint8_t *k_scale, int64_t num_pages, const int32_t *page_table,
                   int32_t max_pages_per_seq, const int32_t *seq_lens, const int32_t *cu_q, int32_t B, int32_t T,
                   int32_t K, int32_t page_size, const int32_t *rows, int32_t n_rows, int32_t *indices,
                   float *scores_out, int64_t ld_scores)
{
    int32_t r, count = rows ? n_rows : T;
    for (r = 0; r < count; ++r) {
        int64_t t = rows ? rows[r] : r;
        int b = orc_seq_of(cu_q, B, t);
        int64_t pos, n_pos;
        float *sc;
        int rc;
        size_t qoff;
        if (b < 0)
            return -3;
        pos = orc_query_pos(seq_lens, cu_q, b, t);
        if (pos < 0)
            return -3;
        n_pos = pos + 1;
        sc = (float *)malloc(sizeof(float) * (size_t)n_pos);
        if (!sc)
            return -2;
        qoff = (size_t)t * (size_t)H_I * (size_t)d_I;
        rc = orc_index_scores_row(dtype, H_I, d_I,
                                  dtype == ORC_IDX_BF16 ? (const void *)((const uint16_t *)q_idx + qoff)
                                                        : (const void *)((const uint8_t *)q_idx + qoff),
                                  q_scale ? q_scale + qoff / 32 : NULL, head_w + (size_t)t * H_I, k_cache, k_scale,
                                  num_pages, page_table + (int64_t)b * max_pages_per_seq, page_size, n_pos, sc);
        if (rc != 0) {
            free(sc);
            return rc;
        }
        if (scores_out) {
            int64_t s;
            for (s = 0; s < n_pos && s < ld_scores; ++s)
                scores_out[(int64_t)r * ld_scores + s] = sc[s];
        }
        if (orc_topk_row(sc, n_pos, K, indices + (int64_t)r * K) < 0) {
            free(sc);
            return -2;
        }
        free(sc);
    }
    return 0;
}

/* FP8 KV tile quantiser: as orc_quant_fp8_rows, but every tile of 128
 * latent dims (dims 128j..128j+127, j = 0..3) has its own scale
 * scale[r*4 + j] = fl32(amax_j / 448) (1 when amax_j is 0), and its elements
 * are E4M3_rne_sat(fl32(x / scale[r*4 + j])). */
void orc_quant_fp8_tiles(const uint16_t *kv, int64_t rows, uint8_t *nope, uint16_t *rope, float *scale)
{
    int64_t r;
    int j, d;
    for (r = 0; r < rows; ++r) {
        const uint16_t *row = kv + r * 576;
        for (j = 0; j < 4; ++j) {
            float amax = 0.0f, s;
            for (d = 128 * j; d < 128 * (j + 1); ++d) {
                float v = (float)fabs(orc_bf16_to_f64(row[d]));
                if (v > amax)
                    amax = v;
            }
            s = (amax == 0.0f) ? 1.0f : amax / 448.0f;
            scale[r * 4 + j] = s;
            for (d = 128 * j; d < 128 * (j + 1); ++d) {
                float xv = (float)orc_bf16_to_f64(row[d]);
                float y = xv / s;
                nope[r * 512 + d] = orc_f64_to_e4m3_sat((double)y);
            }
        }
        for (d = 0; d < 64; ++d)
            rope[r * 64 + d] = row[512 + d];
    }
}

/* ------------------------------------------------------------------------ */
/* Sparse MLA attention.                                                    */
/* ------------------------------------------------------------------------ */

/* Latent row element d of physical row `row` (d < D). */
static double orc_kv_elem(int dtype, const void *kv, const uint16_t *kv_rope, const float *kv_scale, int D,
                          int64_t row, int d)
{
    if (dtype == ORC_KV_BF16)
        return orc_bf16_to_f64(((const uint16_t *)kv)[row * D + d]);
    if (d < 512 && dtype == ORC_KV_FP8_TILE128)
        return orc_e4m3_to_f64(((const uint8_t *)kv)[row * 512 + d]) * (double)kv_scale[row * 4 + d / 128];
    if (d < 512)
        return orc_e4m3_to_f64(((const uint8_t *)kv)[row * 512 + d]) * (double)kv_scale[row];
    return orc_bf16_to_f64(kv_rope[row * 64 + (d - 512)]);
}

/* One query row: out[h][0..Dv) = sum_i p_{h,i} kv_i[0..Dv), p = softmax_i of
 * scale * (q_h . kv_i[0..D)) over the valid entries idx[0..K) (entries < 0
 * are skipped).  q is [H, D] bf16, out [H, Dv] and lse [H] in fp32 (lse may
 * be NULL; natural log).  With no valid entry the output row is 0 and lse is
 * -inf.  Returns 0, or -1 on a bad page / position. */
int orc_sparse_mla_row(int dtype, int H, int D, int Dv, const uint16_t *q, const void *kv, const uint16_t *kv_rope,
                       const float *kv_scale, int64_t num_pages, const int32_t *pt_row, int32_t page_size,
                       const int32_t *idx, int32_t K, double scale, float *out, float *lse)
{
    int32_t i, nv = 0;
    int h, d;
    double *kvd, *logit, *acc;
    for (i = 0; i < K; ++i)
        if (idx[i] >= 0)
            ++nv;
    kvd = (double *)malloc(sizeof(double) * (size_t)(nv > 0 ? nv : 1) * (size_t)D);
    logit = (double *)malloc(sizeof(double) * (size_t)(nv > 0 ? nv : 1));
    acc = (double *)malloc(sizeof(double) * (size_t)Dv);
    if (!kvd || !logit || !acc) {
        free(kvd);
        free(logit);
        free(acc);
        return -2;
    }
    nv = 0;
    for (i = 0; i < K; ++i) {
        int64_t row;
        if (idx[i] < 0)
            continue;
        row = orc_phys_row(pt_row, page_size, num_pages, idx[i]);
        if (row < 0) {
            free(kvd);
            free(logit);
            free(acc);
            return -1;
        }
        for (d = 0; d < D; ++d)
            kvd[(int64_t)nv * D + d] = orc_kv_elem(dtype, kv, kv_rope, kv_scale, D, row, d);
        ++nv;
    }
    for (h = 0; h < H; ++h) {
        double mx = -INFINITY, sum = 0.0;
        for (i = 0; i < nv; ++i) {
            double dot = 0.0;
            for (d = 0; d < D; ++d)
                dot += orc_bf16_to_f64(q[h * D + d]) * kvd[(int64_t)i * D + d];
            logit[i] = scale * dot;
            if (logit[i] > mx)
                mx = logit[i];
        }
        for (d = 0; d < Dv; ++d)
            acc[d] = 0.0;
        for (i = 0; i < nv; ++i) {
            double p = exp(logit[i] - mx);
            sum += p;
            for (d = 0; d < Dv; ++d)
                acc[d] += p * kvd[(int64_t)i * D + d];
        }
        for (d = 0; d < Dv; ++d)
            out[h * Dv + d] = nv > 0 ? (float)(acc[d] / sum) : 0.0f;
        if (lse)
            lse[h] = nv > 0 ? (float)(mx + log(sum)) : -INFINITY;
    }
    free(kvd);
    free(logit);
    free(acc);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Cache append.                                                            */
/* ------------------------------------------------------------------------ */

/* New tokens' index keys and latent rows written into their page slots, each
 * quantised on the way in to the cache's format ("Optimizing Inference for
 * Hybrid Attention LLMs: A Practical Guide to Day-0 Adaptation", §4
 * Hierarchical Quantization, key points 1 and 2: per-token block formats that
 * line up with the page layout, quantised on the indexer's data path with no
 * extra round trip).  Token t of sequence b (t in cu_q[b]..cu_q[b+1]-1) is at
 * position seq_lens[b] - (cu_q[b+1] - cu_q[b]) + (t - cu_q[b]), i.e. the new
 * tokens are the last positions of their sequence, as queries are.
 *   k_new [T, 128] bf16 -> k_cache: bf16 [rows, 128], or MXFP8 codes
 *                          [rows, 128] with e8m0 k_scale [rows, 4]
 *   kv_new [T, 576] bf16 -> kv_cache: bf16 [rows, 576], or FP8 e4m3 [rows, 512]
 *                          with kv_rope [rows, 64] bf16 and kv_scale [rows]
 *                          (row scales) or [rows, 4] (tile scales)
 * Either pair may be NULL (that cache is not written).  Returns 0, or -1 on a
 * page id outside [0, num_pages) or a negative position (nothing is written
 * for that token), -3 on a token outside cu_q. */
int orc_cache_append(const uint16_t *k_new, const uint16_t *kv_new, const int32_t *page_table,
                     int32_t max_pages_per_seq, const int32_t *seq_lens, const int32_t *cu_q, int32_t B, int32_t T,
                     int32_t page_size, int64_t num_pages, int idx_dtype, void *k_cache, uint8_t *k_scale,
                     int kv_dtype, void *kv_cache, uint16_t *kv_rope, float *kv_scale)
{
    int32_t t;
    int rc = 0, d;
    for (t = 0; t < T; ++t) {
        int b = orc_seq_of(cu_q, B, t);
        int64_t pos, row;
        if (b < 0)
            return -3;
        pos = orc_query_pos(seq_lens, cu_q, b, t);
        row = pos < 0 ? -1 : orc_phys_row(page_table + (int64_t)b * max_pages_per_seq, page_size, num_pages, pos);
        if (row < 0) {
            rc = -1;
            continue;
        }
        if (k_new && k_cache) {
            const uint16_t *src = k_new + (int64_t)t * 128;
            if (idx_dtype == ORC_IDX_BF16)
                for (d = 0; d < 128; ++d)
                    ((uint16_t *)k_cache)[row * 128 + d] = src[d];
            else
                orc_quant_mxfp8(src, 128, (uint8_t *)k_cache + row * 128, k_scale + row * 4);
        }
        if (kv_new && kv_cache) {
            const uint16_t *src = kv_new + (int64_t)t * 576;
            if (kv_dtype == ORC_KV_BF16)
                for (d = 0; d < 576; ++d)
                    ((uint16_t *)kv_cache)[row * 576 + d] = src[d];
            else if (kv_dtype == ORC_KV_FP8_TILE128)
                orc_quant_fp8_tiles(src, 1, (uint8_t *)kv_cache + row * 512, kv_rope + row * 64, kv_scale + row * 4);
            else
                orc_quant_fp8_rows(src, 1, (uint8_t *)kv_cache + row * 512, kv_rope + row * 64, kv_scale + row);
        }
    }
    return rc;
}

/* Batch driver: query rows t (rows == NULL: all T) of q [T, H, D]; indices
 * [T, K]; out [n_rows, H, Dv]; lse [n_rows, H] or NULL. */
int orc_sparse_mla(int dtype, int H, int D, int Dv, const uint16_t *q, const void *kv, const uint16_t *kv_rope,
                   const float *kv_scale, int64_t num_pages, const int32_t *page_table, int32_t max_pages_per_seq,
                   const int32_t *cu_q, int32_t B, int32_t T, const int32_t *indices, int32_t K, double scale,
                   int32_t page_size, const int32_t *rows, int32_t n_rows, float *out, float *lse)
{
    int32_t r, count = rows ? n_rows : T;
    for (r = 0; r < count; ++r) {
        int64_t t = rows ? rows[r] : r;
        int b = orc_seq_of(cu_q, B, t);
        int rc;
        if (b < 0)
            return -3;
        rc = orc_sparse_mla_row(dtype, H, D, Dv, q + t * (int64_t)H * D, kv, kv_rope, kv_scale, num_pages,
                                page_table + (int64_t)b * max_pages_per_seq, page_size, indices + t * (int64_t)K, K,
                                scale, out + (int64_t)r * H * Dv, lse ? lse + (int64_t)r * H : NULL);
        if (rc != 0)
            return rc;
    }
    return 0;
}
