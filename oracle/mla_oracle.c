/* CPU oracle for MLA prefill attention.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the bench's
 * cpu_baseline leg may load this file's library. It shares no code, header,
 * table or constant with the CUDA library; it is the plain definition of what
 * that library computes, written out in fp64 with no blocking, fusion or
 * reordering, so that it can be checked against the source pages by eye.
 *
 * Sources (page title, section):
 *  - "More throughput from fewer GPUs: profiling and fixing GLM-5.3 prefill
 *    on NVIDIA B300", section System architecture: multi-head latent
 *    attention keeps one latent vector per token, shared by all heads; the KV
 *    cache is FP8. Section KV hand-off and caching: 256-token KV chunks.
 *  - "GLM-5.3-Optimierungen, Teil 2: PCP, DCP und Hybrid HiSparse auf 16
 *    H200s", section "Warum nicht TP oder DP?": all 64 heads read one latent
 *    row; the indexer scores every earlier token and keeps 2,048. Section
 *    Ausprobieren: sparse MLA runs as MQA, each KV row serving every head.
 *    Footnote 1: QK runs over 576 dims and PV over 512. Footnote 3: indexer
 *    keys are 128 FP8 values plus a 4-byte scale.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - Weight-absorbed form: query row q (576 = 512 latent + 64 RoPE dims, RoPE
 *    already applied) against key K_s = sigma_s * dec(c_s) (576 dims) and value
 *    V_s = first 512 dims of K_s. The head's W_UV is applied outside.
 *  - Causal with a cached prefix: new token i of a sequence with prefix P sits
 *    at position p = P + i and attends to positions 0..p (itself included).
 *  - FP8 is OCP e4m3fn; one fp32 scale per cached token. The 656-byte row of
 *    GLM-5.3 Teil 2, footnote 1, is read as 512 e4m3 latent codes, one fp32
 *    scale per 128 latent dims and 64 bf16 RoPE values.
 *  - Indexer: score(t,s) = sigmaI_s * sum_h w_{t,h} * max(0, q_{t,h} . k_s),
 *    s <= p; the selected set is the first min(topk, p+1) positions in the
 *    order (score descending, position ascending).
 *  - Merge of partial results (DCP section of GLM-5.3 Teil 2): out and lse of
 *    attention over a union of disjoint key sets from each set's out and lse.
 *  - Non-absorbed (MHA) form for short prompts (GLM-5.3 Teil 2, section
 *    Ausprobieren: without the sparse_mla_force_mqa flag, prefill batches whose
 *    prompts fit within the top-k of 2,048 tokens take the dense MHA path): per
 *    head the latent row is up-projected into a 128-dim no-RoPE key and a
 *    128-dim value; the key gets the 64 shared RoPE dims appended (192 dims).
 *  - Cache write (the step before attention): per token and row, scale =
 *    absmax / 448 (1 for a zero row, at least 2^-126 otherwise), codes =
 *    nearest e4m3 of x times the reciprocal of the scale, ties to even,
 *    clamped at 448; every step in IEEE binary32.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORA_PAGE 256
#define ORA_DQK 576
#define ORA_DV 512
#define ORA_DIDX 128

static double e4m3_table[256];
static int table_ready = 0;

/* OCP e4m3fn from its bit fields: sign s (bit 7), exponent e (bits 6..3, bias
 * 7), mantissa m (bits 2..0). e = 0 is subnormal: m/8 * 2^-6. e = 15, m = 7 is
 * NaN. Everything else is (1 + m/8) * 2^(e - 7). There is no infinity. */
static double e4m3_from_fields(unsigned code) {
    unsigned s = (code >> 7) & 1u, e = (code >> 3) & 15u, m = code & 7u;
    double mag;
    if (e == 15u && m == 7u) return NAN;
    if (e == 0u)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return s ? -mag : mag;
}

static void ora_init(void) {
    if (table_ready) return;
    for (unsigned c = 0; c < 256; ++c) e4m3_table[c] = e4m3_from_fields(c);
    table_ready = 1;
}

double ora_e4m3(uint8_t code) {
    ora_init();
    return e4m3_table[code];
}

/* bfloat16: the IEEE binary32 value whose upper 16 bits are b. */
double ora_bf16(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

void ora_bf16_to_f64(const uint16_t *b, int64_t n, double *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = ora_bf16(b[i]);
}

/* Sequence b and in-sequence index i of global new-token t; -1 if out of range. */
static int locate(int32_t batch, const int32_t *cu, int64_t t, int64_t *i_out) {
    for (int b = 0; b < batch; ++b)
        if (t >= cu[b] && t < cu[b + 1]) {
            *i_out = t - cu[b];
            return b;
        }
    return -1;
}

/* Physical row (page*256 + slot) of position s of sequence b; -1 if unmapped. */
static int64_t cache_row(const int32_t *bt, int32_t max_blocks, int32_t num_blocks, int b, int64_t s) {
    int64_t blk = s / ORA_PAGE;
    if (blk >= max_blocks) return -1;
    int32_t page = bt[(int64_t)b * max_blocks + blk];
    if (page < 0 || page >= num_blocks) return -1;
    return (int64_t)page * ORA_PAGE + s % ORA_PAGE;
}

/* Cache row formats. ORA_FMT_580: 576 e4m3 codes in kv (row r at r*576) and one
 * fp32 scale per row in kv_scale: K[d] = sigma_r * dec(c[d]). ORA_FMT_656 (the
 * 656-byte row of GLM-5.3 Teil 2, footnote 1, read as 512 e4m3 latent codes,
 * four fp32 scales, one per 128 dims, then 64 bf16 RoPE values, little-endian):
 * K[d] = sigma_{r,d/128} * dec(c[d]) for d < 512, K[512+i] = bf16 value i. */
#define ORA_FMT_580 0
#define ORA_FMT_656 1
#define ORA_ROW656 656

static float f32_le(const uint8_t *p) {
    uint32_t u = (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* The 576 key values of cache row r. */
static void decode_row(int fmt, const uint8_t *kv, const float *kv_scale, int64_t r, double *k) {
    if (fmt == ORA_FMT_580) {
        const uint8_t *c = kv + r * ORA_DQK;
        double sigma = (double)kv_scale[r];
        for (int d = 0; d < ORA_DQK; ++d) k[d] = sigma * e4m3_table[c[d]];
    } else {
        const uint8_t *row = kv + r * ORA_ROW656;
        for (int d = 0; d < ORA_DV; ++d) k[d] = (double)f32_le(row + ORA_DV + 4 * (d / 128)) * e4m3_table[row[d]];
        for (int i = 0; i < ORA_DQK - ORA_DV; ++i)
            k[ORA_DV + i] = ora_bf16((uint16_t)(row[ORA_DV + 16 + 2 * i] | (row[ORA_DV + 17 + 2 * i] << 8)));
    }
}

/* Softmax attention of one query row over a list of key positions.
 * logit_s = sm_scale * sum_d q[d] * K_s[d] (K_s from the row's format);
 * m = max logit; w_s = exp(logit_s - m); out = sum w_s V_s / sum w_s with
 * V_s = K_s[0..511]; lse = m + ln(sum w_s). Keys with pos < 0 are skipped.
 * Returns 0, or -1 if a position is unmapped. With no keys: out = 0, lse = -inf. */
static int attend_row(int fmt, const double *q, const int64_t *pos, int64_t n, int b,
                      const int32_t *bt, int32_t max_blocks, int32_t num_blocks,
                      const uint8_t *kv, const float *kv_scale, double sm_scale,
                      double *out, double *lse, double *logit) {
    int64_t valid = 0;
    double m = -INFINITY;
    double k[ORA_DQK];
    for (int64_t j = 0; j < n; ++j) {
        if (pos[j] < 0) continue;
        int64_t r = cache_row(bt, max_blocks, num_blocks, b, pos[j]);
        if (r < 0) return -1;
        decode_row(fmt, kv, kv_scale, r, k);
        double dot = 0.0;
        for (int d = 0; d < ORA_DQK; ++d) dot += q[d] * k[d];
        logit[j] = sm_scale * dot;
        if (logit[j] > m) m = logit[j];
        ++valid;
    }
    for (int d = 0; d < ORA_DV; ++d) out[d] = 0.0;
    if (valid == 0) {
        *lse = -INFINITY;
        return 0;
    }
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        if (pos[j] < 0) continue;
        int64_t r = cache_row(bt, max_blocks, num_blocks, b, pos[j]);
        decode_row(fmt, kv, kv_scale, r, k);
        double w = exp(logit[j] - m);
        l += w;
        for (int d = 0; d < ORA_DV; ++d) out[d] += w * k[d];
    }
    for (int d = 0; d < ORA_DV; ++d) out[d] /= l;
    *lse = m + log(l);
    return 0;
}

/* Dense causal MLA prefill for n_sel selected new tokens.
 * q: fp64 [n_sel, H, 576] (the selected tokens' query rows); tokens: global
 * new-token indices into cu_seqlens_q. out: [n_sel, H, 512]; lse: [n_sel, H].
 * Returns 0, or a negative count of failed rows. */
int ora_mla_dense_fmt(int fmt, int32_t batch, const int32_t *cu_seqlens_q, const int32_t *prefix_lens,
                      const int32_t *block_table, int32_t max_blocks, int32_t num_blocks,
                      const double *q, const int64_t *tokens, int64_t n_sel, int32_t H,
                      const uint8_t *kv, const float *kv_scale, double sm_scale,
                      double *out, double *lse) {
    ora_init();
    int64_t fails = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : fails)
    for (int64_t rh = 0; rh < n_sel * H; ++rh) {
        int64_t sel = rh / H, h = rh % H, i;
        int b = locate(batch, cu_seqlens_q, tokens[sel], &i);
        if (b < 0) {
            ++fails;
            continue;
        }
        int64_t p = (int64_t)prefix_lens[b] + i;      /* absolute position of the query */
        int64_t n = p + 1;                            /* keys 0..p */
        int64_t *pos = (int64_t *)malloc((size_t)n * sizeof(int64_t));
        double *logit = (double *)malloc((size_t)n * sizeof(double));
        for (int64_t s = 0; s < n; ++s) pos[s] = s;
        if (attend_row(fmt, q + rh * ORA_DQK, pos, n, b, block_table, max_blocks, num_blocks, kv, kv_scale,
                       sm_scale, out + rh * ORA_DV, lse + rh, logit) != 0)
            ++fails;
        free(pos);
        free(logit);
    }
    return fails ? (int)-fails : 0;
}

/* Sparse MLA: as dense, but query token sel attends only to the positions
 * idx[sel*topk .. +topk] (entries < 0 are padding). The causal limit is not
 * re-applied: the index list is the whole key set. */
int ora_mla_sparse_fmt(int fmt, int32_t batch, const int32_t *cu_seqlens_q, const int32_t *prefix_lens,
                       const int32_t *block_table, int32_t max_blocks, int32_t num_blocks,
                       const double *q, const int64_t *tokens, int64_t n_sel, int32_t H,
                       const uint8_t *kv, const float *kv_scale, double sm_scale,
                       const int32_t *idx, int32_t topk, double *out, double *lse) {
    ora_init();
    (void)prefix_lens;
    int64_t fails = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : fails)
    for (int64_t rh = 0; rh < n_sel * H; ++rh) {
        int64_t sel = rh / H, i;
        int b = locate(batch, cu_seqlens_q, tokens[sel], &i);
        if (b < 0) {
            ++fails;
            continue;
        }
        int64_t *pos = (int64_t *)malloc((size_t)topk * sizeof(int64_t));
        double *logit = (double *)malloc((size_t)topk * sizeof(double));
        for (int64_t j = 0; j < topk; ++j) pos[j] = idx[sel * topk + j];
        if (attend_row(fmt, q + rh * ORA_DQK, pos, topk, b, block_table, max_blocks, num_blocks, kv, kv_scale,
                       sm_scale, out + rh * ORA_DV, lse + rh, logit) != 0)
            ++fails;
        free(pos);
        free(logit);
    }
    return fails ? (int)-fails : 0;
}

/* The 580-byte-row entry points (codes + per-token scale). */
int ora_mla_dense(int32_t batch, const int32_t *cu_seqlens_q, const int32_t *prefix_lens,
                  const int32_t *block_table, int32_t max_blocks, int32_t num_blocks,
                  const double *q, const int64_t *tokens, int64_t n_sel, int32_t H,
                  const uint8_t *kv, const float *kv_scale, double sm_scale,
                  double *out, double *lse) {
    return ora_mla_dense_fmt(ORA_FMT_580, batch, cu_seqlens_q, prefix_lens, block_table, max_blocks, num_blocks, q,
                             tokens, n_sel, H, kv, kv_scale, sm_scale, out, lse);
}
int ora_mla_sparse(int32_t batch, const int32_t *cu_seqlens_q, const int32_t *prefix_lens,
                   const int32_t *block_table, int32_t max_blocks, int32_t num_blocks,
                   const double *q, const int64_t *tokens, int64_t n_sel, int32_t H,
                   const uint8_t *kv, const float *kv_scale, double sm_scale,
                   const int32_t *idx, int32_t topk, double *out, double *lse) {
    return ora_mla_sparse_fmt(ORA_FMT_580, batch, cu_seqlens_q, prefix_lens, block_table, max_blocks, num_blocks, q,
                              tokens, n_sel, H, kv, kv_scale, sm_scale, idx, topk, out, lse);
}

typedef struct {
    double score;
    int64_t pos;
} ora_cand;

/* (score descending, position ascending) */
static int cand_cmp(const void *a, const void *b) {
    const ora_cand *x = (const ora_cand *)a, *y = (const ora_cand *)b;
    if (x->score > y->score) return -1;
    if (x->score < y->score) return 1;
    return (x->pos > y->pos) - (x->pos < y->pos);
}

static int cmp_i32(const void *a, const void *b) {
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

/* Indexer + top-k for n_sel selected new tokens.
 * qi: e4m3 [n_sel, 64, 128]; w: f32, row sel at w + sel*w_stride (64 values;
 * stride 0 shares one row); ki: e4m3 [num_blocks, 256, 128]; ki_scale: f32
 * [num_blocks, 256]. idx_out: [n_sel, topk] selected positions in ascending
 * order, -1 padded. scores_out (optional, may be NULL): [n_sel, ctx_cap],
 * score of position s at [sel*ctx_cap + s] for s <= p (others untouched). */
int ora_indexer_topk(int32_t batch, const int32_t *cu_seqlens_q, const int32_t *prefix_lens,
                     const int32_t *block_table, int32_t max_blocks, int32_t num_blocks,
                     const uint8_t *qi, const float *w, int64_t w_stride,
                     const int64_t *tokens, int64_t n_sel,
                     const uint8_t *ki, const float *ki_scale, int32_t topk,
                     int32_t *idx_out, double *scores_out, int64_t ctx_cap) {
    ora_init();
    int64_t fails = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : fails)
    for (int64_t sel = 0; sel < n_sel; ++sel) {
        int64_t i;
        int b = locate(batch, cu_seqlens_q, tokens[sel], &i);
        int32_t *dst = idx_out + sel * topk;
        for (int32_t j = 0; j < topk; ++j) dst[j] = -1;
        if (b < 0) {
            ++fails;
            continue;
        }
        int64_t p = (int64_t)prefix_lens[b] + i;
        int64_t n = p + 1;
        ora_cand *c = (ora_cand *)malloc((size_t)n * sizeof(ora_cand));
        const uint8_t *qrow = qi + sel * 64 * ORA_DIDX;
        const float *wrow = w + sel * w_stride;
        int bad = 0;
        for (int64_t s = 0; s < n; ++s) {
            int64_t r = cache_row(block_table, max_blocks, num_blocks, b, s);
            if (r < 0) {
                bad = 1;
                break;
            }
            const uint8_t *k = ki + r * ORA_DIDX;
            double e = 0.0;
            for (int h = 0; h < 64; ++h) {
                double dot = 0.0;
                for (int d = 0; d < ORA_DIDX; ++d)
                    dot += e4m3_table[qrow[h * ORA_DIDX + d]] * e4m3_table[k[d]];
                e += (double)wrow[h] * (dot > 0.0 ? dot : 0.0);
            }
            c[s].score = (double)ki_scale[r] * e;
            c[s].pos = s;
            if (scores_out && s < ctx_cap) scores_out[sel * ctx_cap + s] = c[s].score;
        }
        if (bad) {
            ++fails;
            free(c);
            continue;
        }
        qsort(c, (size_t)n, sizeof(ora_cand), cand_cmp);
        int64_t keep = n < topk ? n : topk;
        for (int64_t j = 0; j < keep; ++j) dst[j] = (int32_t)c[j].pos;
        qsort(dst, (size_t)keep, sizeof(int32_t), cmp_i32);
        free(c);
    }
    return fails ? (int)-fails : 0;
}

/* ------------------------------------------------------------------------
 * Cache write of the new tokens (the step before attention).
 *
 * Sources: "More throughput from fewer GPUs", section System architecture
 * (the KV cache is FP8, one latent row per token) and section KV hand-off and
 * caching (256-token chunks); GLM-5.3 Teil 2, footnote 3 (indexer keys: 128
 * FP8 values plus a 4-byte scale). The pages name the format but not the
 * quantiser. Readings: one fp32 scale per token and row, equal to the row's
 * absolute maximum divided by 448 (the largest e4m3 value), 1 for an all-zero
 * row, and never below 2^-126 (the smallest normal binary32 value, so that its
 * reciprocal is finite); each element is multiplied by the reciprocal of the
 * scale and the code is the e4m3 value nearest to that product, ties to the
 * even code, magnitudes above 448 clamped to 448. The division, reciprocal
 * and product are IEEE binary32 operations (the precision the quantised code
 * is decided in); the rounding to e4m3 is then exact.
 * ------------------------------------------------------------------------ */

/* The e4m3 code nearest to v: by definition, the finite code whose value is
 * closest to |v| (codes 0..126 hold increasing magnitudes 0..448; 127 is
 * NaN), the even code on a tie, 448 above the range; the sign bit is v's. */
uint8_t ora_e4m3_nearest(float v) {
    ora_init();
    double a = fabs((double)v);
    unsigned lo = 0, hi = 126;
    if (a >= e4m3_table[126]) return (uint8_t)((signbit(v) ? 0x80u : 0u) | 126u);
    /* largest code lo with table[lo] <= a (table[0] = 0 <= a < table[126]) */
    while (hi - lo > 1) {
        unsigned mid = (lo + hi) / 2;
        if (e4m3_table[mid] <= a) lo = mid; else hi = mid;
    }
    double dlo = a - e4m3_table[lo], dhi = e4m3_table[lo + 1] - a;
    unsigned c = dlo < dhi ? lo : dhi < dlo ? lo + 1 : ((lo & 1u) ? lo + 1 : lo);
    return (uint8_t)((signbit(v) ? 0x80u : 0u) | c);
}

/* One row of n bf16 values -> n e4m3 codes and its scale (see above). */
void ora_quantize_row(const uint16_t *x, int64_t n, uint8_t *codes, float *scale_out) {
    double amax = 0.0;
    for (int64_t d = 0; d < n; ++d) {
        double a = fabs(ora_bf16(x[d]));
        if (a > amax) amax = a;
    }
    /* amax is a bf16 value, so (float)amax is exact */
    float scale = amax > 0.0 ? (float)amax / 448.0f : 1.0f;
    if (scale < FLT_MIN) scale = FLT_MIN;
    float inv = 1.0f / scale;
    for (int64_t d = 0; d < n; ++d) {
        float v = (float)ora_bf16(x[d]) * inv;
        codes[d] = ora_e4m3_nearest(v);
    }
    *scale_out = scale;
}

/* New token t (global index into the batch's new tokens) of sequence b sits
 * at position prefix_lens[b] + (t - cu_seqlens_q[b]); its latent row
 * (576 bf16) and indexer key (128 bf16, optional) are quantised and stored at
 * that position's page and slot. Returns 0, or -(number of tokens whose
 * position has no valid page); those tokens write nothing. */
int ora_kv_append(int32_t batch, const int32_t *cu_seqlens_q, const int32_t *prefix_lens,
                  const int32_t *block_table, int32_t max_blocks, int32_t num_blocks,
                  const uint16_t *latent, const uint16_t *kidx,
                  uint8_t *kv, float *kv_scale, uint8_t *ki, float *ki_scale) {
    int64_t n_tok = cu_seqlens_q[batch];
    int64_t fails = 0;
    for (int64_t t = 0; t < n_tok; ++t) {
        int64_t i;
        int b = locate(batch, cu_seqlens_q, t, &i);
        int64_t r = b < 0 ? -1 : cache_row(block_table, max_blocks, num_blocks, b, prefix_lens[b] + i);
        if (r < 0) {
            ++fails;
            continue;
        }
        ora_quantize_row(latent + t * ORA_DQK, ORA_DQK, kv + r * ORA_DQK, kv_scale + r);
        if (kidx) ora_quantize_row(kidx + t * ORA_DIDX, ORA_DIDX, ki + r * ORA_DIDX, ki_scale + r);
    }
    return fails ? (int)-fails : 0;
}

/* ------------------------------------------------------------------------
 * Merge of partial attention results over disjoint key sets.
 *
 * Source: GLM-5.3 Teil 2, section "DCP: Sharding auch des KV-Caches": when
 * the cache is split by token across GPUs, each runs attention over its own
 * shard and the partial results are combined through their log-sum-exp.
 * Written out: for parts i with outputs o_i (softmax-weighted means over their
 * keys) and lse_i = ln(sum of exp(logit) over their keys),
 *   lse = ln sum_i exp(lse_i),   out = sum_i exp(lse_i - lse) * o_i,
 * which is attention over the union of the key sets. A part with lse_i = -inf
 * (no keys) contributes nothing; with every part empty, out = 0, lse = -inf.
 * ------------------------------------------------------------------------ */
void ora_merge(int32_t n_parts, const double *outs, const double *lses, int64_t rows, int64_t dv,
               double *out, double *lse) {
    for (int64_t r = 0; r < rows; ++r) {
        double m = -INFINITY;
        for (int i = 0; i < n_parts; ++i)
            if (lses[(int64_t)i * rows + r] > m) m = lses[(int64_t)i * rows + r];
        double *o = out + r * dv;
        for (int64_t d = 0; d < dv; ++d) o[d] = 0.0;
        if (m == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double total = 0.0;
        for (int i = 0; i < n_parts; ++i) total += exp(lses[(int64_t)i * rows + r] - m);
        for (int i = 0; i < n_parts; ++i) {
            double wgt = exp(lses[(int64_t)i * rows + r] - m) / total;
            const double *oi = outs + ((int64_t)i * rows + r) * dv;
            for (int64_t d = 0; d < dv; ++d) o[d] += wgt * oi[d];
        }
        lse[r] = m + log(total);
    }
}

/* Non-absorbed (MHA) dense causal prefill for n_sel selected new tokens.
 *
 * Per head h, with c_s = K_s[0..511] and r_s = K_s[512..575] the latent and RoPE
 * parts of the decoded cache row of position s (580-byte rows):
 *   k_{s,h} = [ W_UK_h c_s ; r_s ]        192 dims
 *   v_{s,h} = W_UV_h c_s                  128 dims
 * where w_ukv is [H][256][512]: rows 0..127 of head h are W_UK_h and rows
 * 128..255 are W_UV_h (k_{s,h}[i] = sum_d W_UK_h[i][d] c_s[d]). Query row
 * q_{t,h} (192 dims: 128 no-RoPE, then 64 RoPE, RoPE already applied) attends
 * causally to s = 0..p:
 *   logit_s = sm_scale * q_{t,h} . k_{s,h}
 *   out[t,h] = sum_s exp(logit_s - m) v_{s,h} / sum_s exp(logit_s - m)   (128 dims)
 *   lse[t,h] = m + ln sum_s exp(logit_s - m),   m = max_s logit_s
 * The up-projection of every key a sequence's selected tokens see is computed
 * first (one plain matrix product per key and head), then the attention.
 * q: fp64 [n_sel][H][192]; w_ukv: fp64 [H][256][512]; out: [n_sel][H][128];
 * lse: [n_sel][H]. Returns 0, or a negative count of failed rows (token out of
 * range or a needed key on an unmapped page). */
int ora_mla_mha(int32_t batch, const int32_t *cu_seqlens_q, const int32_t *prefix_lens,
                const int32_t *block_table, int32_t max_blocks, int32_t num_blocks,
                const double *q, const int64_t *tokens, int64_t n_sel, int32_t H,
                const uint8_t *kv, const float *kv_scale, const double *w_ukv, double sm_scale,
                double *out, double *lse) {
    ora_init();
    int64_t fails = 0;
    int *seq_of = (int *)malloc((size_t)(n_sel > 0 ? n_sel : 1) * sizeof(int));
    int64_t *pos_of = (int64_t *)malloc((size_t)(n_sel > 0 ? n_sel : 1) * sizeof(int64_t));
    for (int64_t sel = 0; sel < n_sel; ++sel) {
        int64_t i;
        seq_of[sel] = locate(batch, cu_seqlens_q, tokens[sel], &i);
        pos_of[sel] = seq_of[sel] >= 0 ? (int64_t)prefix_lens[seq_of[sel]] + i : -1;
        if (seq_of[sel] < 0) ++fails;
    }
    for (int b = 0; b < batch; ++b) {
        int64_t need = -1;                     /* the largest position a selected token of b sees */
        for (int64_t sel = 0; sel < n_sel; ++sel)
            if (seq_of[sel] == b && pos_of[sel] > need) need = pos_of[sel];
        if (need < 0) continue;
        const int64_t n_keys = need + 1;
        double *kh = (double *)malloc((size_t)(n_keys * H * 192) * sizeof(double));
        double *vh = (double *)malloc((size_t)(n_keys * H * 128) * sizeof(double));
        int unmapped = 0;
        /* step 1: the up-projection of keys 0..need, every head */
#pragma omp parallel for schedule(dynamic, 4) reduction(| : unmapped)
        for (int64_t s = 0; s < n_keys; ++s) {
            const int64_t r = cache_row(block_table, max_blocks, num_blocks, b, s);
            if (r < 0) {
                unmapped = 1;
                continue;
            }
            double k[ORA_DQK];
            decode_row(ORA_FMT_580, kv, kv_scale, r, k);
            for (int h = 0; h < H; ++h) {
                const double *wk = w_ukv + (int64_t)h * 256 * ORA_DV;      /* W_UK_h: rows 0..127 */
                const double *wv = wk + 128 * ORA_DV;                      /* W_UV_h: rows 128..255 */
                double *kout = kh + (s * H + h) * 192;
                double *vout = vh + (s * H + h) * 128;
                for (int i = 0; i < 128; ++i) {
                    double acc = 0.0;
                    for (int d = 0; d < ORA_DV; ++d) acc += wk[(int64_t)i * ORA_DV + d] * k[d];
                    kout[i] = acc;
                }
                for (int j = 0; j < 64; ++j) kout[128 + j] = k[ORA_DV + j];
                for (int i = 0; i < 128; ++i) {
                    double acc = 0.0;
                    for (int d = 0; d < ORA_DV; ++d) acc += wv[(int64_t)i * ORA_DV + d] * k[d];
                    vout[i] = acc;
                }
            }
        }
        /* step 2: causal softmax attention of each selected token and head */
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : fails)
        for (int64_t rh = 0; rh < n_sel * H; ++rh) {
            const int64_t sel = rh / H, h = rh % H;
            if (seq_of[sel] != b) continue;
            if (unmapped) {
                ++fails;
                continue;
            }
            const int64_t p = pos_of[sel];
            const double *qr = q + rh * 192;
            double *logit = (double *)malloc((size_t)(p + 1) * sizeof(double));
            double m = -INFINITY;
            for (int64_t s = 0; s <= p; ++s) {
                const double *kr = kh + (s * H + h) * 192;
                double dot = 0.0;
                for (int e = 0; e < 192; ++e) dot += qr[e] * kr[e];
                logit[s] = sm_scale * dot;
                if (logit[s] > m) m = logit[s];
            }
            double *o = out + rh * 128;
            for (int i = 0; i < 128; ++i) o[i] = 0.0;
            double l = 0.0;
            for (int64_t s = 0; s <= p; ++s) {
                const double wgt = exp(logit[s] - m);
                const double *vr = vh + (s * H + h) * 128;
                l += wgt;
                for (int i = 0; i < 128; ++i) o[i] += wgt * vr[i];
            }
            for (int i = 0; i < 128; ++i) o[i] /= l;
            lse[rh] = m + log(l);
            free(logit);
        }
        free(kh);
        free(vh);
    }
    free(seq_of);
    free(pos_of);
    return fails ? (int)-fails : 0;
}
