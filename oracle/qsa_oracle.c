/*
 * qsa_oracle.c -- plain CPU oracle for the QSA sparse decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library includes, links
 * or calls this file; only tests/, the smoke check and the benchmark's CPU
 * baseline leg load it.  It is deliberately slow and obvious: one row at a
 * time, a full sort for the top-k, binary64 softmax.
 *
 * Sources (page title + section):
 *   [P1] "vLLM: integrate FP16 packed QSA extension", Summary bullet 3 (the
 *        fused selection: four-head ReLU(Q*K) scores, top-512, expand to
 *        2,048 tokens, three-token tail, [R,2051] int32 padded with -1) and
 *        "Exact contracts" (Selection: shapes/dtypes, tie rule; Attention:
 *        Q/out [R,3,256], exact-packed K/V strides [262144,512,256,1],
 *        V storage_offset 256, indices with holes and duplicates).
 *   [P3] qsa_cache.py: _build_qsa_metadata_kernel (visible blocks =
 *        max(0, min((pos+1)//ratio, seq_len//ratio))),
 *        compressed_qsa_slot_mapping (group g is complete once (pos+1) is a
 *        multiple of the ratio), _logical_to_physical_qsa_slots (physical
 *        block = block_table[req, logical // block_size]; negative = pad).
 *
 * Readings where the pages are silent are listed in the design notes; the
 * ones that shape code here are restated at the functions below.
 */
#include "qsa_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#define TOKEN_TOPK    2048   /* [P1] Exact contracts, Selection */
#define COMPRESS      4      /* [P1] Exact contracts, Selection */
#define TOPK_BLOCKS   (TOKEN_TOPK / COMPRESS)   /* 512 */
#define OUT_WIDTH     (TOKEN_TOPK + COMPRESS - 1) /* 2051 = 2048 + 3-token tail */
#define SEL_HEADS     4      /* Q [R,4,128] */
#define SEL_DIM       128
#define CMP_PAGE_KEYS 128    /* cache [P,128,1,128] */
#define ATT_HEADS     3      /* Q/out [R,3,256] */
#define ATT_DIM       256
#define KV_PAGE_TOK   512    /* stride 262144 = 512 tokens x 512 halves */
#define KV_TOKEN_HALVES 512  /* K = halves 0..255, V = halves 256..511 */

/* IEEE binary16 -> binary64; every fp16 value is exactly representable. */
double qsa_oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int exp = (h >> 10) & 0x1f;
    int man = h & 0x3ff;
    double v;
    if (exp == 0)
        v = ldexp((double)man, -24);              /* subnormal: man * 2^-24 */
    else if (exp == 31)
        v = man ? NAN : INFINITY;
    else
        v = ldexp((double)(man | 0x400), exp - 25); /* 1.man * 2^(exp-15) */
    return sign ? -v : v;
}

static float h2f(uint16_t h) { return (float)qsa_oracle_half_to_double(h); }

/* OCP FP8 E4M3 ("fn" variant): 1 sign, 4 exponent (bias 7), 3 mantissa bits;
 * no infinities, S.1111.111 is NaN; max 448.  Every value is exactly
 * representable in binary16 and binary32.  The optional e4m3 compressed
 * indexer cache of qsa_cache.py (QSAStateBackend's fp8 cache dtypes) stores
 * its keys this way. */
double qsa_oracle_e4m3_to_double(uint8_t v)
{
    int sign = (v >> 7) & 1;
    int exp = (v >> 3) & 0xf;
    int man = v & 0x7;
    double x;
    if (exp == 0xf && man == 0x7)
        x = NAN;
    else if (exp == 0)
        x = ldexp((double)man, -9);                 /* subnormal: man/8 * 2^-6 */
    else
        x = ldexp((double)(man | 0x8), exp - 10);   /* 1.man * 2^(exp-7) */
    return sign ? -x : x;
}

/* floor division for possibly negative numerators, positive divisor */
static int64_t floor_div(int64_t a, int64_t b)
{
    int64_t q = a / b;
    if ((a % b != 0) && (a < 0)) q -= 1;
    return q;
}

/* [P3] _build_qsa_metadata_kernel: max(0, min((pos+1)//4, seq_len//4)). */
int64_t qsa_oracle_visible_blocks(int64_t seq_len, int64_t pos)
{
    int64_t a = floor_div(pos + 1, COMPRESS);
    int64_t b = floor_div(seq_len, COMPRESS);
    int64_t v = a < b ? a : b;
    return v > 0 ? v : 0;
}

/* Tail reading: the not-yet-compressed tokens [4V, min(pos, seq_len-1)].
 * Its length is 0..3; it is 3 exactly when seq_len = 3 (mod 4) and
 * pos = seq_len-1, which is the [P1] "three-token tail" of width 2051. */
int64_t qsa_oracle_tail_end(int64_t seq_len, int64_t pos)
{
    return pos < seq_len - 1 ? pos : seq_len - 1;
}

/*
 * Canonical binary32 score ([P1] "four-head ReLU(Q*K) scores").  The pages
 * fix neither precision nor order; bit-exact top-k needs one, so the score
 * is defined as follows (round-to-nearest-even after every add; each fp16 x
 * fp16 product is exact in binary32, so add-after-multiply and fused
 * multiply-add give the same bits):
 *   for each head h, the 128 dims are cut into four 32-dim slices t=0..3;
 *     E_t = sum over j=0..15 ascending of q[h][32t+2j]   * k[32t+2j]
 *     O_t = sum over j=0..15 ascending of q[h][32t+2j+1] * k[32t+2j+1]
 *           (both sums start at +0)
 *     P_t = E_t + O_t
 *     d_h = (P_0 + P_2) + (P_1 + P_3)
 *   r_h = d_h if d_h > 0 else +0
 *   s   = (r_0 + r_1) + (r_2 + r_3)
 * Every non-positive head contributes +0, so s >= +0 and equal sums compare
 * equal bit for bit.
 */
/* The canonical order over binary32 key values kf[128] (exact decodes). */
static float score_values(const uint16_t* q, const float* kf)
{
    float r[SEL_HEADS];
    for (int h = 0; h < SEL_HEADS; ++h) {
        const uint16_t* qh = q + h * SEL_DIM;
        float P[4];
        for (int t = 0; t < 4; ++t) {
            float E = 0.0f, O = 0.0f;
            for (int j = 0; j < 16; ++j) {
                int de = 32 * t + 2 * j;
                int d_o = de + 1;
                float pe = h2f(qh[de]) * kf[de];    /* exact */
                float po = h2f(qh[d_o]) * kf[d_o];  /* exact */
                E = E + pe;
                O = O + po;
            }
            P[t] = E + O;
        }
        float d = (P[0] + P[2]) + (P[1] + P[3]);
        r[h] = d > 0.0f ? d : 0.0f;
    }
    return (r[0] + r[1]) + (r[2] + r[3]);
}

float qsa_oracle_score(const uint16_t* q, const uint16_t* k)
{
    float kf[SEL_DIM];
    for (int i = 0; i < SEL_DIM; ++i) kf[i] = h2f(k[i]);
    return score_values(q, kf);
}

float qsa_oracle_score_e4m3(const uint16_t* q, const uint8_t* k)
{
    float kf[SEL_DIM];
    for (int i = 0; i < SEL_DIM; ++i) kf[i] = (float)qsa_oracle_e4m3_to_double(k[i]);
    return score_values(q, kf);
}

typedef struct {
    float s;
    int64_t b;
} cand_t;

/* [P1] Exact contracts: descending score, ascending logical index on ties. */
static int cand_cmp(const void* x, const void* y)
{
    const cand_t* a = (const cand_t*)x;
    const cand_t* c = (const cand_t*)y;
    if (a->s > c->s) return -1;
    if (a->s < c->s) return 1;
    if (a->b < c->b) return -1;
    if (a->b > c->b) return 1;
    return 0;
}

/* One row of selection ([P1] Summary bullet 3, Exact contracts/Selection). */
static uint32_t select_row(const uint16_t* q, int key_kind, const void* const* cmp_pages,
                           int64_t num_cmp_pages, const int32_t* cmp_pt,
                           int64_t num_reqs, int64_t max_pages, int64_t pt_stride0,
                           int32_t req, const int32_t* seq_lens, int64_t pos,
                           int32_t* out, int64_t out_width, float* scores_out)
{
    uint32_t err = 0;
    for (int64_t j = 0; j < out_width; ++j) out[j] = -1;   /* padded with -1 */
    if (scores_out)
        for (int j = 0; j < TOPK_BLOCKS; ++j) scores_out[j] = -1.0f;
    if (req < 0 || req >= num_reqs) return QSA_ORACLE_ERR_REQUEST;

    int64_t L = seq_lens[req];
    int64_t V = qsa_oracle_visible_blocks(L, pos);
    int64_t tail_end = qsa_oracle_tail_end(L, pos);

    /* score every visible block reachable through the page table */
    cand_t* c = (cand_t*)malloc(sizeof(cand_t) * (size_t)(V > 0 ? V : 1));
    int64_t n = 0;
    for (int64_t b = 0; b < V; ++b) {
        int64_t col = b / CMP_PAGE_KEYS;
        if (col >= max_pages) { err |= QSA_ORACLE_ERR_CMP_PAGE; continue; }
        int64_t pg = cmp_pt[(int64_t)req * pt_stride0 + col];
        if (pg < 0 || pg >= num_cmp_pages || cmp_pages[pg] == NULL) {
            err |= QSA_ORACLE_ERR_CMP_PAGE;
            continue;
        }
        if (key_kind == QSA_ORACLE_KEY_E4M3)
            c[n].s = qsa_oracle_score_e4m3(
                q, (const uint8_t*)cmp_pages[pg] + (b % CMP_PAGE_KEYS) * SEL_DIM);
        else
            c[n].s = qsa_oracle_score(
                q, (const uint16_t*)cmp_pages[pg] + (b % CMP_PAGE_KEYS) * SEL_DIM);
        c[n].b = b;
        ++n;
    }
    /* exact top-512: the prefix of a full sort under the contract's order */
    qsort(c, (size_t)n, sizeof(cand_t), cand_cmp);
    int64_t keep = n < TOPK_BLOCKS ? n : TOPK_BLOCKS;

    /* expand each kept block to its 4 tokens, then the tail, then -1 */
    int64_t w = 0;
    for (int64_t i = 0; i < keep; ++i) {
        for (int r = 0; r < COMPRESS; ++r) out[w++] = (int32_t)(c[i].b * COMPRESS + r);
        if (scores_out) scores_out[i] = c[i].s;
    }
    for (int64_t t = V * COMPRESS; t <= tail_end; ++t) out[w++] = (int32_t)t;
    free(c);
    return err;
}

static uint32_t select_rows(int64_t R, const uint16_t* q_sel, int key_kind,
                            const void* const* cmp_pages, int64_t num_cmp_pages,
                            const int32_t* cmp_pt, int64_t num_reqs, int64_t max_pages,
                            int64_t pt_stride0, const int32_t* t2r,
                            const int32_t* seq_lens, const int64_t* qpos,
                            int32_t* out, int64_t out_width, float* scores_out)
{
    uint32_t err = 0;
    if (out_width < OUT_WIDTH) return 0xffffffffu;
    for (int64_t r = 0; r < R; ++r)
        err |= select_row(q_sel + r * SEL_HEADS * SEL_DIM, key_kind, cmp_pages, num_cmp_pages,
                          cmp_pt, num_reqs, max_pages, pt_stride0, t2r[r], seq_lens,
                          qpos[r], out + r * out_width, out_width,
                          scores_out ? scores_out + r * TOPK_BLOCKS : NULL);
    return err;
}

uint32_t qsa_oracle_select(int64_t R, const uint16_t* q_sel,
                           const uint16_t* const* cmp_pages, int64_t num_cmp_pages,
                           const int32_t* cmp_pt, int64_t num_reqs, int64_t max_pages,
                           int64_t pt_stride0, const int32_t* t2r,
                           const int32_t* seq_lens, const int64_t* qpos,
                           int32_t* out, int64_t out_width)
{
    return select_rows(R, q_sel, QSA_ORACLE_KEY_F16, (const void* const*)cmp_pages,
                       num_cmp_pages, cmp_pt, num_reqs, max_pages, pt_stride0, t2r, seq_lens,
                       qpos, out, out_width, NULL);
}

uint32_t qsa_oracle_select_keys(int64_t R, const uint16_t* q_sel, int key_kind,
                                const void* const* cmp_pages, int64_t num_cmp_pages,
                                const int32_t* cmp_pt, int64_t num_reqs, int64_t max_pages,
                                int64_t pt_stride0, const int32_t* t2r,
                                const int32_t* seq_lens, const int64_t* qpos,
                                int32_t* out, int64_t out_width)
{
    if (key_kind != QSA_ORACLE_KEY_F16 && key_kind != QSA_ORACLE_KEY_E4M3) return 0xffffffffu;
    return select_rows(R, q_sel, key_kind, cmp_pages, num_cmp_pages, cmp_pt, num_reqs, max_pages,
                       pt_stride0, t2r, seq_lens, qpos, out, out_width, NULL);
}

uint32_t qsa_oracle_select_scored(int64_t R, const uint16_t* q_sel,
                                  const uint16_t* const* cmp_pages, int64_t num_cmp_pages,
                                  const int32_t* cmp_pt, int64_t num_reqs, int64_t max_pages,
                                  int64_t pt_stride0, const int32_t* t2r,
                                  const int32_t* seq_lens, const int64_t* qpos,
                                  int32_t* out, int64_t out_width, float* scores_out)
{
    return select_rows(R, q_sel, QSA_ORACLE_KEY_F16, (const void* const*)cmp_pages,
                       num_cmp_pages, cmp_pt, num_reqs, max_pages, pt_stride0, t2r, seq_lens,
                       qpos, out, out_width, scores_out);
}

/*
 * One row of sparse attention ([P1] Exact contracts/Attention), binary64:
 *   valid entries j: idx_j >= 0 whose K/V page resolves; each occurrence of a
 *   duplicated index is its own softmax term (gather, then dense softmax);
 *   z_j = scale * (q_h . K_j);  out_h = sum_j e^(z_j - m) V_j / sum_j e^(z_j - m)
 *   with m = max_j z_j; no valid entry gives an all-zero output.
 * K/V of logical token i: page kv_pt[req, i // 512], token i % 512; K is the
 * first 256 halves of the token's 512, V the last 256 (V storage_offset 256).
 */
static uint32_t attention_row(const uint16_t* q, const uint16_t* const* kv_pages,
                              int64_t num_kv_pages, const int32_t* kv_pt, int64_t num_reqs,
                              int64_t max_kv_pages, int64_t pt_stride0, int32_t req,
                              const int32_t* idx, int64_t width, double scale, double* out)
{
    uint32_t err = 0;
    for (int i = 0; i < ATT_HEADS * ATT_DIM; ++i) out[i] = 0.0;
    if (req < 0 || req >= num_reqs) return QSA_ORACLE_ERR_REQUEST;

    double qd[ATT_HEADS][ATT_DIM];
    for (int h = 0; h < ATT_HEADS; ++h)
        for (int d = 0; d < ATT_DIM; ++d)
            qd[h][d] = qsa_oracle_half_to_double(q[h * ATT_DIM + d]);

    const uint16_t** tok = (const uint16_t**)malloc(sizeof(uint16_t*) * (size_t)(width > 0 ? width : 1));
    int64_t n = 0;
    for (int64_t j = 0; j < width; ++j) {
        int64_t i = idx[j];
        if (i < 0) continue;                      /* hole */
        int64_t col = i / KV_PAGE_TOK;
        if (col >= max_kv_pages) { err |= QSA_ORACLE_ERR_KV_PAGE; continue; }
        int64_t pg = kv_pt[(int64_t)req * pt_stride0 + col];
        if (pg < 0 || pg >= num_kv_pages || kv_pages[pg] == NULL) {
            err |= QSA_ORACLE_ERR_KV_PAGE;
            continue;
        }
        tok[n++] = kv_pages[pg] + (i % KV_PAGE_TOK) * KV_TOKEN_HALVES;
    }
    if (n == 0) { free(tok); return err; }

    double* z = (double*)malloc(sizeof(double) * (size_t)n);
    for (int h = 0; h < ATT_HEADS; ++h) {
        double m = -INFINITY;
        for (int64_t j = 0; j < n; ++j) {
            double dot = 0.0;
            for (int d = 0; d < ATT_DIM; ++d)
                dot += qd[h][d] * qsa_oracle_half_to_double(tok[j][d]);
            z[j] = dot * scale;
            if (z[j] > m) m = z[j];
        }
        double l = 0.0;
        double acc[ATT_DIM];
        for (int d = 0; d < ATT_DIM; ++d) acc[d] = 0.0;
        for (int64_t j = 0; j < n; ++j) {
            double p = exp(z[j] - m);
            l += p;
            for (int d = 0; d < ATT_DIM; ++d)
                acc[d] += p * qsa_oracle_half_to_double(tok[j][ATT_DIM + d]);
        }
        for (int d = 0; d < ATT_DIM; ++d) out[h * ATT_DIM + d] = acc[d] / l;
    }
    free(z);
    free(tok);
    return err;
}

uint32_t qsa_oracle_attention(int64_t R, const uint16_t* q,
                              const uint16_t* const* kv_pages, int64_t num_kv_pages,
                              const int32_t* kv_pt, int64_t num_reqs, int64_t max_kv_pages,
                              int64_t pt_stride0, const int32_t* t2r,
                              const int32_t* idx, int64_t width, double scale,
                              double* out)
{
    uint32_t err = 0;
    for (int64_t r = 0; r < R; ++r)
        err |= attention_row(q + r * ATT_HEADS * ATT_DIM, kv_pages, num_kv_pages, kv_pt,
                             num_reqs, max_kv_pages, pt_stride0, t2r[r], idx + r * width,
                             width, scale, out + r * ATT_HEADS * ATT_DIM);
    return err;
}
