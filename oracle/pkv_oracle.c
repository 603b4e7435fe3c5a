/*
 * Paged KV-cache oracle (TEST INFRASTRUCTURE ONLY; see pkv_oracle.h).
 *
 * Plain C, one thread, no blocking, no fusion.  Attention is evaluated in
 * float64 from exactly widened bf16 inputs.  The two steps whose results
 * decide integers or bytes downstream (block pooling and block scores) are
 * evaluated in float32 in one fixed, stated order, because the pages pin
 * "no sum changes order" and a top-k decision must be taken in the same
 * precision on both sides.
 *
 * Build with -ffp-contract=off: no multiply-add may be fused unless the code
 * says fmaf().
 */
#include "pkv_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------
 * Page layout and row translation.
 *
 * #1169 "fn-paged-kv", What this changes: a page of n positions holds, for
 * each attention layer, the keys, values and indexer keys of its n positions
 * and the pooled rows of their n/4 blocks; a cache pointer is its layer's
 * part of page 0.  #1170, commit 3f5b87d: inside a page the keys and values
 * are [layer][key,value][head][ptok][row]; with no table the old expression
 * holds, "cap rows a head".  Reading taken: the indexer keys follow the
 * values as [ptok][idx_dim] and the pooled rows follow as [ptok/4][idx_dim];
 * the contiguous buffer is the same layout with a single page of ptok = cap.
 * ---------------------------------------------------------------------- */

/* Bytes of one layer's block of a page of ptok positions, either format.
 * e4m3 (#1170, commit 5c09685: a row's codes and fp32 scale, a layer's block
 * at ptok rows).  Reading taken for the order inside the block: K codes
 * [H][ptok][D], V codes [H][ptok][D], K scales [H][ptok], V scales [H][ptok],
 * then the indexer and pooled rows in bf16 as in the bf16 format. */
static int64_t layer_bytes(const orc_shape *s, int32_t ptok)
{
    int64_t h = s->n_kv_heads, d = s->head_dim;
    int64_t ik = 2 * (int64_t)ptok * s->idx_dim;
    int64_t pooled = 2 * (int64_t)(ptok / 4) * s->idx_dim;
    if (s->kv_format == ORC_E4M3)
        return 2 * h * ptok * d + 2 * 4 * h * ptok + ik + pooled;
    return 2 * 2 * h * ptok * d + ik + pooled;
}

int64_t orc_layer_elems(const orc_shape *s, int32_t ptok)
{
    return layer_bytes(s, ptok) / 2; /* 16-bit elements; every block is even */
}

int64_t orc_page_elems(const orc_shape *s, int32_t ptok)
{
    return (int64_t)s->n_layers * orc_layer_elems(s, ptok);
}

int32_t orc_row_elems(const orc_shape *s, int32_t kind)
{
    return (kind == ORC_K || kind == ORC_V) ? s->head_dim : s->idx_dim;
}

/* Offset of a row inside its layer's part of one page. */
static int64_t in_page(const orc_shape *s, int32_t ptok, int32_t kind, int32_t head,
                       int32_t row)
{
    int64_t d = s->head_dim;
    int64_t heads_block = (int64_t)s->n_kv_heads * ptok * d; /* all heads of K (or V) */
    switch (kind) {
    case ORC_K:
        return (int64_t)head * ptok * d + (int64_t)row * d;
    case ORC_V:
        return heads_block + (int64_t)head * ptok * d + (int64_t)row * d;
    case ORC_IK:
        return 2 * heads_block + (int64_t)row * s->idx_dim;
    default: /* ORC_P: row is the block index inside the page */
        return 2 * heads_block + (int64_t)ptok * s->idx_dim + (int64_t)row * s->idx_dim;
    }
}

/*
 * Element offset, from c->base, of the row (layer, kind, head, pos); for
 * ORC_P, pos is a block index (positions 4*pos .. 4*pos+3).  Returns -1 for
 * anything outside the cache.
 */
int64_t orc_row(const orc_shape *s, const orc_cache *c, int32_t layer, int32_t kind,
                int32_t head, int32_t pos)
{
    if (layer < 0 || layer >= s->n_layers || pos < 0 || c->ptok <= 0)
        return -1;
    if (kind < ORC_K || kind > ORC_P)
        return -1;
    if ((kind == ORC_K || kind == ORC_V) && (head < 0 || head >= s->n_kv_heads))
        return -1;
    if ((kind == ORC_IK || kind == ORC_P) && s->idx_dim == 0)
        return -1;
    if (s->kv_format == ORC_E4M3) {
        /* only the indexer and pooled rows of an e4m3 cache are bf16 elements */
        if (kind != ORC_IK && kind != ORC_P)
            return -1;
        int64_t b = orc_row8(s, c, layer, kind, head, pos);
        return b < 0 ? -1 : b / 2;
    }
    int32_t position = (kind == ORC_P) ? 4 * pos : pos; /* first position of the block */
    int64_t layer_part = (int64_t)layer * orc_layer_elems(s, c->ptok);
    if (c->table == NULL) {
        /* no table: the stream's own buffer, cap = ptok rows a head */
        if (position >= c->ptok)
            return -1;
        return layer_part + in_page(s, c->ptok, kind, head, pos);
    }
    int32_t page = position / c->ptok;
    if (page >= c->n_table)
        return -1;
    int32_t id = c->table[page];
    if (id < 0 || id >= c->n_pages)
        return -1;
    int32_t row = (kind == ORC_P) ? (position % c->ptok) / 4 : position % c->ptok;
    return (int64_t)id * c->ps + layer_part + in_page(s, c->ptok, kind, head, row);
}

/* Byte offset of a row inside its layer's block of an e4m3-format page. */
static int64_t in_page8(const orc_shape *s, int32_t ptok, int32_t kind, int32_t head,
                        int32_t row)
{
    int64_t d = s->head_dim, h = s->n_kv_heads;
    int64_t codes = h * ptok * d;   /* bytes of one kind's codes, all heads */
    int64_t scales = 4 * h * ptok;  /* bytes of one kind's scales */
    switch (kind) {
    case ORC_K:
        return (int64_t)head * ptok * d + (int64_t)row * d;
    case ORC_V:
        return codes + (int64_t)head * ptok * d + (int64_t)row * d;
    case ORC_KS:
        return 2 * codes + 4 * ((int64_t)head * ptok + row);
    case ORC_VS:
        return 2 * codes + scales + 4 * ((int64_t)head * ptok + row);
    case ORC_IK:
        return 2 * codes + 2 * scales + 2 * (int64_t)row * s->idx_dim;
    default: /* ORC_P: row is the block index inside the page */
        return 2 * codes + 2 * scales + 2 * (int64_t)ptok * s->idx_dim +
               2 * (int64_t)row * s->idx_dim;
    }
}

int64_t orc_row8(const orc_shape *s, const orc_cache *c, int32_t layer, int32_t kind,
                 int32_t head, int32_t pos)
{
    if (s->kv_format != ORC_E4M3 || layer < 0 || layer >= s->n_layers || pos < 0 || c->ptok <= 0)
        return -1;
    if (kind < ORC_K || kind > ORC_VS)
        return -1;
    int kv = kind == ORC_K || kind == ORC_V || kind == ORC_KS || kind == ORC_VS;
    if (kv && (head < 0 || head >= s->n_kv_heads))
        return -1;
    if (!kv && s->idx_dim == 0)
        return -1;
    int32_t position = (kind == ORC_P) ? 4 * pos : pos;
    int64_t layer_part = (int64_t)layer * layer_bytes(s, c->ptok);
    if (c->table == NULL) {
        if (position >= c->ptok)
            return -1;
        return layer_part + in_page8(s, c->ptok, kind, head, pos);
    }
    int32_t page = position / c->ptok;
    if (page >= c->n_table)
        return -1;
    int32_t id = c->table[page];
    if (id < 0 || id >= c->n_pages)
        return -1;
    int32_t row = (kind == ORC_P) ? (position % c->ptok) / 4 : position % c->ptok;
    return (int64_t)id * 2 * c->ps + layer_part + in_page8(s, c->ptok, kind, head, row);
}

/* Rows per position for a kind: K and V have a row per KV head. */
static int32_t heads_of(const orc_shape *s, int32_t kind)
{
    return (kind == ORC_K || kind == ORC_V) ? s->n_kv_heads : 1;
}

/*
 * Copy n positions' rows (token-major: [n][heads][row]) into the cache
 * (the store; bytes move unchanged).  Returns 0, or -1 if a row falls outside.
 */
int orc_put_rows(const orc_shape *s, const orc_cache *c, int32_t layer, int32_t kind,
                 int32_t pos0, int32_t n, const uint16_t *rows)
{
    int32_t nh = heads_of(s, kind), re = orc_row_elems(s, kind);
    for (int32_t i = 0; i < n; i++)
        for (int32_t h = 0; h < nh; h++) {
            int64_t off = orc_row(s, c, layer, kind, h, pos0 + i);
            if (off < 0)
                return -1;
            memcpy(c->base + off, rows + ((int64_t)i * nh + h) * re, (size_t)re * 2);
        }
    return 0;
}

/* The inverse: read n positions' rows out of the cache, token-major. */
int orc_get_rows(const orc_shape *s, const orc_cache *c, int32_t layer, int32_t kind,
                 int32_t pos0, int32_t n, uint16_t *rows)
{
    int32_t nh = heads_of(s, kind), re = orc_row_elems(s, kind);
    for (int32_t i = 0; i < n; i++)
        for (int32_t h = 0; h < nh; h++) {
            int64_t off = orc_row(s, c, layer, kind, h, pos0 + i);
            if (off < 0)
                return -1;
            memcpy(rows + ((int64_t)i * nh + h) * re, c->base + off, (size_t)re * 2);
        }
    return 0;
}

/* ------------------------------------------------------------------------
 * bf16 conversions (IEEE binary32 truncated to its top 16 bits).
 * ---------------------------------------------------------------------- */

double orc_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

static float bf16_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round a float to the nearest bf16, ties to even (NaN -> quiet NaN). */
uint16_t orc_bf16_round(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------------
 * e4m3 codes (#1170, commit 5c09685: a row's e4m3 codes and fp32 scale).
 * The format: sign, 4 exponent bits with bias 7, 3 mantissa bits; exponent
 * 0 is subnormal (m * 2^-9); no infinities; S.1111.111 is NaN, so the
 * largest magnitude is 1.75 * 2^8 = 448.  The pages do not say how a row's
 * scale is chosen.  Reading taken: scale = max|x| / 448 in float32, each
 * code the e4m3 value nearest x / scale (float32 division), ties to the even
 * code, magnitudes from 448 up saturating to 448; an all-zero row has scale
 * 0 and codes 0.
 * ---------------------------------------------------------------------- */

double orc_e4m3_to_double(uint8_t code)
{
    int e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7)
        return NAN;
    double v = e == 0 ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
    return (code & 0x80) ? -v : v;
}

uint8_t orc_e4m3_from_float(float x)
{
    if (isnan(x))
        return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x); /* exact */
    if (a >= 448.0)
        return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: multiples of 2^-9; rint rounds half to even */
        int m = (int)rint(a * 512.0);
        return sign | (uint8_t)m; /* m == 8 is the smallest normal, code 0x08 */
    }
    int ex;
    frexp(a, &ex); /* a = f * 2^ex, f in [0.5, 1) */
    int e = ex - 1; /* a in [2^e, 2^(e+1)) */
    int m = (int)rint((ldexp(a, -e) - 1.0) * 8.0); /* exact arguments */
    if (m == 8) {
        m = 0;
        e += 1;
    }
    if (e + 7 > 15 || (e + 7 == 15 && m == 7))
        return sign | 0x7E;
    return sign | (uint8_t)((e + 7) << 3) | (uint8_t)m;
}

void orc_e4m3_decode_n(const uint8_t *codes, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = orc_e4m3_to_double(codes[i]);
}

void orc_e4m3_encode_n(const float *x, int64_t n, uint8_t *codes)
{
    for (int64_t i = 0; i < n; i++)
        codes[i] = orc_e4m3_from_float(x[i]);
}

void orc_quantize_row(const uint16_t *bf16_row, int32_t n, uint8_t *codes, float *scale)
{
    float amax = 0.0f;
    for (int32_t i = 0; i < n; i++) {
        float v = fabsf(bf16_to_float(bf16_row[i]));
        if (v > amax)
            amax = v;
    }
    float sc = amax / 448.0f;
    for (int32_t i = 0; i < n; i++) {
        float q = sc > 0.0f ? bf16_to_float(bf16_row[i]) / sc : 0.0f;
        codes[i] = orc_e4m3_from_float(q);
    }
    *scale = sc;
}

int orc_put_rows8(const orc_shape *s, const orc_cache *c, int32_t layer, int32_t kind,
                  int32_t pos0, int32_t n, const uint16_t *rows)
{
    if (kind != ORC_K && kind != ORC_V)
        return -1;
    int32_t nh = s->n_kv_heads, d = s->head_dim;
    uint8_t *bytes = (uint8_t *)c->base;
    for (int32_t i = 0; i < n; i++)
        for (int32_t h = 0; h < nh; h++) {
            int64_t off = orc_row8(s, c, layer, kind, h, pos0 + i);
            int64_t soff = orc_row8(s, c, layer, kind == ORC_K ? ORC_KS : ORC_VS, h, pos0 + i);
            if (off < 0 || soff < 0)
                return -1;
            float sc;
            orc_quantize_row(rows + ((int64_t)i * nh + h) * d, d, bytes + off, &sc);
            memcpy(bytes + soff, &sc, 4);
        }
    return 0;
}

int orc_get_rows8(const orc_shape *s, const orc_cache *c, int32_t layer, int32_t kind,
                  int32_t pos0, int32_t n, void *out)
{
    int32_t nh = s->n_kv_heads, d = s->head_dim;
    int scales = kind == ORC_KS || kind == ORC_VS;
    if (!scales && kind != ORC_K && kind != ORC_V)
        return -1;
    size_t len = scales ? 4 : (size_t)d;
    const uint8_t *bytes = (const uint8_t *)c->base;
    for (int32_t i = 0; i < n; i++)
        for (int32_t h = 0; h < nh; h++) {
            int64_t off = orc_row8(s, c, layer, kind, h, pos0 + i);
            if (off < 0)
                return -1;
            memcpy((uint8_t *)out + ((int64_t)i * nh + h) * len, bytes + off, len);
        }
    return 0;
}

/* One K or V row as float64: bf16 widened, or e4m3 code x scale (the
 * dequantization the pages' fp8 reference runs in float64). */
static int load_row(const orc_shape *s, const orc_cache *c, int32_t layer, int32_t kind,
                    int32_t head, int32_t pos, double *out)
{
    int32_t d_n = s->head_dim;
    if (s->kv_format == ORC_E4M3) {
        int64_t off = orc_row8(s, c, layer, kind, head, pos);
        int64_t soff = orc_row8(s, c, layer, kind == ORC_K ? ORC_KS : ORC_VS, head, pos);
        if (off < 0 || soff < 0)
            return -1;
        const uint8_t *bytes = (const uint8_t *)c->base;
        float sc;
        memcpy(&sc, bytes + soff, 4);
        for (int32_t d = 0; d < d_n; d++)
            out[d] = orc_e4m3_to_double(bytes[off + d]) * (double)sc;
        return 0;
    }
    int64_t off = orc_row(s, c, layer, kind, head, pos);
    if (off < 0)
        return -1;
    for (int32_t d = 0; d < d_n; d++)
        out[d] = orc_bf16_to_double(c->base[off + d]);
    return 0;
}

/* ------------------------------------------------------------------------
 * Pooling (#1169, What this changes: the pool kernel reads indexer keys once
 * per block of four and writes the pooled rows of the n/4 blocks of a page).
 * Readings taken: a pooled row is the mean of its block's four indexer keys,
 * as a float32 sum in position order ((k0 + k1) + k2) + k3, times 0.25
 * (exact), rounded to bf16 to nearest-even.
 * ---------------------------------------------------------------------- */

int orc_pool(const orc_shape *s, const orc_cache *c, int32_t layer, int32_t block0,
             int32_t n_blocks)
{
    int32_t di = s->idx_dim;
    for (int32_t b = block0; b < block0 + n_blocks; b++) {
        int64_t dst = orc_row(s, c, layer, ORC_P, 0, b);
        if (dst < 0)
            return -1;
        int64_t src[4];
        for (int32_t i = 0; i < 4; i++) {
            src[i] = orc_row(s, c, layer, ORC_IK, 0, 4 * b + i);
            if (src[i] < 0)
                return -1;
        }
        for (int32_t d = 0; d < di; d++) {
            float sum = bf16_to_float(c->base[src[0] + d]);
            sum = sum + bf16_to_float(c->base[src[1] + d]);
            sum = sum + bf16_to_float(c->base[src[2] + d]);
            sum = sum + bf16_to_float(c->base[src[3] + d]);
            c->base[dst + d] = orc_bf16_round(sum * 0.25f);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------
 * Attention over an explicit key list, float64.
 *
 * The pages fix which rows are read (through pg_at) but not the attention
 * arithmetic.  Readings taken: scale 1/sqrt(head_dim); query head h reads
 * KV head h / (n_q_heads / n_kv_heads); softmax with the maximum subtracted;
 * an empty key list gives a zero row.
 * ---------------------------------------------------------------------- */

static int attend_list(const orc_shape *s, const orc_cache *c, int32_t layer,
                       int32_t kv_head, const uint16_t *q_row, const int32_t *pos,
                       int32_t n_keys, double *out_row)
{
    int32_t d_n = s->head_dim;
    double scale = 1.0 / sqrt((double)d_n);
    for (int32_t d = 0; d < d_n; d++)
        out_row[d] = 0.0;
    if (n_keys == 0)
        return 0;
    double *logit = (double *)malloc(sizeof(double) * (size_t)n_keys);
    if (!logit)
        return -1;
    double qd[1024];
    for (int32_t d = 0; d < d_n; d++)
        qd[d] = orc_bf16_to_double(q_row[d]);
    double mx = -INFINITY;
    double kv[1024];
    for (int32_t j = 0; j < n_keys; j++) {
        if (load_row(s, c, layer, ORC_K, kv_head, pos[j], kv) < 0) {
            free(logit);
            return -1;
        }
        double dot = 0.0;
        for (int32_t d = 0; d < d_n; d++)
            dot += qd[d] * kv[d];
        logit[j] = dot * scale;
        if (logit[j] > mx)
            mx = logit[j];
    }
    double denom = 0.0;
    for (int32_t j = 0; j < n_keys; j++) {
        double w = exp(logit[j] - mx);
        denom += w;
        if (load_row(s, c, layer, ORC_V, kv_head, pos[j], kv) < 0) {
            free(logit);
            return -1;
        }
        for (int32_t d = 0; d < d_n; d++)
            out_row[d] += w * kv[d];
    }
    for (int32_t d = 0; d < d_n; d++)
        out_row[d] /= denom;
    free(logit);
    return 0;
}

/*
 * One (query, head) row of causal attention: the query sits at position
 * `pos` and reads keys 0..pos.
 */
int orc_attend_row(const orc_shape *s, const orc_cache *c, int32_t layer,
                   int32_t n_q_heads, int32_t head, int32_t pos, const uint16_t *q_row,
                   double *out_row)
{
    if (s->head_dim > 1024 || n_q_heads % s->n_kv_heads != 0)
        return -1;
    int32_t group = n_q_heads / s->n_kv_heads;
    int32_t n_keys = pos + 1;
    int32_t *list = (int32_t *)malloc(sizeof(int32_t) * (size_t)n_keys);
    if (!list)
        return -1;
    for (int32_t j = 0; j < n_keys; j++)
        list[j] = j;
    int rc = attend_list(s, c, layer, head / group, q_row, list, n_keys, out_row);
    free(list);
    return rc;
}

/*
 * Causal attention for the last nq positions of a cache holding len
 * positions (decode: nq = 1; a drafted window or a prefill chunk: nq > 1).
 * Query j sits at position len - nq + j and reads keys 0 .. len - nq + j.
 * q: bf16 [nq][n_q_heads][head_dim]; out: float64, same shape.
 */
int orc_attend(const orc_shape *s, const orc_cache *c, int32_t layer, int32_t n_q_heads,
               int32_t len, int32_t nq, const uint16_t *q, double *out)
{
    if (nq > len)
        return -1;
    int64_t row = s->head_dim;
    for (int32_t j = 0; j < nq; j++)
        for (int32_t h = 0; h < n_q_heads; h++) {
            int64_t o = ((int64_t)j * n_q_heads + h) * row;
            int rc = orc_attend_row(s, c, layer, n_q_heads, h, len - nq + j, q + o, out + o);
            if (rc)
                return rc;
        }
    return 0;
}

/* ------------------------------------------------------------------------
 * Block scores (#1169, What this changes and Receipt: fn_qsa_scores reads
 * pooled rows and gives block scores from the indexer queries).  Readings
 * taken: a block's score is the dot product of the indexer query with the
 * block's pooled row; one indexer query per query head, the complete blocks
 * b < len/4 only, no scale, float32 accumulation acc = fmaf(qi[d], P[b][d], acc) for d = 0, 1,
 * ... in that order from acc = 0.
 * scores: float [n_q_heads][nb], nb = len / 4.
 * ---------------------------------------------------------------------- */

int orc_scores(const orc_shape *s, const orc_cache *c, int32_t layer, int32_t n_q_heads,
               int32_t len, const uint16_t *qi, float *scores)
{
    int32_t nb = len / 4, di = s->idx_dim;
    for (int32_t h = 0; h < n_q_heads; h++)
        for (int32_t b = 0; b < nb; b++) {
            int64_t off = orc_row(s, c, layer, ORC_P, 0, b);
            if (off < 0)
                return -1;
            float acc = 0.0f;
            for (int32_t d = 0; d < di; d++)
                acc = fmaf(bf16_to_float(qi[(int64_t)h * di + d]),
                           bf16_to_float(c->base[off + d]), acc);
            scores[(int64_t)h * nb + b] = acc;
        }
    return 0;
}

/* ------------------------------------------------------------------------
 * Top-k block selection.  Readings taken: rank by score, higher first, an
 * exact tie going to the lower block id (+0 and -0 are equal); keep
 * min(k, nb); emit the kept ids in ascending order; pad with -1 to k.
 * scores: [n_rows][ld] (first nb of each row used); ids: [n_rows][k].
 * ---------------------------------------------------------------------- */

static const float *g_row;

static int by_rank(const void *a, const void *b)
{
    int32_t i = *(const int32_t *)a, j = *(const int32_t *)b;
    float si = g_row[i], sj = g_row[j];
    if (si > sj)
        return -1;
    if (si < sj)
        return 1;
    return (i < j) ? -1 : (i > j);
}

static int by_id(const void *a, const void *b)
{
    int32_t i = *(const int32_t *)a, j = *(const int32_t *)b;
    return (i < j) ? -1 : (i > j);
}

int orc_topk(int32_t n_rows, int32_t nb, const float *scores, int32_t ld, int32_t k,
             int32_t *ids)
{
    if (nb < 0 || k < 0 || ld < nb)
        return -1;
    int32_t *order = (int32_t *)malloc(sizeof(int32_t) * (size_t)(nb > 0 ? nb : 1));
    if (!order)
        return -1;
    int32_t keep = k < nb ? k : nb;
    for (int32_t r = 0; r < n_rows; r++) {
        for (int32_t b = 0; b < nb; b++)
            order[b] = b;
        g_row = scores + (int64_t)r * ld;
        qsort(order, (size_t)nb, sizeof(int32_t), by_rank);
        qsort(order, (size_t)keep, sizeof(int32_t), by_id);
        for (int32_t i = 0; i < k; i++)
            ids[(int64_t)r * k + i] = i < keep ? order[i] : -1;
    }
    free(order);
    return 0;
}

/*
 * Block-sparse attention: query head h of one decode query reads only the
 * keys of its selected blocks, ascending (ids[h][*], -1 entries skipped).
 * q: bf16 [n_q_heads][head_dim]; ids: [n_q_heads][k]; out: float64
 * [n_q_heads][head_dim].  Blocks at or beyond len/4 are refused.
 */
int orc_sparse_attend(const orc_shape *s, const orc_cache *c, int32_t layer,
                      int32_t n_q_heads, int32_t len, const uint16_t *q,
                      const int32_t *ids, int32_t k, double *out)
{
    if (s->head_dim > 1024 || n_q_heads % s->n_kv_heads != 0)
        return -1;
    int32_t group = n_q_heads / s->n_kv_heads;
    int32_t *list = (int32_t *)malloc(sizeof(int32_t) * (size_t)(4 * (k > 0 ? k : 1)));
    if (!list)
        return -1;
    for (int32_t h = 0; h < n_q_heads; h++) {
        int32_t n = 0;
        for (int32_t i = 0; i < k; i++) {
            int32_t b = ids[(int64_t)h * k + i];
            if (b < 0)
                continue;
            if (b >= len / 4) {
                free(list);
                return -1;
            }
            for (int32_t r = 0; r < 4; r++)
                list[n++] = 4 * b + r;
        }
        int rc = attend_list(s, c, layer, h / group, q + (int64_t)h * s->head_dim, list, n,
                             out + (int64_t)h * s->head_dim);
        if (rc) {
            free(list);
            return rc;
        }
    }
    free(list);
    return 0;
}
