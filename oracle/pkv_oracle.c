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

int64_t orc_layer_elems(const orc_shape *s, int32_t ptok)
{
    int64_t kv = 2 * (int64_t)s->n_kv_heads * ptok * s->head_dim;
    int64_t ik = (int64_t)ptok * s->idx_dim;
    int64_t pooled = (int64_t)(ptok / 4) * s->idx_dim;
    return kv + ik + pooled;
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
    for (int32_t j = 0; j < n_keys; j++) {
        int64_t off = orc_row(s, c, layer, ORC_K, kv_head, pos[j]);
        if (off < 0) {
            free(logit);
            return -1;
        }
        double dot = 0.0;
        for (int32_t d = 0; d < d_n; d++)
            dot += qd[d] * orc_bf16_to_double(c->base[off + d]);
        logit[j] = dot * scale;
        if (logit[j] > mx)
            mx = logit[j];
    }
    double denom = 0.0;
    for (int32_t j = 0; j < n_keys; j++) {
        double w = exp(logit[j] - mx);
        denom += w;
        int64_t off = orc_row(s, c, layer, ORC_V, kv_head, pos[j]);
        if (off < 0) {
            free(logit);
            return -1;
        }
        for (int32_t d = 0; d < d_n; d++)
            out_row[d] += w * orc_bf16_to_double(c->base[off + d]);
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
