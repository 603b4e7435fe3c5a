/*
 * Paged KV-cache oracle: a plain, slow, single-threaded CPU statement of what
 * the paged attention path computes.  TEST INFRASTRUCTURE ONLY: it may be
 * loaded by the tests, by the smoke check and by the benchmark's CPU-baseline
 * leg, and by nothing else.  It shares no code, header or constant with the
 * CUDA library; both read the same seeded inputs and nothing more.
 *
 * Sources (TensorFold pull requests, as published):
 *   #1169 "fn-paged-kv", What this changes: the Pg argument (an int page
 *       table, the elements in a page, the positions in a page); pg_at() with
 *       no table is the old expression, with a table the start of the page
 *       holding the position plus the row inside it; a page of n positions
 *       holds, per attention layer, the keys, values and indexer keys of its
 *       n positions and the pooled rows of their n/4 blocks; a cache pointer
 *       is its layer's part of page 0; only addresses change, no sum changes
 *       order.
 *   #1170 "the streams beside the first take KV pages from the core pool",
 *       commit 3f5b87d: kv_row() with no table is "cap rows a head", with a
 *       table the page holding the position laid out as
 *       [layer][key,value][head][ptok][256].
 *   #1170, commit 5c09685 ("--kv-cache fp8 through the page table too"):
 *       a row's e4m3 codes and fp32 scale found through row8(), cap rows a
 *       head or the row's page laid out as a layer's block at ptok rows; the
 *       reference dequantizes e4m3 x scale in float64.
 * Where the pages leave the arithmetic open (softmax scale, head grouping,
 * pooling order, score order, top-k ties) the reading taken is stated at the
 * function that takes it.
 */
#ifndef PKV_ORACLE_H
#define PKV_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Shape of one model's caches (the same for every stream). */
typedef struct {
    int32_t n_layers;   /* attention layers held in one page              */
    int32_t n_kv_heads; /* key/value heads                                 */
    int32_t head_dim;   /* elements in a key or value row                  */
    int32_t idx_dim;    /* elements in an indexer-key or pooled row (0: none) */
    int32_t kv_format;  /* ORC_BF16: bf16 K/V rows; ORC_E4M3: e4m3 codes + fp32 scale */
} orc_shape;

enum { ORC_BF16 = 0, ORC_E4M3 = 1 };

/* Where one stream's caches live. */
typedef struct {
    uint16_t *base;        /* page 0 of the arena, or the stream's own buffer */
    const int32_t *table;  /* page ids by logical page; NULL = contiguous       */
    int32_t n_table;       /* entries in table                                  */
    int32_t ptok;          /* positions in a page (cap rows when contiguous)    */
    int64_t ps;            /* elements in a page, over all layers               */
    int32_t n_pages;       /* pages in the arena (1 when contiguous)            */
    int32_t pad_;
} orc_cache;

enum { ORC_K = 0, ORC_V = 1, ORC_IK = 2, ORC_P = 3, ORC_KS = 4, ORC_VS = 5 };

int64_t orc_layer_elems(const orc_shape *s, int32_t ptok);
int64_t orc_page_elems(const orc_shape *s, int32_t ptok);
int64_t orc_row(const orc_shape *s, const orc_cache *c, int32_t layer, int32_t kind,
                int32_t head, int32_t pos);
int32_t orc_row_elems(const orc_shape *s, int32_t kind);

int orc_put_rows(const orc_shape *s, const orc_cache *c, int32_t layer, int32_t kind,
                 int32_t pos0, int32_t n, const uint16_t *rows);
int orc_get_rows(const orc_shape *s, const orc_cache *c, int32_t layer, int32_t kind,
                 int32_t pos0, int32_t n, uint16_t *rows);

uint16_t orc_bf16_round(float x);
double orc_bf16_to_double(uint16_t b);

/* e4m3 (4 exponent bits, bias 7, 3 mantissa bits, no infinities, S.1111.111
 * is NaN): exact value of a code, and the code nearest a float (ties to the
 * even code, magnitudes from 448 up saturate to +-448). */
double orc_e4m3_to_double(uint8_t code);
uint8_t orc_e4m3_from_float(float x);
void orc_e4m3_decode_n(const uint8_t *codes, int64_t n, double *out);
void orc_e4m3_encode_n(const float *x, int64_t n, uint8_t *codes);
/* One row's codes and scale: scale = max|x| / 448 and code_i = e4m3(x_i /
 * scale), both in float32 (codes 0 for an all-zero row). */
void orc_quantize_row(const uint16_t *bf16_row, int32_t n, uint8_t *codes, float *scale);

/* Byte offset from c->base of a row of an e4m3-format cache: K and V codes
 * (head_dim bytes), their scales (ORC_KS, ORC_VS: one float), the indexer
 * and pooled rows (bf16).  -1 outside the cache. */
int64_t orc_row8(const orc_shape *s, const orc_cache *c, int32_t layer, int32_t kind,
                 int32_t head, int32_t pos);
/* Quantize and store n positions' K or V rows (bf16 [n][heads][head_dim]). */
int orc_put_rows8(const orc_shape *s, const orc_cache *c, int32_t layer, int32_t kind,
                  int32_t pos0, int32_t n, const uint16_t *rows);
/* Read back codes (ORC_K, ORC_V: [n][heads][head_dim] bytes) or scales
 * (ORC_KS, ORC_VS: [n][heads] floats). */
int orc_get_rows8(const orc_shape *s, const orc_cache *c, int32_t layer, int32_t kind,
                  int32_t pos0, int32_t n, void *out);

int orc_pool(const orc_shape *s, const orc_cache *c, int32_t layer, int32_t block0,
             int32_t n_blocks);

int orc_attend(const orc_shape *s, const orc_cache *c, int32_t layer, int32_t n_q_heads,
               int32_t len, int32_t nq, const uint16_t *q, double *out);
int orc_attend_row(const orc_shape *s, const orc_cache *c, int32_t layer,
                   int32_t n_q_heads, int32_t head, int32_t pos, const uint16_t *q_row,
                   double *out_row);

int orc_scores(const orc_shape *s, const orc_cache *c, int32_t layer, int32_t n_q_heads,
               int32_t len, const uint16_t *qi, float *scores);
int orc_topk(int32_t n_rows, int32_t nb, const float *scores, int32_t ld, int32_t k,
             int32_t *ids);
int orc_sparse_attend(const orc_shape *s, const orc_cache *c, int32_t layer,
                      int32_t n_q_heads, int32_t len, const uint16_t *q,
                      const int32_t *ids, int32_t k, double *out);

#ifdef __cplusplus
}
#endif
#endif
