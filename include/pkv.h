/*
 * pkv.h - paged KV-cache attention on one GB300 (sm_103a), C ABI.
 *
 * What is paged (TensorFold PR #1169 "fn-paged-kv", What this changes; PR
 * #1170 "the streams beside the first take KV pages from the core pool",
 * commit 3f5b87d): each stream's attention caches are n-position pages of
 * one device arena, found through an int page table.  A page of n positions
 * holds, for every attention layer, the keys, values and indexer keys of its
 * n positions and the pooled rows of their n/4 blocks, so n is a multiple of
 * 4.  Row lookup (pg_at): with no table, the old contiguous expression ("cap
 * rows a head"); with a table, the start of the page holding the position
 * plus the row inside that page.  Only addresses change and no sum changes
 * order, so paged results are bit-identical to contiguous ones.
 *
 * Layout of one page, in bf16 elements (page_pos = n positions, D = head_dim,
 * Di = idx_dim, H = n_kv_heads), repeated for layer 0 .. n_layers-1:
 *     K  [H][n][D]   V  [H][n][D]   IK [n][Di]   P [n/4][Di]
 * A contiguous stream buffer is the same layout with one page of n = cap.
 * page_elems = n_layers * (2*H*n*D + n*Di + (n/4)*Di).
 *
 * Conventions for every call:
 *   - Returns PKV_OK (0) or a PKV_E* code; nothing else crosses the ABI (no
 *     C++ exceptions).  Argument checks happen before anything is launched.
 *   - Device pointers are the caller's (allocated by the caller, e.g. with
 *     PyTorch).  The library allocates no device memory.  Work buffers are
 *     sized by the *_ws_size calls and passed in.
 *   - Every launch goes on the caller's `stream`; no call synchronizes.
 *   - Kernels launch with programmatic dependent launch: a call's kernels
 *     may start while the kernel before them on the stream is still running,
 *     and wait for it before touching anything it may write.  Two things are
 *     read before that wait: page tables, and the rows of cached positions
 *     more than 32 below a stream's new tokens (below len - n_new - 32) in
 *     pkv_decode / pkv_decode_static.  So those must not
 *     be written by the kernel immediately before on the stream, unless that
 *     kernel is pkv_store, which makes its rows visible before letting the
 *     next kernel start.  A pkv_decode with k_new writes only its own new
 *     rows (at most 32 a stream), which for a stream decoding in order lie
 *     within the 32 positions below the next call's new tokens, so decode
 *     calls of the same stream and layer may follow each other directly.
 *     Rows, tables and inputs written earlier on the stream, or by a copy or
 *     a kernel launched without programmatic dependent launch, need nothing.
 *   - A multi-stream launch takes one pkv_seq per stream, each with its own
 *     page table (PR #2244 "the grouped draft head's lanes carry their page
 *     table": a grouped launch built without each stream's table read and
 *     wrote other streams' pages).
 *   - Kernels never trap.  A table entry outside [0, n_pages) is reported by
 *     OR-ing PKV_DEV_* bits into *dev_status (a device int32 owned by the
 *     caller; NULL disables reporting) and the access is skipped or replaced
 *     by a read of page 0; results are then unspecified.
 *   - Data types: K, V, IK, P, queries and outputs are bf16; scores float32;
 *     ids int32.  Head dim 256 and indexer dim 128 (or 0) are supported.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define PKV_OK 0
#define PKV_EINVAL 1  /* an argument is malformed or unsupported            */
#define PKV_EAGAIN 2  /* not enough free pages right now; retry after give   */
#define PKV_ECUDA 3   /* a CUDA runtime call failed                          */
#define PKV_EDEVICE 4 /* reserved: a device-side check failed                */

/* ---- bits a kernel ORs into *dev_status ---------------------------------- */
#define PKV_DEV_BAD_PAGE 1u /* a table entry was outside [0, n_pages)     */
#define PKV_DEV_TIMEOUT 2u  /* a pipeline wait ran past its time limit     */
#define PKV_DEV_SMEM 4u     /* a kernel's shared memory was not at the
                               alignment its layout needs; it did nothing  */
#define PKV_DEV_RANGE 8u    /* the tensor-core attention (pkv_prefill, and
                               a decode call's tensor-core route) summed a
                               non-finite value: a V entry beyond fp16's
                               range (|v| > 65,504) in a call whose PV
                               product runs in fp16, or non-finite inputs */

/* kinds of rows (pkv_pg_row, pkv_gather) */
#define PKV_K 0
#define PKV_V 1
#define PKV_IK 2
#define PKV_P 3 /* pooled rows: `pos` counts blocks of 4 positions */
#define PKV_KS 4 /* e4m3 format only: the float32 scale of a K row */
#define PKV_VS 5 /* e4m3 format only: the float32 scale of a V row */

/* K/V formats (pkv_layout.kv_format) */
#define PKV_KV_BF16 0
#define PKV_KV_E4M3 1 /* #1170, commit 5c09685 ("--kv-cache fp8 through the page
                         table too"): each K and V row (one head, one position)
                         is head_dim e4m3 codes and one float32 scale, the row's
                         value being code x scale */

#define PKV_MAX_SEQS 64 /* streams in one launch */

/* Shape of a model's caches; the same for every stream. */
typedef struct pkv_layout {
    int32_t n_layers;   /* attention layer slots in one page (>= 1)           */
    int32_t n_kv_heads; /* key/value heads (>= 1)                              */
    int32_t head_dim;   /* elements in a key or value row (256)                */
    int32_t idx_dim;    /* elements in an indexer-key / pooled row (128, or 0) */
    int32_t kv_format;  /* PKV_KV_BF16 (0) or PKV_KV_E4M3                         */
} pkv_layout;

/*
 * The e4m3 format.  Inside a page, each layer's block holds K codes
 * [H][n][D] bytes, V codes [H][n][D], K scales [H][n] float32, V scales
 * [H][n], then the bf16 indexer [n][Di] and pooled [n/4][Di] rows.  Page and
 * row sizes stay counted in 16-bit elements (page_elems, pkv_layout_page_
 * elems), and pkv_pg_row gives BYTE offsets for every kind of an e4m3
 * layout.  Quantization (the pages do not say how a scale is chosen; this is
 * the plainest reading): scale = max|x| / 448 in float32; code = the e4m3
 * value nearest x / scale (float32 division), ties to even, saturating at
 * +-448; an all-zero row has scale 0 and codes 0.  Calls that take the
 * format: the layout and arena calls, pkv_pg_row, pkv_store (quantizes),
 * pkv_gather (codes, scales, indexer and pooled rows), pkv_pool,
 * pkv_block_scores, pkv_topk, and pkv_decode / pkv_decode_static (with k_new
 * the call quantizes and stores the new rows itself, by the same rule as
 * pkv_store).  pkv_prefill and pkv_sparse_decode answer PKV_EINVAL.
 */

/*
 * Pg: where one stream's caches live (#1169: "an int page table, the
 * elements in a page, and the positions in a page").
 */
typedef struct pkv_pg {
    void *base;            /* device, 16-byte aligned: page 0 of the arena, or the
                              stream's own contiguous buffer when table == NULL      */
    const int32_t *table;  /* device: page id of each logical page; NULL = contiguous */
    int64_t page_elems;    /* elements (bf16) in one page over all layers             */
    int32_t page_pos;      /* positions in one page (cap when table == NULL); %4 == 0 */
    int32_t n_pages;       /* pages in the arena; table entries must be below it;
                              1 when table == NULL                                    */
    int32_t n_table;       /* entries in table (positions must be < n_table*page_pos);
                              1 when table == NULL                                    */
    int32_t reserved;      /* set to 0 */
} pkv_pg;

/*
 * One stream in a launch.  Positions 0 .. len-1 are valid after this call's
 * new tokens; the last n_new of them (len-n_new .. len-1) are this call's new
 * tokens.  New-token rows (k_new, v_new, ik_new, q, out) are packed in stream
 * order: stream s owns rows sum_{t<s} n_new[t] .. + n_new[s]-1.
 */
typedef struct pkv_seq {
    pkv_pg pg;
    int32_t len;
    int32_t n_new;
} pkv_seq;

/* ---- layout ------------------------------------------------------------- */

/* Elements in one page of `page_pos` positions.  EINVAL: bad layout or
 * page_pos <= 0 or not a multiple of 4 (#1170: "n must be a multiple of 4"). */
int pkv_layout_page_elems(const pkv_layout *layout, int32_t page_pos, int64_t *out);

/*
 * pg_at on the host (#1169 What this changes; #1170 commit 3f5b87d kv_row):
 * element offset from pg->base of row (layer, kind, head, pos).  host_table
 * is a host copy of pg->table (ignored when pg->table == NULL).  For PKV_P,
 * pos is a block index.  EINVAL if the row lies outside the cache.
 */
int pkv_pg_row(const pkv_layout *layout, const pkv_pg *pg, const int32_t *host_table,
               int32_t layer, int32_t kind, int32_t head, int32_t pos, int64_t *out);

/* ---- arena: the page pool (#1170 What this changes; commit 1ac2075) ------
 * The arena is caller-owned device memory cut into pages.  Free pages are
 * handed out lowest id first ("the free stack hands out KV pages from the
 * bottom").  Pages given back with a stream become free again only once the
 * work already queued on that stream has finished ("a lane's pages go back
 * once the engine's stream drains"); the arena polls with an event, never
 * blocks.  A request that finds too few free pages gets PKV_EAGAIN and waits
 * (LaneMemory in the pages): it is not an error.  Not thread-safe per arena.
 */
typedef struct pkv_arena pkv_arena;

/* Cut [dev_base, dev_base+bytes) into pages of page_pos positions.  The
 * memory stays the caller's; destroy before freeing it.  EINVAL on a bad
 * layout, a misaligned base or room for no page. */
int pkv_arena_create(const pkv_layout *layout, int32_t page_pos, void *dev_base, size_t bytes,
                     pkv_arena **out);
/* Forget the arena (pending releases are dropped with their events). */
int pkv_arena_destroy(pkv_arena *arena);
/* Pages in the arena, pages free now (after polling pending releases), and
 * elements a page. Any pointer may be NULL. */
int pkv_arena_info(pkv_arena *arena, int32_t *n_pages, int32_t *n_free, int64_t *page_elems);
/* Take n pages (lowest free ids, ascending) into host ids_out[n].
 * EAGAIN if fewer than n are free; nothing is taken then. */
int pkv_pages_take(pkv_arena *arena, int32_t n, int32_t *ids_out);
/* Give pages back.  With `defer` nonzero the pages return once the work
 * queued on `stream` so far has finished (an event is recorded); with defer
 * == 0 they return now and the caller asserts the stream has drained.
 * EINVAL for an id outside the arena or not taken (nothing changes then). */
int pkv_pages_give(pkv_arena *arena, const int32_t *ids, int32_t n, cudaStream_t stream,
                   int32_t defer);
/* Fill a pkv_pg for a stream of this arena; dev_table holds n_table ids. */
int pkv_arena_pg(const pkv_arena *arena, const int32_t *dev_table, int32_t n_table,
                 pkv_pg *out);

/* Event operations used for deferred release; the default is CUDA events.
 * record: 0 and *ev set on success; query: 0 done, 1 pending, <0 failed. */
typedef struct pkv_event_ops {
    int (*record)(void *ctx, cudaStream_t stream, void **ev);
    int (*query)(void *ctx, void *ev);
    void (*destroy)(void *ctx, void *ev);
    void *ctx;
} pkv_event_ops;
/* Replace the event operations (NULL restores CUDA events).  For hosts that
 * track completion themselves, and for tests without a GPU. */
int pkv_arena_set_event_ops(pkv_arena *arena, const pkv_event_ops *ops);

/* ---- runs (#1170, commit 1ac2075: core kv_pool findRun / claimRun /
 * releaseRun, Layout.run_bytes and runPages(); commit 51f8354: mapRun) ------
 * A run is k consecutive pages of the arena leased to one stream for its
 * state that is not attention cache (recurrent states, convolution tails,
 * draft buffers).  Runs come from the top of the arena (the highest ids)
 * while KV pages come from the bottom; a run's pages are never handed out
 * by pkv_pages_take and cannot be given back by pkv_pages_give.  When no k
 * consecutive pages are free (too few, or too fragmented) the request gets
 * PKV_EAGAIN and waits, as one short of pages does.  A run goes back with
 * the same deferral as pages.  Only addresses are handed out: the library
 * never touches the run's bytes. */

/* Pages a run of run_bytes needs (runPages): ceil(run_bytes / page bytes),
 * 0 for 0 bytes. */
int pkv_run_pages(const pkv_arena *arena, uint64_t run_bytes, int32_t *k_out);
/* Claim the run of k >= 1 free pages with the highest first id (the first
 * such window met scanning down from the top) into *first_out.  EAGAIN if
 * there is none; nothing is taken then. */
int pkv_run_take(pkv_arena *arena, int32_t k, int32_t *first_out);
/* Give back the run [first, first + k) exactly as taken, now (defer == 0)
 * or once the work queued on `stream` has finished.  EINVAL if it is not a
 * run held now (nothing changes then). */
int pkv_run_give(pkv_arena *arena, int32_t first, int32_t k, cudaStream_t stream, int32_t defer);
/* Lay n_parts buffers of part_bytes[i] bytes one after another in the run's
 * memory, each starting at a device address that is a multiple of `align`
 * (a power of two, 16 .. 4096), and write their device addresses into
 * ptrs_out[i] (mapRun).  EINVAL (nothing written) when the parts do not fit
 * in the run (a run shorter than its parts is refused), or when
 * [first, first + k) is not a run held now. */
int pkv_run_map(const pkv_arena *arena, int32_t first, int32_t k, const uint64_t *part_bytes,
                int32_t n_parts, uint64_t align, void **ptrs_out);

/* ---- cache store (#1169: fn_attn_prep writes key, value and indexer-key
 * rows through pg_at; #1170 commit 3f5b87d: rope's store through kv_row) ---
 * Copy each stream's n_new new tokens into positions len-n_new .. len-1 of
 * `layer`: k_new, v_new [tokens][H][D] bf16; ik_new [tokens][Di] bf16 (NULL
 * iff idx_dim == 0).  Bytes move unchanged. */
int pkv_store(const pkv_layout *layout, const pkv_seq *seqs, int32_t n_seqs, int32_t layer,
              const void *k_new, const void *v_new, const void *ik_new, int32_t *dev_status,
              cudaStream_t stream);

/* ---- gather (prompt-cache save: #1169 "saves and restores copy page runs
 * in the contiguous layout") -----------------------------------------------
 * Copy rows of `kind` for positions 0 .. len-1 of every stream into `out`,
 * packed in stream order: K/V [sum len][H][D]; IK [sum len][Di]; P
 * [sum len/4][Di].  Restoring is pkv_store with n_new = len. */
int pkv_gather(const pkv_layout *layout, const pkv_seq *seqs, int32_t n_seqs, int32_t layer,
               int32_t kind, void *out, int32_t *dev_status, cudaStream_t stream);

/* ---- pooling (#1169: fn_qsa_pool reads indexer keys once per block of
 * four and writes pooled rows through the table) ------------------------------
 * For every block b completed by this call's new tokens (4b+3 in
 * [len-n_new, len)): P[b] = bf16_rn(((ik[4b]+ik[4b+1])+ik[4b+2])+ik[4b+3]) * 0.25)
 * with float32 sums.  EINVAL if idx_dim == 0. */
int pkv_pool(const pkv_layout *layout, const pkv_seq *seqs, int32_t n_seqs, int32_t layer,
             int32_t *dev_status, cudaStream_t stream);

/* ---- decode attention with split-KV partials and their combine (#1169:
 * fn_attn_chunks(_ahead) reads key and value tiles through key_at, one
 * lookup per key per tile; #1170 commit ce5b78d: tf_q35_attn_partial reads
 * rows through the table, the contiguous path branches once) ---------------
 * Causal attention of each stream's n_new queries: query j (position
 * len-n_new+j) of head h reads keys 0 .. len-n_new+j of KV head
 * h / (n_q_heads/H), softmax(q.k / sqrt(D)) . v.  q, out: [tokens][n_q_heads][D]
 * bf16.  Float32 accumulation.  n_new * (n_q_heads/H) <= 32 per stream.
 * The split of each stream's keys depends only on its length and the GPU's
 * SM count, never on page size, so paged output equals contiguous output
 * bit for bit and a stream's output does not depend on the other streams.
 * Fused store: with k_new and v_new (and ik_new when idx_dim > 0) non-NULL,
 * laid out as for pkv_store, the call also writes the new tokens' rows into
 * the cache (as pkv_store would; quantized by the same rule for an e4m3
 * layout) and reads them from those inputs; with them NULL the new rows must
 * already be in the cache.
 * Ordering: the call may read cached rows more than 32 positions below the
 * new tokens (positions below len - n_new - 32) before the kernel queued
 * just before it on the stream has finished, so that kernel must not write
 * them unless it is pkv_store (see the conventions above); q, k_new, v_new,
 * ik_new, ws, out and the rows above are only touched after it finishes.
 * The split partials go to ws and a second kernel combines them, splits in
 * ascending order.  ws: device, >= pkv_decode_ws_size bytes (0 when no
 * stream needs more than one split), 256-byte aligned, no initialization;
 * one ws per in-flight call.  q and out 16-byte aligned.
 * A bf16 call in which some stream has more than 16 query columns a unit
 * (n_new * n_q_heads / H > 16: a draft window of several tokens) runs on
 * the tensor cores instead, as pkv_prefill does (with k_new, the new
 * positions' keys and values read from the inputs and stored into their
 * pages by the same kernel; nothing read before the wait); the result agrees
 * with the warp-MMA path within the attention tolerance, and paged output
 * still equals contiguous output bit for bit. */
int pkv_decode_ws_size(const pkv_layout *layout, const pkv_seq *seqs, int32_t n_seqs,
                       int32_t n_q_heads, size_t *bytes);
int pkv_decode(const pkv_layout *layout, const pkv_seq *seqs, int32_t n_seqs, int32_t layer,
               int32_t n_q_heads, const void *q, const void *k_new, const void *v_new,
               const void *ik_new, void *out, void *ws, size_t ws_bytes, int32_t *dev_status,
               cudaStream_t stream);

/* ---- chunked prefill on the tensor cores (#1170, maintainer notes on the
 * Qwen slice: contiguous tensor-core attention for flat batches, a page-run
 * path for paged or mixed batches; #1169 maintainer reply: the grouped prompt
 * loop gains the page table) ------------------------------------------------
 * The same causal attention as pkv_decode for streams whose n_new is large
 * (a prompt chunk appended to a cached context): query j of head h (position
 * len-n_new+j) reads keys 0 .. len-n_new+j.  The chunk's rows must be in the
 * cache already (pkv_store, and pkv_pool for its blocks).  QK^T and PV run as
 * tcgen05 MMAs with float32 accumulation in tensor memory (P in two bf16
 * parts).  Whole 16-position page runs are read by TMA when the page size is
 * a multiple of 16; other tiles key by key.  When every stream of the call
 * has more than 32 queries and at least 8 blocks of 128 query columns a KV
 * head (n_new * n_q_heads / H >= 897), a first kernel converts the streams'
 * V rows to fp16 in ws (their bytes are part of pkv_prefill_ws_size) and the
 * PV product runs in fp16 (P rounded to 11 significant bits, one MMA where
 * the two bf16 parts take two): exact for V entries of magnitude 2^-14 to
 * 65,280, rounded to fp16's 2^-24 grid below that, and a V entry beyond
 * 65,504 makes the output non-finite and sets PKV_DEV_RANGE.  q, out:
 * [tokens][n_q_heads][D].  ws: device, >= pkv_prefill_ws_size bytes,
 * 256-byte aligned.  Paged output equals contiguous output bit for bit. */
int pkv_prefill_ws_size(const pkv_layout *layout, const pkv_seq *seqs, int32_t n_seqs,
                        int32_t n_q_heads, size_t *bytes);
int pkv_prefill(const pkv_layout *layout, const pkv_seq *seqs, int32_t n_seqs, int32_t layer,
                int32_t n_q_heads, const void *q, void *out, void *ws, size_t ws_bytes,
                int32_t *dev_status, cudaStream_t stream);

/* ---- decode without a caller-provided workspace ------------------------------
 * No counterpart on the pages: an addition for callers that cannot allocate
 * device memory, such as plugins inside a host framework that owns every
 * device allocation, or serving loops that must not call cudaMalloc (it can
 * synchronize the device and its latency is unbounded).  Same arguments and
 * result as pkv_decode, but the split partials live in a fixed device array
 * inside the library (4 MiB; every GPU that loads the library holds it until
 * the process exits) instead of a workspace.  The call allocates nothing.
 * EINVAL if the batch needs more than 4 MiB of partials (pkv_decode_ws_size
 * tells).  The first call on a device looks the array's address up on that
 * device, so make it before capturing a stream into a graph.  The address is
 * kept for the life of the process: after cudaDeviceReset on a device the
 * kept address is stale, so the call must not be used on that device again
 * in the same process.  All calls share
 * the one array: calls that may run at the same time on the GPU (different
 * streams, or graphs launched concurrently) race on it; issue them in order.
 * Nothing in the array needs to start at zero. */
int pkv_decode_static(const pkv_layout *layout, const pkv_seq *seqs, int32_t n_seqs,
                      int32_t layer, int32_t n_q_heads, const void *q, const void *k_new,
                      const void *v_new, const void *ik_new, void *out, int32_t *dev_status,
                      cudaStream_t stream);

/* ---- block scores (#1169: fn_qsa_scores reads pooled rows) ---------------
 * For each stream's one decode query (n_new == 1), head h and complete block
 * b < len/4: scores[s][h][b] = sum_d qi[h][d] * P[b][d], float32, as the
 * chain acc = fmaf(qi[d], P[b][d], acc) for d = 0 .. Di-1 from acc = 0.
 * qi [tokens][n_q_heads][Di] bf16, 16-byte aligned; scores
 * [n_seqs][n_q_heads][ld] float32, entries b >= len/4 set to -infinity.
 * EINVAL if ld < len/4 or qi is not 16-byte aligned. */
int pkv_block_scores(const pkv_layout *layout, const pkv_seq *seqs, int32_t n_seqs,
                     int32_t layer, int32_t n_q_heads, const void *qi, float *scores,
                     int32_t ld, int32_t *dev_status, cudaStream_t stream);

/* ---- top-k block selection ------------------------------------------------
 * Per (stream, head): the min(k, len/4) blocks with the highest scores, an
 * exact tie going to the lower block id (+0 == -0), written in ascending id
 * order to ids [n_seqs][n_q_heads][k] and padded with -1.  1 <= k <= 256. */
int pkv_topk(const pkv_seq *seqs, int32_t n_seqs, int32_t n_q_heads, const float *scores,
             int32_t ld, int32_t k, int32_t *ids, cudaStream_t stream);

/* ---- block-sparse decode (#1169 Receipt: "sparse attention rows") -------
 * Each stream's one decode query, head h, reads only the keys of its selected
 * blocks ids[s][h][0..k-1] (ascending, -1 = none), softmax(q.k/sqrt(D)) . v
 * over them; no selected block gives a zero row.  Blocks must be < len/4.
 * q, out [tokens][n_q_heads][D] bf16; ws as for pkv_decode. */
int pkv_sparse_ws_size(const pkv_layout *layout, const pkv_seq *seqs, int32_t n_seqs,
                       int32_t n_q_heads, int32_t k, size_t *bytes);
int pkv_sparse_decode(const pkv_layout *layout, const pkv_seq *seqs, int32_t n_seqs,
                      int32_t layer, int32_t n_q_heads, const void *q, const int32_t *ids,
                      int32_t k, void *out, void *ws, size_t ws_bytes, int32_t *dev_status,
                      cudaStream_t stream);

/* ---- diagnostics ------------------------------------------------------------
 * Every pipeline wait in the kernels (a stage or product barrier) gives up
 * after about a second, ORs PKV_DEV_TIMEOUT into *dev_status and returns, so
 * a lost copy ends a launch with an error instead of hanging the GPU.  This
 * call launches one warp whose wait on a barrier nothing arrives on runs out
 * the same way (about a second of GPU time).  dev_status: a device int32,
 * required (EINVAL if NULL). */
int pkv_diag_wait_runs_out(int32_t *dev_status, cudaStream_t stream);
/* The same inside one CTA shaped like the decode's partial CTA (eight warps
 * in four key slices of two, twelve stage slots with full and empty
 * barriers): the lead warp of slice `withheld_slice` (0..3) never arrives for
 * its second tile, both warps of that slice run out of time and raise the
 * CTA's abort flag, the other slices finish, and the whole CTA meets at its
 * barrier and returns with PKV_DEV_TIMEOUT set (about a second).  EINVAL if
 * dev_status is NULL or the slice is out of range. */
int pkv_diag_cta_wait_runs_out(int32_t *dev_status, int32_t withheld_slice, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* PKV_H */
