// Internal declarations shared by the host entry points and the kernels.
// Nothing here is part of the ABI.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "pkv.h"

namespace pkv {

// Supported row widths (the pages' head_dim 256 and indexer keys of 128).
constexpr int kHeadDim = 256;
constexpr int kIdxDim = 128;

// One stream as a kernel sees it.  `layer_base` is the stream's base plus
// the layer's part of page 0 (#1169: "a cache pointer is its layer's part of
// page 0"); every row of that layer is layer_base + page offset + the row's
// place inside the page's layer part.
struct SeqDev {
    const uint16_t *layer_base;
    const int32_t *table;  // nullptr: contiguous (one page of ptok = cap rows)
    int64_t ps;            // elements in a page
    int32_t ptok;          // positions in a page
    int32_t n_pages;       // arena pages (table entries must be below)
    int32_t n_table;       // table entries (1 when contiguous)
    int32_t len;           // valid positions after the new tokens
    int32_t n_new;         // new tokens (queries) of this call
    int32_t tok_off;       // first packed row of this stream's new tokens
    int32_t work_off;      // first CTA (work item) of this stream in a launch
    int32_t nsplit;        // splits of each unit's key range (decode)
    int32_t split_len;     // keys in a split (multiple of the key tile)
    int32_t comb_off;      // first CTA of this stream in the combine launch
    int32_t ncols;         // query columns of one unit: n_new * group (decode)
    int64_t ws_off;        // float offset of this stream's partials in ws
    int32_t tma;           // index of the stream's 2D row map (16-row boxes of 64 dims), or -1
    int16_t tma_k;         // bf16, chunk kernel: its 3D map of 128-row runs over 128 dims, or -1
    int16_t tma_v;         // bf16, chunk kernel: its 3D map of 64-row runs over 256 dims, or -1
    int64_t layer_row;     // row (256 elements) of layer_base from the map's base
    int64_t page_rows;     // rows in a page (page_elems / 256)
};

// A 2D TMA view of a buffer as rows of 256 bf16 (512 B), boxes of 64 x 16
// elements with 128-byte swizzle: one box is 16 consecutive key (or value)
// rows of one 64-element column chunk.  The 3D tile view of the same rows
// adds the four column chunks as the outer dimension (dims {64, rows, 4},
// strides 512 B and 128 B): one box of {64, R, C} lands as C swizzled planes
// of R rows x 128 B, chunk after chunk, the layout R/16 x C 2D boxes give,
// in one copy.
constexpr int kMaxMaps = 16;
struct alignas(64) RowMap {
    unsigned char bytes[128];  // CUtensorMap
};
struct DecodeMaps {
    RowMap map[kMaxMaps];
};
// Index of the map for [base, base + rows*512 B) in `maps` (added if new),
// or -1 when none can be made (no driver entry point, or maps full).
// bytes8: rows of 256 bytes (e4m3 codes, boxes of 128 x 16) instead of 256
// bf16 elements (boxes of 64 x 16); tile: the 3D tile view of bf16 rows,
// boxes of {64, box_rows, box_chunks} (box_rows 64 or 128, box_chunks 2 or 4).
int row_map(DecodeMaps &maps, int &n_maps, const void *base, uint64_t rows, bool bytes8,
            bool tile = false, int box_rows = 16, int box_chunks = 1);

struct Common {
    int32_t n_seqs;
    int32_t n_kv_heads;
    int32_t idx_dim;
    int32_t layer;
    int32_t n_q_heads;
    int32_t group;  // n_q_heads / n_kv_heads
    int32_t kv_fp8; // K/V rows are e4m3 codes + float32 scales (PKV_KV_E4M3)
    uint32_t *status;
    SeqDev seq[PKV_MAX_SEQS];
};

// Row offsets inside one layer's part of a page of `ptok` positions.
__host__ __device__ inline int64_t off_k(int32_t ptok, int32_t head, int32_t row) {
    return (int64_t)head * ptok * kHeadDim + (int64_t)row * kHeadDim;
}
__host__ __device__ inline int64_t off_v(int32_t h_kv, int32_t ptok, int32_t head, int32_t row) {
    return (int64_t)h_kv * ptok * kHeadDim + off_k(ptok, head, row);
}
__host__ __device__ inline int64_t off_ik(int32_t h_kv, int32_t idx_dim, int32_t ptok,
                                          int32_t row) {
    return 2 * (int64_t)h_kv * ptok * kHeadDim + (int64_t)row * idx_dim;
}
__host__ __device__ inline int64_t off_p(int32_t h_kv, int32_t idx_dim, int32_t ptok,
                                         int32_t block_row) {
    return 2 * (int64_t)h_kv * ptok * kHeadDim + (int64_t)ptok * idx_dim +
           (int64_t)block_row * idx_dim;
}
__host__ __device__ inline int64_t layer_elems(int32_t h_kv, int32_t idx_dim, int32_t ptok) {
    return 2 * (int64_t)h_kv * ptok * kHeadDim + (int64_t)ptok * idx_dim +
           (int64_t)(ptok / 4) * idx_dim;
}

// Either K/V format (#1170, commit 5c09685: a row's e4m3 codes and float32
// scale, a layer's block at ptok rows).  The e4m3 block holds K codes
// [H][ptok][256] bytes, V codes, K scales [H][ptok] float32, V scales, then
// the bf16 indexer and pooled rows as in the bf16 format.  Offsets of the
// bf16 rows are in 16-bit units, of codes and scales in bytes.
__host__ __device__ inline int64_t kv_part(bool fp8, int32_t h_kv, int32_t ptok) {
    return fp8 ? (int64_t)h_kv * ptok * kHeadDim + 4 * (int64_t)h_kv * ptok
               : 2 * (int64_t)h_kv * ptok * kHeadDim;
}
__host__ __device__ inline int64_t off_ik_f(bool fp8, int32_t h_kv, int32_t idx_dim, int32_t ptok,
                                            int32_t row) {
    return kv_part(fp8, h_kv, ptok) + (int64_t)row * idx_dim;
}
__host__ __device__ inline int64_t off_p_f(bool fp8, int32_t h_kv, int32_t idx_dim, int32_t ptok,
                                           int32_t block_row) {
    return kv_part(fp8, h_kv, ptok) + (int64_t)ptok * idx_dim + (int64_t)block_row * idx_dim;
}
__host__ __device__ inline int64_t layer_elems_f(bool fp8, int32_t h_kv, int32_t idx_dim,
                                                 int32_t ptok) {
    return kv_part(fp8, h_kv, ptok) + (int64_t)ptok * idx_dim + (int64_t)(ptok / 4) * idx_dim;
}
// byte offsets of an e4m3 code row and of its scale inside a layer block
__host__ __device__ inline int64_t off8_code(bool v, int32_t h_kv, int32_t ptok, int32_t head,
                                             int32_t row) {
    return (v ? (int64_t)h_kv * ptok * kHeadDim : 0) + ((int64_t)head * ptok + row) * kHeadDim;
}
__host__ __device__ inline int64_t off8_scale(bool v, int32_t h_kv, int32_t ptok, int32_t head,
                                              int32_t row) {
    return 2 * (int64_t)h_kv * ptok * kHeadDim + (v ? 4 * (int64_t)h_kv * ptok : 0) +
           4 * ((int64_t)head * ptok + row);
}

// Runs set() on the current device until it succeeds there once: a kernel's
// attributes belong to each device's context, so a process that uses several
// GPUs sets them on each.  Two threads may both run set() the first time
// (it only sets attributes).  Returns set()'s code, or PKV_ECUDA.
template <typename F>
inline int once_per_device(std::atomic<uint64_t> &done, F set) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PKV_ECUDA;
    const uint64_t bit = 1ull << dev;
    if (done.load(std::memory_order_acquire) & bit) return PKV_OK;
    const int rc = set();
    if (rc == PKV_OK) done.fetch_or(bit, std::memory_order_release);
    return rc;
}
inline int cuda_rc(cudaError_t e) { return e == cudaSuccess ? PKV_OK : PKV_ECUDA; }

// Host helpers (pkv_host.cu).
int validate_layout(const pkv_layout *layout);
inline bool fp8_of(const pkv_layout *L) { return L->kv_format == PKV_KV_E4M3; }
// page sizes are whole blocks of 4 positions (#1169 What this changes)
inline bool page_pos_ok(int32_t page_pos) { return page_pos > 0 && page_pos % 4 == 0; }
int fill_common(const pkv_layout *layout, const pkv_seq *seqs, int32_t n_seqs, int32_t layer,
                int32_t n_q_heads, int32_t *dev_status, Common *c);
int sm_count(int *out);
int launch_status(cudaError_t e);

// Kernel launchers (one per kernel file); all return PKV_OK or PKV_ECUDA.
int launch_store(const Common &c, int32_t total_tokens, const uint16_t *k_new,
                 const uint16_t *v_new, const uint16_t *ik_new, cudaStream_t stream);
// e4m3 format: quantize the new K and V rows, copy the indexer rows
int launch_store8(const Common &c, int32_t total_tokens, const uint16_t *k_new,
                  const uint16_t *v_new, const uint16_t *ik_new, cudaStream_t stream);
// e4m3 format: codes (PKV_K, PKV_V: 256 bytes a head and row) or scales
// (PKV_KS, PKV_VS: a float32 a head and row) of positions 0 .. len-1
int launch_gather8(const Common &c, int32_t kind, int64_t total_rows, void *out,
                   cudaStream_t stream);
int launch_gather(const Common &c, int32_t kind, int64_t total_rows, uint16_t *out,
                  cudaStream_t stream);
int launch_pool(const Common &c, int32_t total_blocks, cudaStream_t stream);

struct DecodePlan {
    int32_t total_items;   // CTAs of the partial kernel
    int32_t total_comb;    // CTAs of the combine kernel
    size_t ws_bytes;       // counters + partials
};
int plan_decode(Common &c, bool sparse, int32_t k, int nsm, DecodePlan *plan);
// Give each eligible dense stream its row map (page size a multiple of 16,
// rows of 256 elements aligned to the buffer base), and with `tiles` (a
// chunk-kernel call) its tile maps: 64-row runs of V where pages hold a
// multiple of 64 positions, 128-row runs of K where they hold a multiple of
// 128.
void plan_maps(Common &c, const pkv_layout *layout, const pkv_seq *seqs, DecodeMaps &maps,
               bool tiles);
int launch_decode(const Common &c, const DecodePlan &plan, const DecodeMaps &maps, bool sparse,
                  const uint16_t *q, const int32_t *ids, int32_t k, uint16_t *out, float *ws,
                  const uint16_t *k_new, const uint16_t *v_new, const uint16_t *ik_new,
                  cudaStream_t stream);
// Chunked prefill (pkv_prefill.cu): plan and launch; split partials use the
// decode layout and are merged by the decode combine kernel.
int plan_prefill(Common &c, int nsm, DecodePlan *plan);
// With k_new (a decode call's new rows, [token][KV head][256], and ik_new
// [token][Di] or null), the kernel reads the new positions' K and V from there
// and stores them (and the indexer-key rows) into their pages.
int launch_prefill(const Common &c, const DecodePlan &plan, const DecodeMaps &maps,
                   const uint16_t *q, uint16_t *out, float *ws, const uint16_t *k_new,
                   const uint16_t *v_new, const uint16_t *ik_new, cudaStream_t stream);
// CTAs the combine gives one (unit, query column) of a stream with ns splits:
// two (each half the dims, the splits in two groups) past 32 splits, where
// one thread would need a second round of loads; one otherwise.  It depends
// only on the stream's own split count.
__host__ __device__ inline int comb_ctas(int ns) { return ns > 32 ? 2 : 1; }
int launch_combine(const Common &c, const DecodePlan &plan, const uint16_t *q, uint16_t *out,
                   float *ws, cudaStream_t stream);
// Decode over e4m3 K/V (pkv_decode8.cu): the same plan and partial layout as
// the bf16 decode, merged by the same combine kernel; with k_new, the new
// rows are quantized and stored by the same call.
int launch_decode8(const Common &c, const DecodePlan &plan, const DecodeMaps &maps,
                   const uint16_t *q, uint16_t *out, float *ws, const uint16_t *k_new,
                   const uint16_t *v_new, const uint16_t *ik_new, cudaStream_t stream);

// Fixed scratch of pkv_decode_static (pkv_decode.cu): its size, and its
// device address on the current device (looked up on the first call there).
constexpr size_t kStaticScratchBytes = 4u << 20;
int static_scratch(void **out);
int launch_scores(const Common &c, float *scores, int32_t ld, const uint16_t *qi,
                  int32_t max_nb, cudaStream_t stream);
int launch_topk(const Common &c, const float *scores, int32_t ld, int32_t k, int32_t *ids,
                cudaStream_t stream);

}  // namespace pkv
