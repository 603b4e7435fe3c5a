// Cache store, gather and block pooling, for the bf16 and the e4m3 K/V
// formats (the e4m3 store quantizes each new K and V row).  Rows are located
// with pg_at once per row (store, gather) or once per block of four positions
// (pool: a page holds whole blocks because its size is a multiple of 4),
// never per load.  Stores let the next kernel start only once their rows are
// visible: a decode may read cached rows before its grid-dependency wait.
#include "pkv_dev.cuh"

namespace pkv {
namespace {

constexpr int kThreads = 256;
constexpr int kChunk = 8;  // bf16 elements in a 16-byte chunk
constexpr int kBatch = 4;  // 16-byte chunks a lane loads before it stores them

// Offset of the page holding `pos`, or -1 for a table entry outside the
// arena (reported); row is the row inside the page.
__device__ __forceinline__ int64_t page_or_bad(const SeqDev &s, int32_t pos, int32_t *row,
                                               uint32_t *status) {
    if (s.table == nullptr) {
        *row = pos;
        return 0;
    }
    int32_t page = pos / s.ptok;
    *row = pos - page * s.ptok;
    int32_t id = __ldg(s.table + page);
    if (static_cast<uint32_t>(id) >= static_cast<uint32_t>(s.n_pages)) {
        if (status) atomicOr(status, PKV_DEV_BAD_PAGE);
        return -1;
    }
    return (int64_t)id * s.ps;
}

// A warp stores one new token at a time: its 2*H rows of 256 (K then V)
// and, with indexer keys, its row of 128.  The stream, page and row are found
// once per token; lane l copies the token's 16-byte chunks l, l + 32, ...,
// up to kBatch of them loaded before any is stored.
__global__ void __launch_bounds__(kThreads) store_kernel(const __grid_constant__ Common c,
                                                         int32_t total_tokens,
                                                         const uint16_t *__restrict__ k_new,
                                                         const uint16_t *__restrict__ v_new,
                                                         const uint16_t *__restrict__ ik_new) {
    pdl_wait();
    const int H = c.n_kv_heads;
    constexpr int row_chunks = kHeadDim / kChunk;  // 32
    const int kv_chunks = 2 * H * row_chunks;
    const int per_tok = kv_chunks + c.idx_dim / kChunk;
    const int lane = threadIdx.x & 31;
    const int nwarps = gridDim.x * (kThreads / 32);
    for (int tok = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); tok < total_tokens;
         tok += nwarps) {
        const int s = find_seq(c.n_seqs, tok, [&](int t) { return c.seq[t].tok_off; });
        const SeqDev &sd = c.seq[s];
        const int32_t pos = sd.len - sd.n_new + (tok - sd.tok_off);
        int32_t row;
        const int64_t page = page_or_bad(sd, pos, &row, lane == 0 ? c.status : nullptr);
        if (page < 0) continue;
        uint16_t *base = const_cast<uint16_t *>(sd.layer_base) + page;
        for (int r0 = 0; r0 < per_tok; r0 += 32 * kBatch) {
            uint4 val[kBatch];
            int64_t dst[kBatch];
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
                const int r = r0 + 32 * b + lane;
                dst[b] = -1;
                if (r >= per_tok) continue;
                const uint16_t *src;
                if (r < kv_chunks) {
                    const int kh = r / row_chunks, ch = r % row_chunks;  // kh: K heads, then V heads
                    const int kind = kh >= H, head = kh - kind * H;
                    src = (kind ? v_new : k_new) + ((int64_t)tok * H + head) * kHeadDim + ch * kChunk;
                    dst[b] = (kind ? off_v(H, sd.ptok, head, row) : off_k(sd.ptok, head, row)) +
                             ch * kChunk;
                } else {
                    const int ch = r - kv_chunks;
                    src = ik_new + (int64_t)tok * c.idx_dim + ch * kChunk;
                    dst[b] = off_ik(H, c.idx_dim, sd.ptok, row) + ch * kChunk;
                }
                val[b] = __ldg(reinterpret_cast<const uint4 *>(src));
            }
#pragma unroll
            for (int b = 0; b < kBatch; ++b)
                if (dst[b] >= 0) *reinterpret_cast<uint4 *>(base + dst[b]) = val[b];
        }
    }
    pdl_trigger_after_writes();  // the next decode may read these rows early
}

// Gather of one kind into packed rows; work_off holds each stream's first
// output row.  K or V (kKV): a warp per output row (a position's rows of every
// head, 32 chunks of 16 bytes a head), lane l taking chunk l of each head and
// loading up to kBatch heads before it stores them.  Indexer or pooled rows
// (128 dims, 16 chunks): a half-warp per row.  The stream, page and row are
// found once per row; rows behind a bad table entry come out as zeros.
template <bool kKV>
__global__ void __launch_bounds__(kThreads) gather_kernel(const __grid_constant__ Common c,
                                                          int32_t kind, int32_t total_rows,
                                                          uint16_t *__restrict__ out) {
    pdl_wait();
    pdl_trigger();
    constexpr int row_chunks = (kKV ? kHeadDim : kIdxDim) / kChunk;  // 32 or 16
    constexpr int rows_per_warp = 32 / row_chunks;                     // 1 or 2
    const int H = c.n_kv_heads;
    const int lane = threadIdx.x & 31, sub = lane / row_chunks, ch = lane % row_chunks;
    const int nwarps = gridDim.x * (kThreads / 32);
    for (int w = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); w * rows_per_warp < total_rows;
         w += nwarps) {
        const int orow = w * rows_per_warp + sub;
        if (orow >= total_rows) continue;
        const int s = find_seq(c.n_seqs, orow, [&](int t) { return c.seq[t].work_off; });
        const SeqDev &sd = c.seq[s];
        const int32_t idx = orow - sd.work_off;  // position, or block for PKV_P
        const int32_t pos = kind == PKV_P ? 4 * idx : idx;
        int32_t row;
        const int64_t page = page_or_bad(sd, pos, &row, ch == 0 ? c.status : nullptr);
        const uint16_t *lb = sd.layer_base + page;
        if (kKV) {
            uint16_t *dst = out + ((int64_t)orow * H * row_chunks + ch) * kChunk;
            const uint16_t *src = lb + (kind == PKV_V ? off_v(H, sd.ptok, 0, row) : off_k(sd.ptok, 0, row)) +
                                  ch * kChunk;
            const int64_t head_step = (int64_t)sd.ptok * kHeadDim;  // the next head's row
            for (int h0 = 0; h0 < H; h0 += kBatch) {
                uint4 val[kBatch];
#pragma unroll
                for (int b = 0; b < kBatch; ++b)
                    val[b] = page >= 0 && h0 + b < H
                                 ? *reinterpret_cast<const uint4 *>(src + (h0 + b) * head_step)
                                 : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int b = 0; b < kBatch; ++b)
                    if (h0 + b < H)
                        *reinterpret_cast<uint4 *>(dst + (int64_t)(h0 + b) * row_chunks * kChunk) = val[b];
            }
        } else {
            const int64_t off = kind == PKV_IK ? off_ik_f(c.kv_fp8, H, c.idx_dim, sd.ptok, row)
                                               : off_p_f(c.kv_fp8, H, c.idx_dim, sd.ptok, row / 4);
            const uint4 val = page >= 0 ? *reinterpret_cast<const uint4 *>(lb + off + ch * kChunk)
                                        : make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4 *>(out + ((int64_t)orow * row_chunks + ch) * kChunk) = val;
        }
    }
}

// One thread per (block, 8 dims): P[b] = bf16_rn((((k0 + k1) + k2) + k3) * 0.25f),
// float32 sums in position order.  work_off holds each stream's first block item.
__global__ void __launch_bounds__(kThreads) pool_kernel(const __grid_constant__ Common c,
                                                        int64_t total_chunks) {
    pdl_wait();
    pdl_trigger();
    const int H = c.n_kv_heads;
    constexpr int per_block = kIdxDim / kChunk;  // 16 (idx_dim is 128 when there are indexer rows)
    for (int64_t i = blockIdx.x * (int64_t)kThreads + threadIdx.x; i < total_chunks;
         i += (int64_t)gridDim.x * kThreads) {
        const int32_t item = static_cast<int32_t>(i / per_block);
        const int ch = static_cast<int>(i % per_block);
        const int s = find_seq(c.n_seqs, item, [&](int t) { return c.seq[t].work_off; });
        const SeqDev &sd = c.seq[s];
        const int32_t b = (sd.len - sd.n_new) / 4 + (item - sd.work_off);
        int32_t row;
        const int64_t page = page_or_bad(sd, 4 * b, &row, c.status);  // one lookup a block
        if (page < 0) continue;
        uint16_t *lb = const_cast<uint16_t *>(sd.layer_base) + page;
        const uint16_t *ik = lb + off_ik_f(c.kv_fp8, H, c.idx_dim, sd.ptok, row) + ch * kChunk;
        float sum[kChunk];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            uint4 u = *reinterpret_cast<const uint4 *>(ik + (int64_t)r * c.idx_dim);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < kChunk; ++e) {
                const uint32_t half = (e & 1) ? (w[e / 2] & 0xffff0000u) : (w[e / 2] << 16);
                const float x = __uint_as_float(half);
                sum[e] = r == 0 ? x : __fadd_rn(sum[e], x);
            }
        }
        uint32_t packed[4];
#pragma unroll
        for (int e = 0; e < kChunk; e += 2)
            packed[e / 2] = pack_bf16(__fmul_rn(sum[e], 0.25f), __fmul_rn(sum[e + 1], 0.25f));
        *reinterpret_cast<uint4 *>(lb + off_p_f(c.kv_fp8, H, c.idx_dim, sd.ptok, row / 4) + ch * kChunk) =
            make_uint4(packed[0], packed[1], packed[2], packed[3]);
    }
}

// e4m3 store: one warp per new row.  K and V rows are quantized (scale =
// max|x| / 448; code = e4m3 nearest x / scale, ties to even, saturating; the
// divisions in float32 with IEEE rounding), indexer rows copied.  Items per
// token: 2H quantized rows, then the indexer row.
__global__ void __launch_bounds__(kThreads) store8_kernel(const __grid_constant__ Common c,
                                                          int64_t total_items,
                                                          const uint16_t *__restrict__ k_new,
                                                          const uint16_t *__restrict__ v_new,
                                                          const uint16_t *__restrict__ ik_new) {
    pdl_wait();
    const int H = c.n_kv_heads, lane = threadIdx.x & 31;
    const int per_tok = 2 * H + (c.idx_dim ? 1 : 0);
    const int64_t warps = (int64_t)gridDim.x * (kThreads / 32);
    for (int64_t i = blockIdx.x * (int64_t)(kThreads / 32) + (threadIdx.x >> 5); i < total_items;
         i += warps) {
        const int32_t tok = static_cast<int32_t>(i / per_tok);
        const int32_t r = static_cast<int32_t>(i % per_tok);
        const int s = find_seq(c.n_seqs, tok, [&](int t) { return c.seq[t].tok_off; });
        const SeqDev &sd = c.seq[s];
        const int32_t pos = sd.len - sd.n_new + (tok - sd.tok_off);
        int32_t row;
        const int64_t page = page_or_bad(sd, pos, &row, c.status);
        if (page < 0) continue;  // warp-uniform: one row a warp
        uint8_t *lb = reinterpret_cast<uint8_t *>(const_cast<uint16_t *>(sd.layer_base)) + 2 * page;
        if (r < 2 * H) {
            const bool v = r >= H;
            const int head = r % H;
            const uint16_t *src = (v ? v_new : k_new) + ((int64_t)tok * H + head) * kHeadDim;
            uint2 codes;
            const float scale = quantize_row8(__ldg(reinterpret_cast<const uint4 *>(src) + lane), &codes);
            *reinterpret_cast<uint2 *>(lb + off8_code(v, H, sd.ptok, head, row) + lane * 8) = codes;
            if (lane == 0)
                *reinterpret_cast<float *>(lb + off8_scale(v, H, sd.ptok, head, row)) = scale;
        } else if (lane < c.idx_dim / kChunk) {
            const uint4 u = __ldg(reinterpret_cast<const uint4 *>(ik_new + (int64_t)tok * c.idx_dim) + lane);
            *reinterpret_cast<uint4 *>(lb + 2 * off_ik_f(true, H, c.idx_dim, sd.ptok, row) + 16 * lane) = u;
        }
    }
    pdl_trigger_after_writes();  // the next decode may read these rows early
}

// e4m3 gather: codes ([rows][H][256] bytes out) or scales ([rows][H] float32
// out) of positions 0 .. len-1 through the table.  A warp per position: the
// stream, page and row are found once; for codes lane l takes 16-byte chunk
// l & 15 of heads l >> 4, (l >> 4) + 2, ...; for scales lane l takes head l.
__global__ void __launch_bounds__(kThreads) gather8_kernel(const __grid_constant__ Common c,
                                                           int32_t kind, int32_t total_rows,
                                                           uint8_t *__restrict__ out) {
    pdl_wait();
    pdl_trigger();
    const int H = c.n_kv_heads;
    const bool codes = kind == PKV_K || kind == PKV_V;
    const bool v = kind == PKV_V || kind == PKV_VS;
    const int lane = threadIdx.x & 31;
    const int nwarps = gridDim.x * (kThreads / 32);
    for (int orow = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); orow < total_rows;
         orow += nwarps) {
        const int s = find_seq(c.n_seqs, orow, [&](int t) { return c.seq[t].work_off; });
        const SeqDev &sd = c.seq[s];
        int32_t row;
        const int64_t page = page_or_bad(sd, orow - sd.work_off, &row, lane == 0 ? c.status : nullptr);
        const uint8_t *lb = reinterpret_cast<const uint8_t *>(sd.layer_base) + 2 * page;
        if (codes) {
            const int ch = lane & 15;
            uint8_t *dst = out + (int64_t)orow * H * kHeadDim + 16 * ch;
            for (int h0 = lane >> 4; h0 < H; h0 += 2 * kBatch) {
                uint4 val[kBatch];
#pragma unroll
                for (int b = 0; b < kBatch; ++b) {
                    const int head = h0 + 2 * b;
                    val[b] = page >= 0 && head < H
                                 ? *reinterpret_cast<const uint4 *>(lb + off8_code(v, H, sd.ptok, head, row) + 16 * ch)
                                 : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int b = 0; b < kBatch; ++b)
                    if (h0 + 2 * b < H)
                        *reinterpret_cast<uint4 *>(dst + (int64_t)(h0 + 2 * b) * kHeadDim) = val[b];
            }
        } else {
            for (int head = lane; head < H; head += 32)
                reinterpret_cast<float *>(out)[(int64_t)orow * H + head] =
                    page >= 0 ? *reinterpret_cast<const float *>(lb + off8_scale(v, H, sd.ptok, head, row)) : 0.f;
        }
    }
}

unsigned grid_for(int64_t work) {
    int64_t g = (work + kThreads - 1) / kThreads;
    return static_cast<unsigned>(g < 1 ? 1 : (g > 65535 * 4 ? 65535 * 4 : g));
}

}  // namespace

int launch_store(const Common &c, int32_t total_tokens, const uint16_t *k_new,
                 const uint16_t *v_new, const uint16_t *ik_new, cudaStream_t stream) {
    // a warp a token
    return launch_status(launch_pdl(store_kernel, grid_for((int64_t)total_tokens * 32), kThreads,
                                    0, stream, c, total_tokens, k_new, v_new, ik_new));
}

int launch_gather(const Common &c, int32_t kind, int64_t total_rows, uint16_t *out,
                  cudaStream_t stream) {
    if (total_rows > INT32_MAX - 64) return PKV_EINVAL;  // int32 row indices
    const int rows = static_cast<int32_t>(total_rows);
    if (kind == PKV_K || kind == PKV_V)  // a warp a row
        return launch_status(launch_pdl(gather_kernel<true>, grid_for(total_rows * 32), kThreads,
                                        0, stream, c, kind, rows, out));
    return launch_status(launch_pdl(gather_kernel<false>, grid_for(total_rows * 16), kThreads, 0,
                                    stream, c, kind, rows, out));  // a half-warp a row
}

int launch_store8(const Common &c, int32_t total_tokens, const uint16_t *k_new,
                  const uint16_t *v_new, const uint16_t *ik_new, cudaStream_t stream) {
    const int64_t items = (int64_t)total_tokens * (2 * c.n_kv_heads + (c.idx_dim ? 1 : 0));
    return launch_status(launch_pdl(store8_kernel, grid_for(items * 32), kThreads, 0, stream, c,
                                    items, k_new, v_new, ik_new));
}

int launch_gather8(const Common &c, int32_t kind, int64_t total_rows, void *out,
                   cudaStream_t stream) {
    if (total_rows > INT32_MAX - 64) return PKV_EINVAL;  // int32 row indices
    return launch_status(launch_pdl(gather8_kernel, grid_for(total_rows * 32), kThreads, 0, stream,
                                    c, kind, static_cast<int32_t>(total_rows),
                                    static_cast<uint8_t *>(out)));  // a warp a position
}

int launch_pool(const Common &c, int32_t total_blocks, cudaStream_t stream) {
    const int64_t total = (int64_t)total_blocks * (c.idx_dim / kChunk);
    return launch_status(launch_pdl(pool_kernel, grid_for(total), kThreads, 0, stream, c, total));
}

}  // namespace pkv
