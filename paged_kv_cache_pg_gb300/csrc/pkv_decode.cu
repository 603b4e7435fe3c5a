// Decode attention over paged caches: split-KV partials and their combine.
//
// Work unit: (stream, KV head, split) for dense decode, where the G query
// heads of the KV head (times the stream's n_new queries) share every staged
// key/value tile; (stream, query head, split) for block-sparse decode, whose
// keys are the positions of that head's selected blocks.
//
// One CTA = eight warps.  The unit's 16-key tiles are dealt round robin to
// key slices; each slice is a pair of warps per column group of 8 query
// columns (both compute S for the tile, each accumulates O for half of the
// 256 dims).  A slice's lead warp stages its tiles into the slice's share of
// the CTA's twelve 16 KB stage slots: it looks each key's row up once per
// tile (#1169: key_at once per key per tile, beside the key ids; kept here as
// the split's page offsets in shared memory and the row addresses in the
// lanes) and copies a whole 16-row page run by 2D TMA, or key by key with
// cp.async.  Cached rows more than 32 positions below the new tokens stream
// before the grid-dependency wait, and every dense CTA lets the next kernel
// start at entry; tiles past the slots are prefetched into L2.  The warps
// compute S^T = K Q^T and O^T += V^T P^T with warp MMAs (bf16 in, float32
// accumulate), keep an online softmax per query column, and merge their key
// slices in a fixed order.  Splits have a fixed length set by the stream's
// key count and the SM count, so paged and contiguous caches give the same
// bits.  A second kernel merges the splits: a CTA a query column
// (decode_combine), or, for calls with thousands of columns and few splits
// (a prefill chunk), a warp a column (combine_cols).  Units of more than 16
// query columns (draft windows) are routed to the tensor-core chunk kernel
// by the host and never reach these kernels.
#include <algorithm>
#include <cfloat>
#include <mutex>

#include "pkv_dev.cuh"

namespace pkv {
namespace {

#ifndef PKV_DECODE_SLOTS
#define PKV_DECODE_SLOTS 12
#endif
#ifndef PKV_DECODE_MIN_SPLIT
#define PKV_DECODE_MIN_SPLIT 256
#endif
#ifndef PKV_SPARSE_MIN_SPLIT
#define PKV_SPARSE_MIN_SPLIT 64
#endif

constexpr int kTile = 16;                    // keys a stage slot
constexpr int kPlane = 2048;                 // one 64-dim column chunk of 16 rows (bytes)
constexpr int kHalfStage = 4 * kPlane;       // the K (or V) tile: 16 rows x 512 B, swizzled
constexpr int kStageBytes = 2 * kHalfStage;
constexpr int kSlots = PKV_DECODE_SLOTS;     // stage slots of a CTA, shared by its key slices
constexpr int kWarps = 8;                    // 2 per tile share the dims (halves)
constexpr int kThreads = kWarps * 32;
constexpr int kMaxCols = 32;                 // query columns of one unit
constexpr int kMinSplitDense = PKV_DECODE_MIN_SPLIT;    // keys
constexpr int kMinSplitSparse = PKV_SPARSE_MIN_SPLIT;
constexpr int kMaxSplitLen = 1024;           // keys of one split (bounds the page list)
constexpr int kMaxSplits = 2048;
// Rows read before the grid-dependency wait lie at least this many positions
// below a stream's new tokens: a decode of the same stream queued just before
// (its fused store writes at most 32 rows, right below this call's new
// tokens) may still be writing the rows above.
constexpr int kFreshGuard = 32;
constexpr int kCombThreads = 256;
constexpr int kMaxPages = kMaxSplitLen / 4 + 2;  // pages one split can touch
constexpr int kMaxSparseBlocks = kMaxSplitLen / 4;
constexpr int kMergeStride = kHeadDim + 4;   // floats; spreads the 4 column pairs over banks
constexpr float kScaleLog2 = 0.0625f * 1.4426950408889634f;  // log2(e) / sqrt(256)

constexpr size_t kOffPos = (size_t)kSlots * kStageBytes;
constexpr size_t kOffPage = kOffPos + kSlots * kTile * 4;
constexpr size_t kOffBar = kOffPage + ((kMaxPages + 1) & ~1) * 8;
constexpr size_t kSmemBytes = 1024 + kOffBar + 2 * kSlots * 8 + 16;  // + alignment slack
static_assert(kMaxPages >= kMaxSparseBlocks, "the page list also holds block rows");
static_assert(kSlots % (kWarps / 2) == 0, "every key slice gets the same number of slots");
static_assert(kMaxCols * kMergeStride * 4 + kMaxCols * 2 * 4 <= kSlots * kStageBytes,
              "merge buffers reuse the stages");

struct DecodeArgs {
    const uint16_t *q;
    uint16_t *out;
    float *ws;
    const int32_t *ids;  // sparse: [n_seqs][n_q_heads][k]
    int32_t k;
    const uint16_t *k_new;   // fused store of the new tokens (dense), or null
    const uint16_t *v_new;
    const uint16_t *ik_new;
};

// Byte offset of 16-byte chunk c (0..31 along the 512-byte row) of row r
// (0..15) inside a K or V tile.  The tile is four 2 KB planes (one per 64
// dims), each 16 rows of 128 B with the TMA 128-byte swizzle: chunk c & 7 of
// row r sits at position (c & 7) ^ (r & 7).
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return (c >> 3) * kPlane + r * 128 + ((((c & 7) ^ (r & 7))) << 4);
}

__device__ __forceinline__ float warp_max_lanes(float v) {
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
    return v;
}

__device__ __forceinline__ float warp_sum_lanes(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    v += __shfl_xor_sync(0xffffffffu, v, 8);
    v += __shfl_xor_sync(0xffffffffu, v, 16);
    return v;
}

struct Unit {
    int s, unit, split, kvh;
    int key0, key1, ntiles;
};

template <bool kSparse>
__device__ __forceinline__ Unit locate(const Common &c, const DecodeArgs &a) {
    Unit u;
    u.s = find_seq(c.n_seqs, blockIdx.x, [&](int t) { return c.seq[t].work_off; });
    const SeqDev &sd = c.seq[u.s];
    const int r = blockIdx.x - sd.work_off;
    u.unit = r / sd.nsplit;
    u.split = r - u.unit * sd.nsplit;
    u.kvh = kSparse ? u.unit / c.group : u.unit;
    const int nkeys = kSparse ? 4 * a.k : sd.len;
    u.key0 = u.split * sd.split_len;
    u.key1 = min(nkeys, u.key0 + sd.split_len);
    u.ntiles = (u.key1 - u.key0 + kTile - 1) / kTile;
    return u;
}

// Packed row of query column `col` of the unit.
template <bool kSparse>
__device__ __forceinline__ int64_t q_row(const Common &c, const SeqDev &sd, const Unit &u,
                                         int col) {
    if (kSparse) return (int64_t)sd.tok_off * c.n_q_heads + u.unit;
    const int j = col / c.group;
    return ((int64_t)sd.tok_off + j) * c.n_q_heads + u.kvh * c.group + (col - j * c.group);
}


// The state one CTA shares between its warps.
struct Ctx {
    uint8_t *stages;
    int32_t *kpos;       // [slot][16] key positions (-1 masked)
    int64_t *rows;       // dense: offsets of the split's pages; sparse: K rows of its blocks
    uint64_t *full;      // [slot]
    uint64_t *empty;     // [slot]
    volatile int *abort_flag;
    int first_page;      // dense: page of the split's first key
    int64_t fallback;    // sparse: a row surely written (position 0)
};

// Stage tile t of the unit into `slot` (one warp).  A whole tile of cached
// rows inside one page whose rows sit on the stream's TMA map is one 2D tensor
// copy per 64-dim chunk (8 per tile, K and V); any other tile (the ragged
// tail, new rows, pages not a multiple of 16, selected blocks) goes key by key
// with 16-byte cp.async through the same swizzle, from one row lookup per key.
// With a fused store, new rows come from k_new/v_new and are written to the
// cache here as well.  The copies complete on `bar`.
template <bool kSparse>
__device__ __forceinline__ void stage_tile(const Common &c, const DecodeArgs &a,
                                           const DecodeMaps &maps, const SeqDev &sd,
                                           const Unit &u, const Ctx &x, int t, int slot,
                                           uint64_t *bar, int lane, uint64_t pol) {
    const int H = c.n_kv_heads;
    const int qbase = sd.len - sd.n_new;
    const int64_t v_gap = (int64_t)H * sd.ptok * kHeadDim;  // V row - K row
    const bool fuse_store = !kSparse && a.k_new != nullptr;
    const int i = u.key0 + t * kTile + lane;  // key index of this lane (lane < 16)
    const bool mine = lane < kTile && i < u.key1;
    int pos = -1;            // live key position, or -1 (masked)
    int64_t krow = 0;        // element offset of the K row from layer_base
    bool bad = false;        // its page id was outside the arena
    bool fresh = false;      // the row comes from the new-token input
    if (kSparse) {
        krow = x.fallback;
        if (mine) {
            const int64_t off = x.rows[(i - u.key0) >> 2];
            if (off >= 0) {
                pos = i;
                krow = off + (int64_t)(i & 3) * kHeadDim;
            }
        }
    } else {
        const int key = lane < kTile ? min(i, u.key1 - 1) : u.key0;
        int row = key;
        int64_t pg = 0;
        if (sd.table) {
            const int page = key / sd.ptok;
            row = key - page * sd.ptok;
            pg = x.rows[page - x.first_page];
            if (pg < 0) {
                bad = true;
                pg = 0;
            }
        }
        krow = pg + off_k(sd.ptok, u.kvh, row);
        if (mine) pos = i;
        fresh = fuse_store && key >= qbase;
    }
    if (lane < kTile) x.kpos[slot * kTile + lane] = pos;
    uint8_t *kst = x.stages + slot * kStageBytes;
    uint8_t *vst = kst + kHalfStage;
    const void *map = (!kSparse && sd.tma >= 0) ? &maps.map[sd.tma] : nullptr;
    const bool tile_tma =
        map != nullptr && __all_sync(0xffffffffu, lane >= kTile || (pos >= 0 && !fresh));
    __syncwarp();
    if (tile_tma) {
        if (lane == 0) {
            const int y = static_cast<int>(sd.layer_row + krow / kHeadDim);  // row-aligned
            const int yv = y + static_cast<int>(v_gap / kHeadDim);
            mbar_arrive_expect_tx(bar, kTile * 2 * 512);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                tma_load_2d(kst + j * kPlane, map, 64 * j, y, bar, pol);
                tma_load_2d(vst + j * kPlane, map, 64 * j, yv, bar, pol);
            }
        }
    } else {
        const uint16_t *ksrc, *vsrc;
        if (fresh) {
            const int key = min(i, u.key1 - 1);
            const int64_t r = ((int64_t)sd.tok_off + (key - qbase)) * H + u.kvh;
            ksrc = a.k_new + r * kHeadDim;
            vsrc = a.v_new + r * kHeadDim;
        } else {
            ksrc = sd.layer_base + krow;
            vsrc = ksrc + v_gap;
        }
        const int64_t kp = reinterpret_cast<int64_t>(ksrc);
        const int64_t vp = reinterpret_cast<int64_t>(vsrc);
#pragma unroll 4
        for (int r = 0; r < kTile; ++r) {
            const uint16_t *kr = reinterpret_cast<const uint16_t *>(shfl64(kp, r));
            const uint16_t *vr = reinterpret_cast<const uint16_t *>(shfl64(vp, r));
            cp_async16(kst + swz(r, lane), kr + lane * 8, pol);
            cp_async16(vst + swz(r, lane), vr + lane * 8, pol);
        }
        cp_async_mbar_arrive(bar);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar);
    }
    if (fuse_store) {
        unsigned todo = __ballot_sync(0xffffffffu, fresh && pos >= 0 && !bad);
        while (todo) {
            const int src = __ffs(todo) - 1;
            todo &= todo - 1;
            const int p = __shfl_sync(0xffffffffu, pos, src);
            const int64_t kr = shfl64(krow, src);
            const int64_t r = (int64_t)sd.tok_off + (p - qbase);
            uint16_t *dst = const_cast<uint16_t *>(sd.layer_base) + kr;
            const uint4 kv =
                __ldg(reinterpret_cast<const uint4 *>(a.k_new + (r * H + u.kvh) * kHeadDim) + lane);
            const uint4 vv =
                __ldg(reinterpret_cast<const uint4 *>(a.v_new + (r * H + u.kvh) * kHeadDim) + lane);
            reinterpret_cast<uint4 *>(dst)[lane] = kv;
            reinterpret_cast<uint4 *>(dst + v_gap)[lane] = vv;
            if (u.kvh == 0 && a.ik_new != nullptr && lane < c.idx_dim / 8) {
                // the indexer-key row of the same position, written once (KV head 0)
                const int prow = sd.table ? p % sd.ptok : p;
                const int64_t page_start = kr - (int64_t)prow * kHeadDim;
                uint16_t *idst = const_cast<uint16_t *>(sd.layer_base) + page_start +
                                 off_ik(H, c.idx_dim, sd.ptok, prow);
                reinterpret_cast<uint4 *>(idst)[lane] =
                    __ldg(reinterpret_cast<const uint4 *>(a.ik_new + r * c.idx_dim) + lane);
            }
        }
    }
}

// Prefetch the cached K and V rows of dense tile t into L2 (one warp).  Tiles
// past a key slice's stage slots are only staged after the slice consumes its
// first tiles; fetching their rows into L2 while the CTA waits on the previous
// kernel takes them off that path.  Tiles holding new positions are skipped.
__device__ __forceinline__ void prefetch_tile(const Common &c, const SeqDev &sd, const Unit &u,
                                              const Ctx &x, int t, int lane) {
    const int qbase = sd.len - sd.n_new;
    const int k0 = u.key0 + t * kTile;
    if (k0 + kTile > min(u.key1, qbase)) return;  // ragged or holds new rows
    const int64_t v_gap = (int64_t)c.n_kv_heads * sd.ptok * kHeadDim;
    const bool run = sd.table == nullptr || sd.ptok % kTile == 0;  // 16 rows in one page
    const int key = k0 + (run ? 0 : (lane & 15));
    int row = key;
    int64_t pg = 0;
    if (sd.table) {
        const int page = key / sd.ptok;
        row = key - page * sd.ptok;
        pg = x.rows[page - x.first_page];
        if (pg < 0) return;  // reported when the tile is staged
    }
    const uint16_t *kr = sd.layer_base + pg + off_k(sd.ptok, u.kvh, row);
    if (run) {
        if (lane == 0) {
            bulk_prefetch_l2(kr, kTile * 512);
            bulk_prefetch_l2(kr + v_gap, kTile * 512);
        }
    } else if (lane < kTile) {
        bulk_prefetch_l2(kr, 512);
        bulk_prefetch_l2(kr + v_gap, 512);
    }
}

template <bool kSparse>
__global__ void __launch_bounds__(kThreads, 1)
    decode_partial(const __grid_constant__ Common c, const __grid_constant__ DecodeMaps maps,
                   const DecodeArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ctx x;
    x.stages = smem;
    x.kpos = reinterpret_cast<int32_t *>(smem + kOffPos);
    x.rows = reinterpret_cast<int64_t *>(smem + kOffPage);
    x.full = reinterpret_cast<uint64_t *>(smem + kOffBar);
    x.empty = x.full + kSlots;
    x.abort_flag = reinterpret_cast<volatile int *>(x.empty + kSlots);

    const int tid = threadIdx.x, lane = tid & 31;
    const int dh = (tid >> 5) & 1;              // which half of the 256 dims this warp sums
    const int warp = tid >> 6;                  // warp pair: one column group of one key slice
    const Unit u = locate<kSparse>(c, a);
    const SeqDev &sd = c.seq[u.s];
    const int ncols = sd.ncols;
    const int ncg = (ncols + 7) >> 3;           // column groups
    const int ks_n = (kWarps / 2) / ncg;        // key slices
    const int S = kSlots / ks_n;                // slots of one key slice
    const int cg = warp % ncg, ks = warp / ncg;
    const bool active = ks < ks_n;
    const bool leader = active && cg == 0 && dh == 0;  // stages its slice's tiles
    const int qbase = sd.len - sd.n_new;

    if (tid == 0) {
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(&x.full[i], 1);
            mbar_init(&x.empty[i], 2 * ncg);
        }
        *x.abort_flag = 0;
        fence_mbar_init();
    }
    // one row lookup per page (dense) or per selected block (sparse) of the split
    x.first_page = 0;
    x.fallback = 0;
    if (kSparse) {
        pdl_wait();  // the selected ids come from the previous kernel
        const int32_t *ids = a.ids + ((int64_t)u.s * c.n_q_heads + u.unit) * a.k;
        const int nb = sd.len / 4;
        const int b0 = u.key0 >> 2, nblk = (u.key1 - u.key0 + 3) >> 2;
        for (int j = tid; j < nblk; j += kThreads) {
            const int b = __ldg(ids + b0 + j);
            int64_t off = -1;
            if (b >= 0 && b < nb) {
                int32_t row;
                int64_t pg = 0;
                if (sd.table) {
                    const int page = (4 * b) / sd.ptok;
                    row = 4 * b - page * sd.ptok;
                    const int id = __ldg(sd.table + page);
                    pg = static_cast<uint32_t>(id) < static_cast<uint32_t>(sd.n_pages)
                             ? (int64_t)id * sd.ps
                             : -1;
                } else {
                    row = 4 * b;
                }
                if (pg >= 0) off = pg + off_k(sd.ptok, u.kvh, row);
            }
            if ((b >= nb || (b >= 0 && off < 0)) && c.status) atomicOr(c.status, PKV_DEV_BAD_PAGE);
            x.rows[j] = off;
        }
        int64_t fb = 0;
        if (sd.table) {
            const int id = __ldg(sd.table);
            if (static_cast<uint32_t>(id) < static_cast<uint32_t>(sd.n_pages)) fb = (int64_t)id * sd.ps;
        }
        x.fallback = fb + off_k(sd.ptok, u.kvh, 0);
    } else if (sd.table) {
        x.first_page = u.key0 / sd.ptok;
        const int npages = (u.key1 - 1) / sd.ptok - x.first_page + 1;
        for (int j = tid; j < npages; j += kThreads) {
            const int p = x.first_page + j;
            int64_t off = -1;
            if (p < sd.n_table) {
                const int id = __ldg(sd.table + p);
                if (static_cast<uint32_t>(id) < static_cast<uint32_t>(sd.n_pages))
                    off = (int64_t)id * sd.ps;
            }
            if (off < 0 && c.status) atomicOr(c.status, PKV_DEV_BAD_PAGE);
            x.rows[j] = off;
        }
    }
    __syncthreads();
    // dense: nothing this CTA writes is read by the next kernel before its own
    // wait (a decode reads no row within kFreshGuard of its new tokens early)
    if (!kSparse && tid == 0) pdl_trigger();

    const uint64_t pol = policy_evict_first();
    // Rows of cached positions more than kFreshGuard below the new tokens do
    // not depend on the previous kernel on the stream: the first tiles stream
    // before the grid-dependency wait (the call's prefetch kernel has asked L2
    // for the rest).  Other tiles, the queries and every write wait for it.
    const int early_end = qbase - kFreshGuard;
    const int my_tiles = active ? (u.ntiles - ks + ks_n - 1) / ks_n : 0;  // tiles ks, ks+ks_n, ...
    bool waited = kSparse;
    int issued = 0;
    if (leader) {
        for (; issued < S && issued < my_tiles; ++issued) {
            const int t = ks + issued * ks_n;
            if (!waited && u.key0 + t * kTile + kTile > early_end) {
                pdl_wait();
                waited = true;
            }
            stage_tile<kSparse>(c, a, maps, sd, u, x, t, ks * S + issued, &x.full[ks * S + issued], lane, pol);
        }
        if (!kSparse && !waited)
            for (int j = issued; j < my_tiles && j < 2 * S; ++j)
                if (u.key0 + (ks + j * ks_n) * kTile + kTile <= early_end)
                    prefetch_tile(c, sd, u, x, ks + j * ks_n, lane);
    }
    // the query row's address from the launch parameters before the wait
    // (an asm use the compiler cannot move past it): only its load waits
    const int bcol = cg * 8 + (lane >> 2);
    const uint16_t *const qr =
        (active && bcol < ncols) ? a.q + q_row<kSparse>(c, sd, u, bcol) * kHeadDim : nullptr;
    asm volatile("" ::"l"(qr));
    if (!waited) pdl_wait();

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float acc[8][4];  // O^T for dims 128*dh .. 128*dh+127
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

    if (active) {
        uint32_t qf[16][2];
        {
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) {
                const int d = kk * 16 + 2 * (lane & 3);
                qf[kk][0] = qr ? __ldg(reinterpret_cast<const uint32_t *>(qr + d)) : 0u;
                qf[kk][1] = qr ? __ldg(reinterpret_cast<const uint32_t *>(qr + d + 8)) : 0u;
            }
        }
        // the two columns this lane owns in S^T and O^T fragments, and the
        // last key position each may read (causal; -1 for a padding column)
        const int c0 = cg * 8 + 2 * (lane & 3), c1 = c0 + 1;
        const int lim0 = c0 < ncols ? (kSparse ? INT32_MAX : qbase + c0 / c.group) : -1;
        const int lim1 = c1 < ncols ? (kSparse ? INT32_MAX : qbase + c1 / c.group) : -1;

        const uint32_t s_base = smem_u32(x.stages);
        // ldmatrix rows: K fragments take keys (lane & 7) + 8 * bit 3, V^T fragments
        // keys (lane & 7) + 8 * bit 4; column chunk bit from bit 4 (K) or bit 3 (V)
        const int kr_ = (lane & 7) + 8 * ((lane >> 3) & 1), kcb = lane >> 4;
        const int vr_ = (lane & 7) + 8 * (lane >> 4), vcb = (lane >> 3) & 1;

        for (int j = 0; j < my_tiles; ++j) {
            const int slot = ks * S + j % S;
            if (!mbar_wait(&x.full[slot], (j / S) & 1, c.status)) {
                *x.abort_flag = 1;
                break;
            }
            const uint32_t kb = s_base + slot * kStageBytes;
            const uint32_t vb = kb + kHalfStage;
            // S^T[16 keys x 8 cols] = K Q^T, two accumulator chains
            float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < 16; kk += 2) {
                uint32_t x0, x1, x2, x3;
                ldsm_x4(kb + swz(kr_, 2 * kk + kcb), x0, x1, x2, x3);
                mma_bf16(sa, x0, x1, x2, x3, qf[kk][0], qf[kk][1]);
                ldsm_x4(kb + swz(kr_, 2 * (kk + 1) + kcb), x0, x1, x2, x3);
                mma_bf16(sb, x0, x1, x2, x3, qf[kk + 1][0], qf[kk + 1][1]);
            }
            const int kp0 = x.kpos[slot * kTile + (lane >> 2)];
            const int kp1 = x.kpos[slot * kTile + (lane >> 2) + 8];
            const float x0 = (kp0 >= 0 && kp0 <= lim0) ? (sa[0] + sb[0]) * kScaleLog2 : -INFINITY;
            const float x1 = (kp0 >= 0 && kp0 <= lim1) ? (sa[1] + sb[1]) * kScaleLog2 : -INFINITY;
            const float x2 = (kp1 >= 0 && kp1 <= lim0) ? (sa[2] + sb[2]) * kScaleLog2 : -INFINITY;
            const float x3 = (kp1 >= 0 && kp1 <= lim1) ? (sa[3] + sb[3]) * kScaleLog2 : -INFINITY;
            const float n0 = fmaxf(m0, warp_max_lanes(fmaxf(x0, x2)));
            const float n1 = fmaxf(m1, warp_max_lanes(fmaxf(x1, x3)));
            const float b0 = n0 == -INFINITY ? 0.f : n0;
            const float b1 = n1 == -INFINITY ? 0.f : n1;
            const float al0 = ex2(m0 - b0), al1 = ex2(m1 - b1);
            const float p0 = ex2(x0 - b0), p1 = ex2(x1 - b1);
            const float p2 = ex2(x2 - b0), p3 = ex2(x3 - b1);
            l0 = l0 * al0 + (p0 + p2);
            l1 = l1 * al1 + (p1 + p3);
            m0 = n0;
            m1 = n1;
            // P as a bf16 pair hi + lo (lo = p - hi is exact in float32), so the
            // weights reach the float32 accumulator with ~16 significant bits
            const uint32_t h01 = pack_bf16(p0, p1), h23 = pack_bf16(p2, p3);
            const uint32_t l01 = pack_bf16(p0 - bf16_lo(h01), p1 - bf16_hi(h01));
            const uint32_t l23 = pack_bf16(p2 - bf16_lo(h23), p3 - bf16_hi(h23));
            const uint32_t pb0 = movmatrix_t(h01), pb1 = movmatrix_t(h23);
            const uint32_t pc0 = movmatrix_t(l01), pc1 = movmatrix_t(l23);
            // O^T[16 dims x 8 cols] += V^T P^T for this warp's 8 dim tiles
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                acc[i][0] *= al0;
                acc[i][1] *= al1;
                acc[i][2] *= al0;
                acc[i][3] *= al1;
                uint32_t y0, y1, y2, y3;
                ldsm_x4_t(vb + swz(vr_, 2 * (8 * dh + i) + vcb), y0, y1, y2, y3);
                mma_bf16(acc[i], y0, y1, y2, y3, pb0, pb1);
                mma_bf16(acc[i], y0, y1, y2, y3, pc0, pc1);
            }
            // release the slot; the slice's leader refills it with tile j + S
            __syncwarp();
            if (lane == 0) mbar_arrive(&x.empty[slot]);
            if (leader && issued < my_tiles) {
                if (!mbar_wait(&x.empty[slot], (j / S) & 1, c.status)) {
                    *x.abort_flag = 1;
                    break;
                }
                fence_proxy_async_smem();  // this slot's reads come before the next tile's writes
                stage_tile<kSparse>(c, a, maps, sd, u, x, ks + (j + S) * ks_n, slot, &x.full[slot], lane, pol);
                ++issued;
            }
        }
        l0 = warp_sum_lanes(l0);
        l1 = warp_sum_lanes(l1);
    }
    if (leader && *x.abort_flag) {
        // let every copy this slice issued land before the CTA's memory is released
        for (int j = issued > S ? issued - S : 0; j < issued; ++j)
            mbar_wait(&x.full[ks * S + j % S], (j / S) & 1, nullptr);
    }

    __syncthreads();
    if (kSparse) pdl_trigger();  // every thread has passed its grid-dependency wait
    if (*x.abort_flag) return;

    // ---- merge the key slices (ks = 0, 1, ...) in order, inside the CTA ----
    const int NC = ncg * 8;
    float *mbuf = reinterpret_cast<float *>(x.stages);            // [ks][NC][kMergeStride]
    float *mlb = mbuf + ks_n * NC * kMergeStride;                  // [ks][NC][2]
    if (active) {
        const int c0 = cg * 8 + 2 * (lane & 3);
        float *b0 = mbuf + (ks * NC + c0) * kMergeStride;
        float *b1 = b0 + kMergeStride;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int d = (8 * dh + i) * 16 + (lane >> 2);
            b0[d] = acc[i][0];
            b1[d] = acc[i][1];
            b0[d + 8] = acc[i][2];
            b1[d + 8] = acc[i][3];
        }
        if (dh == 0 && (lane >> 2) == 0) {
            mlb[(ks * NC + c0) * 2 + 0] = m0;
            mlb[(ks * NC + c0) * 2 + 1] = l0;
            mlb[(ks * NC + c0 + 1) * 2 + 0] = m1;
            mlb[(ks * NC + c0 + 1) * 2 + 1] = l1;
        }
    }
    __syncthreads();

    const bool single = sd.nsplit == 1;
    const int units = kSparse ? c.n_q_heads : c.n_kv_heads;
    float *part_acc = a.ws + sd.ws_off;
    float *part_ml = part_acc + (int64_t)units * sd.nsplit * ncols * kHeadDim;
    const int64_t pidx = ((int64_t)u.unit * sd.nsplit + u.split) * ncols;
    // four consecutive dims a thread: the slices' weights of the column
    // (each thread of a column computes the same ones), O = sum over slices in order
    for (int idx = tid; idx < ncols * (kHeadDim / 4); idx += kThreads) {
        const int col = idx / (kHeadDim / 4), d = 4 * (idx - col * (kHeadDim / 4));
        float M = -INFINITY;
        for (int k = 0; k < ks_n; ++k) M = fmaxf(M, mlb[(k * NC + col) * 2]);
        float L = 0.f;
        float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int k = 0; k < ks_n; ++k) {
            const float w = M == -INFINITY ? 0.f : ex2(mlb[(k * NC + col) * 2] - M);
            L += w * mlb[(k * NC + col) * 2 + 1];
            const float4 v = *reinterpret_cast<const float4 *>(mbuf + (k * NC + col) * kMergeStride + d);
            O.x += w * v.x;
            O.y += w * v.y;
            O.z += w * v.z;
            O.w += w * v.w;
        }
        if (single) {
            const float inv = L > 0.f ? 1.f : 0.f;
            const float lz = L > 0.f ? L : 1.f;
            uint2 pk;
            pk.x = pack_bf16(inv * (O.x / lz), inv * (O.y / lz));
            pk.y = pack_bf16(inv * (O.z / lz), inv * (O.w / lz));
            *reinterpret_cast<uint2 *>(a.out + q_row<kSparse>(c, sd, u, col) * kHeadDim + d) = pk;
        } else {
            *reinterpret_cast<float4 *>(part_acc + (pidx + col) * kHeadDim + d) = O;
            if (d == 0) {
                part_ml[(pidx + col) * 2 + 0] = M;
                part_ml[(pidx + col) * 2 + 1] = L;
            }
        }
    }
}

// Combine a unit's split partials for one query column:
// M = max m_i, L = sum 2^(m_i-M) l_i, O = sum 2^(m_i-M) acc_i, out = O / L.
// A column of a stream with up to 32 splits is one CTA, a thread a dim; past
// 32 splits it is two CTAs of 128 dims whose threads form two groups of 128
// (one thread a dim): group 0 sums the first ceil(ns/2) splits, group 1 the
// rest, and O = O_0 + O_1 (comb_ctas).  Every sum of O runs in split order.
// Each warp finds M and L itself: lane l reads (m, l) of splits l, l + 32,
// ..., and shuffles reduce them in a fixed order, so every warp gets the same
// bits without waiting on another warp.  The weights of each batch of 32
// splits (lane l: split b + l) pass through the warp's own shared row.  A
// thread issues its first 32 values together with those pairs, so one memory
// round trip covers a column of up to 64 splits.  At most 64 registers a
// thread: a combine CTA then fits on an SM beside a partial CTA of the next
// call, which can start streaming its keys without waiting for the SM.
template <bool kSparse>
__global__ void __launch_bounds__(kCombThreads, 4)
    decode_combine(const __grid_constant__ Common c, const DecodeArgs a) {
    constexpr int kBatch = 32;
    __shared__ float sh_o[kHeadDim / 2];
    __shared__ float sh_w[kCombThreads / 32][kBatch];  // a warp's weights of one batch
    // the next kernel may start now: it waits for this grid before reading
    // anything this grid writes, and its CTAs stream their cached rows meanwhile
    pdl_trigger();
    // everything below up to the partials' loads reads the launch parameters
    // only: done before the wait, its constant-cache misses (the stream
    // search, the stream's fields) overlap the partial kernel's tail
    const int s = find_seq(c.n_seqs, blockIdx.x, [&](int t) { return c.seq[t].comb_off; });
    const SeqDev &sd = c.seq[s];
    const int ns = sd.nsplit;
    const int halves = comb_ctas(ns);
    const int r = (blockIdx.x - sd.comb_off) / halves;  // (unit, column) of the stream
    const int unit = r / sd.ncols, col = r - unit * sd.ncols;
    const int units = kSparse ? c.n_q_heads : c.n_kv_heads;
    const float *part_acc = a.ws + sd.ws_off;
    const float2 *part_ml =
        reinterpret_cast<const float2 *>(part_acc + (int64_t)units * ns * sd.ncols * kHeadDim);
    const int64_t p0 = (int64_t)unit * ns * sd.ncols + col;  // split i at p0 + i * ncols
    const int64_t stride = (int64_t)sd.ncols * kHeadDim;
    const float2 *col_ml = part_ml + p0;
    const int tid = threadIdx.x, lane = tid & 31;
    // two CTAs: 128 dims each, thread t in group t >> 7; one CTA: all 256 dims, one group
    const int grp = halves == 2 ? tid >> 7 : 0, dd = halves == 2 ? tid & 127 : tid;
    const int d = halves == 2 ? (((blockIdx.x - sd.comb_off) & 1) << 7) + dd : dd;
    const int i0 = halves == 2 && grp ? (ns + 1) >> 1 : 0;  // this group's splits
    const int i1 = halves == 2 && !grp ? (ns + 1) >> 1 : ns;
    const float *col_acc = part_acc + p0 * kHeadDim + d;
    const int warp = tid >> 5;
    const int64_t orow = q_row<kSparse>(c, sd, Unit{0, unit, 0, kSparse ? unit / c.group : unit, 0, 0, 0}, col);
    // the addresses are in registers before the wait (an asm use the compiler
    // cannot move past it)
    asm volatile("" ::"l"(col_acc), "l"(col_ml), "l"(stride), "l"(orow), "r"(i0), "r"(i1), "r"(ns));
    pdl_wait();
    float xs[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) xs[j] = i0 + j < i1 ? __ldcg(col_acc + (i0 + j) * stride) : 0.f;
    const float2 none = make_float2(-INFINITY, 0.f);
    const float2 ml0 = lane < ns ? __ldcg(col_ml + (int64_t)lane * sd.ncols) : none;
    const float2 ml1 = lane + 32 < ns ? __ldcg(col_ml + (int64_t)(lane + 32) * sd.ncols) : none;
    float2 mlb = i0 + lane < i1 ? __ldcg(col_ml + (int64_t)(i0 + lane) * sd.ncols) : none;
    float M = fmaxf(ml0.x, ml1.x);
    for (int i = lane + 64; i < ns; i += 32) M = fmaxf(M, __ldcg(col_ml + (int64_t)i * sd.ncols).x);
#pragma unroll
    for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const bool empty = M == -INFINITY;  // no split saw a key
    float L = (empty ? 0.f : ex2(ml0.x - M)) * ml0.y + (empty ? 0.f : ex2(ml1.x - M)) * ml1.y;
    for (int i = lane + 64; i < ns; i += 32) {
        const float2 v = __ldcg(col_ml + (int64_t)i * sd.ncols);
        L += (empty ? 0.f : ex2(v.x - M)) * v.y;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    float O = 0.f;
    for (int b = i0; b < i1; b += kBatch) {
        if (b > i0) {
#pragma unroll
            for (int j = 0; j < kBatch; ++j) xs[j] = b + j < i1 ? __ldcg(col_acc + (b + j) * stride) : 0.f;
            mlb = b + lane < i1 ? __ldcg(col_ml + (int64_t)(b + lane) * sd.ncols) : none;
            __syncwarp();  // the previous batch's weights are read
        }
        sh_w[warp][lane] = empty ? 0.f : ex2(mlb.x - M);
        __syncwarp();
#pragma unroll
        for (int j = 0; j < kBatch; ++j)
            if (b + j < i1) O += sh_w[warp][j] * xs[j];
    }
    if (halves == 2) {
        if (grp == 1) sh_o[dd] = O;
        __syncthreads();
        if (grp == 1) return;
        O += sh_o[dd];
    }
    const float o = L > 0.f ? O / L : 0.f;
    a.out[orow * kHeadDim + d] = __bfloat16_as_ushort(__float2bfloat16_rn(o));
}
static_assert(kCombThreads == kHeadDim, "a thread a dim (one group), or two groups of half the dims");

// The same merge for calls with many query columns and few splits (a prefill
// chunk: thousands of columns, a few splits each), where a CTA a column
// would spend its time being scheduled: a warp a (unit, column), eight
// columns a CTA, lane l summing dims 8l .. 8l+7.  Lane i holds split i's
// (m, l) (and i + 32's), so M and L reduce by shuffles as in decode_combine,
// and O sums the splits in order, loading eight splits' values at a time.
// comb_off counts these CTAs (set by launch_combine).
__global__ void __launch_bounds__(kCombThreads)
    combine_cols(const __grid_constant__ Common c, const DecodeArgs a) {
    constexpr int kB = 8;  // splits loaded at a time
    // the setup reads the launch parameters only: before the wait
    const int s = find_seq(c.n_seqs, blockIdx.x, [&](int t) { return c.seq[t].comb_off; });
    const SeqDev &sd = c.seq[s];
    const int ns = sd.nsplit;
    const int lane = threadIdx.x & 31;
    const int r = (blockIdx.x - sd.comb_off) * (kCombThreads / 32) + (threadIdx.x >> 5);
    if (r >= c.n_kv_heads * sd.ncols) return;  // past the stream's last column
    const int unit = r / sd.ncols, col = r - unit * sd.ncols;
    const float *part_acc = a.ws + sd.ws_off;
    const float2 *col_ml =
        reinterpret_cast<const float2 *>(part_acc + (int64_t)c.n_kv_heads * ns * sd.ncols * kHeadDim) +
        (int64_t)unit * ns * sd.ncols + col;
    const int64_t p0 = (int64_t)unit * ns * sd.ncols + col;  // split i at p0 + i * ncols
    const float *col_acc = part_acc + p0 * kHeadDim + 8 * lane;
    const int64_t stride = (int64_t)sd.ncols * kHeadDim;
    asm volatile("" ::"l"(col_acc), "l"(col_ml), "l"(stride), "r"(ns));
    pdl_wait();
    pdl_trigger();
    const float2 none = make_float2(-INFINITY, 0.f);
    const float2 ml0 = lane < ns ? __ldcg(col_ml + (int64_t)lane * sd.ncols) : none;
    const float2 ml1 = lane + 32 < ns ? __ldcg(col_ml + (int64_t)(lane + 32) * sd.ncols) : none;
    float M = fmaxf(ml0.x, ml1.x);
    for (int i = lane + 64; i < ns; i += 32) M = fmaxf(M, __ldcg(col_ml + (int64_t)i * sd.ncols).x);
#pragma unroll
    for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const bool empty = M == -INFINITY;
    const float w0 = empty ? 0.f : ex2(ml0.x - M), w1 = empty ? 0.f : ex2(ml1.x - M);
    float L = w0 * ml0.y + w1 * ml1.y;
    for (int i = lane + 64; i < ns; i += 32) {
        const float2 v = __ldcg(col_ml + (int64_t)i * sd.ncols);
        L += (empty ? 0.f : ex2(v.x - M)) * v.y;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    float O[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int b = 0; b < ns; b += kB) {
        float4 v[kB][2];
#pragma unroll
        for (int j = 0; j < kB; ++j)
            if (b + j < ns) {
                v[j][0] = __ldcg(reinterpret_cast<const float4 *>(col_acc + (b + j) * stride));
                v[j][1] = __ldcg(reinterpret_cast<const float4 *>(col_acc + (b + j) * stride) + 1);
            }
#pragma unroll
        for (int j = 0; j < kB; ++j) {
            const int i = b + j;
            if (i >= ns) break;
            float w;
            if (i < 64) w = __shfl_sync(0xffffffffu, i < 32 ? w0 : w1, i & 31);
            else w = empty ? 0.f : ex2(__ldcg(col_ml + (int64_t)i * sd.ncols).x - M);
            O[0] += w * v[j][0].x;
            O[1] += w * v[j][0].y;
            O[2] += w * v[j][0].z;
            O[3] += w * v[j][0].w;
            O[4] += w * v[j][1].x;
            O[5] += w * v[j][1].y;
            O[6] += w * v[j][1].z;
            O[7] += w * v[j][1].w;
        }
    }
    // o = O / L as in decode_combine, so both give the same bits for up to
    // 32 splits (the same sums in the same order)
    const bool any = L > 0.f;
    const float lz = any ? L : 1.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) O[k] = any ? O[k] / lz : 0.f;
    uint4 pk;
    pk.x = pack_bf16(O[0], O[1]);
    pk.y = pack_bf16(O[2], O[3]);
    pk.z = pack_bf16(O[4], O[5]);
    pk.w = pack_bf16(O[6], O[7]);
    Unit u;
    u.unit = unit;
    u.kvh = unit;
    *reinterpret_cast<uint4 *>(a.out + q_row<false>(c, sd, u, col) * kHeadDim + 8 * lane) = pk;
}

}  // namespace

// ---- fixed scratch for pkv_decode_static -------------------------------------
// A file-scope device array holds the split partials for callers that cannot
// allocate device memory.  Every GPU that loads the library holds it until the
// process exits.  In host code `g_static_scratch` is only a stand-in for the
// symbol; the device address is looked up per device below.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

int static_scratch(void **out) {
    static std::mutex mu;
    static void *ptrs[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PKV_ECUDA;
    std::lock_guard<std::mutex> g(mu);
    if (ptrs[dev] == nullptr) {
        void *p = nullptr;
        // with `dev` current: the array's address on this device
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr)
            return PKV_ECUDA;
        ptrs[dev] = p;
    }
    *out = ptrs[dev];
    return PKV_OK;
}

// Splits: a fixed number of keys per split, a multiple of the tile, at least
// the minimum, and enough splits for about two CTAs per SM from one stream.
int plan_decode(Common &c, bool sparse, int32_t k, int nsm, DecodePlan *plan) {
    int32_t items = 0, comb = 0;
    int64_t floats = 0;
    const int units = sparse ? c.n_q_heads : c.n_kv_heads;
    for (int s = 0; s < c.n_seqs; ++s) {
        SeqDev &d = c.seq[s];
        d.work_off = items;
        d.comb_off = comb;
        d.ws_off = floats;
        const int nkeys = sparse ? 4 * k : d.len;
        d.ncols = sparse ? 1 : d.n_new * c.group;
        if (d.ncols > kMaxCols) return PKV_EINVAL;
        if (d.n_new == 0 || nkeys == 0) {
            d.nsplit = 1;
            d.split_len = kTile;
            d.ncols = 0;
            continue;  // no queries: nothing to launch for this stream
        }
        const int max_splits = std::max(1, 2 * nsm / units);
        int sl = (nkeys + max_splits - 1) / max_splits;
        sl = (sl + kTile - 1) / kTile * kTile;
        sl = std::max(sl, sparse ? kMinSplitSparse : kMinSplitDense);
        sl = std::min(sl, kMaxSplitLen);
        const int ns = (nkeys + sl - 1) / sl;
        if (ns > kMaxSplits) return PKV_EINVAL;  // more than 2M keys in one stream
        d.nsplit = ns;
        d.split_len = sl;
        items += units * ns;
        if (ns > 1) {
            comb += units * d.ncols * comb_ctas(ns);
            floats += (int64_t)units * ns * d.ncols * (kHeadDim + 2);
            floats = (floats + 63) / 64 * 64;
        }
    }
    plan->total_items = items;
    plan->total_comb = comb;
    plan->ws_bytes = static_cast<size_t>(floats) * 4;
    return PKV_OK;
}

// Every kernel of a decode call asks for the largest shared-memory carveout:
// an SM configured for a small one (as a kernel using little shared memory
// would leave it) cannot take a partial CTA of the next call until it drains.
// The partial kernels' dynamic shared memory is set in the same pass.
static int set_carveout() {
    static std::atomic<uint64_t> done{0};
    return once_per_device(done, [] {
        const void *fns[] = {reinterpret_cast<const void *>(decode_combine<false>),
                             reinterpret_cast<const void *>(decode_combine<true>),
                             reinterpret_cast<const void *>(combine_cols),
                             reinterpret_cast<const void *>(decode_partial<false>),
                             reinterpret_cast<const void *>(decode_partial<true>)};
        for (const void *f : fns)
            if (cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared) != cudaSuccess)
                return PKV_ECUDA;
        for (int i = 3; i < 5; ++i)
            if (cudaFuncSetAttribute(fns[i], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kSmemBytes)) != cudaSuccess)
                return PKV_ECUDA;
        return PKV_OK;
    });
}

int launch_combine(const Common &c, const DecodePlan &plan, const uint16_t *q, uint16_t *out,
                   float *ws, cudaStream_t stream) {
    if (set_carveout() != PKV_OK) return PKV_ECUDA;
    DecodeArgs a{q, out, ws, nullptr, 0, nullptr, nullptr, nullptr};
    // many split columns with few splits each (a prefill chunk): a warp a column
    int nsm = 0;
    if (sm_count(&nsm) != PKV_OK) return PKV_ECUDA;
    int64_t cols = 0;
    int max_ns = 0;
    for (int s = 0; s < c.n_seqs; ++s)
        if (c.seq[s].nsplit > 1) {
            cols += (int64_t)c.n_kv_heads * c.seq[s].ncols;
            max_ns = std::max(max_ns, c.seq[s].nsplit);
        }
    if (cols >= 8 * (int64_t)nsm && max_ns <= 64) {
        Common cc = c;
        int32_t ctas = 0;
        for (int s = 0; s < cc.n_seqs; ++s) {
            cc.seq[s].comb_off = ctas;
            if (cc.seq[s].nsplit > 1)
                ctas += (c.n_kv_heads * cc.seq[s].ncols + kCombThreads / 32 - 1) / (kCombThreads / 32);
        }
        return launch_status(launch_pdl(combine_cols, ctas, kCombThreads, 0, stream, cc, a));
    }
    return launch_status(
        launch_pdl(decode_combine<false>, plan.total_comb, kCombThreads, 0, stream, c, a));
}

int launch_decode(const Common &c, const DecodePlan &plan, const DecodeMaps &maps, bool sparse,
                  const uint16_t *q, const int32_t *ids, int32_t k, uint16_t *out, float *ws,
                  const uint16_t *k_new, const uint16_t *v_new, const uint16_t *ik_new,
                  cudaStream_t stream) {
    DecodeArgs a{q, out, ws, ids, k, k_new, v_new, ik_new};
    // streams with no queries own no CTAs: give them an empty range
    Common cc = c;
    // units of more than 16 query columns take the tensor-core route instead
    for (int s = 0; s < c.n_seqs; ++s)
        if (c.seq[s].ncols > 16) return PKV_EINVAL;
    auto part = sparse ? decode_partial<true> : decode_partial<false>;
    auto comb = sparse ? decode_combine<true> : decode_combine<false>;
    if (set_carveout() != PKV_OK) return PKV_ECUDA;
    cudaError_t e = launch_pdl(part, plan.total_items, kThreads, kSmemBytes, stream, cc, maps, a);
    if (e != cudaSuccess) return PKV_ECUDA;
    if (plan.total_comb > 0) {
        e = launch_pdl(comb, plan.total_comb, kCombThreads, 0, stream, cc, a);
        if (e != cudaSuccess) return PKV_ECUDA;
    }
    return PKV_OK;
}

}  // namespace pkv
