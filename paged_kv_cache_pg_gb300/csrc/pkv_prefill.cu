// Chunked-prefill attention on the fifth-generation tensor cores (tcgen05).
//
// Rows: the (query, head) pairs of one KV head, 128 to an M-tile (16 queries
// x 8 heads for the pages' 16/2 heads).  A CTA takes one M-tile and one split
// of the keys and runs, per tile of 128 keys:
//   S = Q K^T  -> TMEM (128 lanes x 128 columns)               [MMA thread]
//   softmax of S with the causal mask, P = hi + lo bf16 parts   [8 warps]
//   O += P_hi V + P_lo V -> TMEM (128 lanes x 256 columns)      [MMA thread]
// or, in the fp16 V mode (long chunks; below), P in fp16 and O += P V on V
// rows converted to fp16 once a call by v16_gather.
// A tcgen05 MMA with M = 128 costs about the same for every N up to 128, so
// a 128-key S product takes the instructions a 64-key one did.  Q sits in
// TMEM (columns 0-127, bf16 pairs) and is the S product's A operand there;
// that leaves shared memory for P (hi and lo, 64 KB) and one ring of five
// 32 KB slots (P in fp16, 32 KB, and six slots in the fp16 V mode): a K slot
// holds the tile's keys over 128 of the dims, a V slot 64 of its keys over
// all dims.  The softmax takes two threads a row (TMEM lane), each on 64 of
// the tile's keys and 128 of O's columns; the pair agrees on the row maximum
// through shared memory.  S has one TMEM buffer: the next S product starts
// once the softmax threads have read S, and P has one buffer, which the
// softmax fills once the previous tile's PV product is done.
// Four producer warps, one for each slot kind (K over the first or second
// dims, V over the first or second keys), fill the ring in the order the
// MMAs take the slots.  In the fp16 V mode a V slot is one 3D copy of the
// converted rows (contiguous: no page lookups).  Otherwise the producers
// look a tile's rows up before its slots are free: a
// cached tile inside one page needs one page lookup and comes by one 3D TMA
// copy a slot (pages of a multiple of 128 positions), a cached tile in pages
// of a multiple of 16 needs its eight 16-row run starts and comes by 2D
// copies of the runs (each copy costs the issuing thread about 40 ns,
// whatever its size), and any other tile (a ragged tail, new rows, other page
// sizes) comes key by key by cp.async from one row lookup per key, fenced by
// the copying threads before the tensor cores read it.  The max of a row is
// rescaled lazily: O in TMEM is corrected only when the running max grows by
// more than 2^8.  Split partials use the decode layout and its combine
// kernel.
#include <algorithm>
#include <climits>

#include "pkv_dev.cuh"

namespace pkv {
namespace {

constexpr int kM = 128;              // rows of an M-tile
constexpr int kN = 128;              // keys a tile
constexpr int kSoftWarps = 8;        // two threads a row, each on 64 keys of a tile
constexpr int kWarpMma = 9;         // warps 8 and 10-12 produce: K and V slots of dims or keys 0..,
constexpr int kPThreads = 416;       // then of the second half; warps 0-7 softmax
constexpr int kSoftThreads = kSoftWarps * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kQCol = 0;        // Q: 256 dims as bf16 pairs
constexpr uint32_t kSCol = 128;      // S: 128 keys
constexpr uint32_t kOCol = 256;      // O: 256 dims
constexpr int kKRegion = kN * 128;   // one 64-dim region of 128 K rows
constexpr int kVRegion = 64 * 128;   // one 64-dim region of 64 V rows
constexpr int kSlotBytes = 2 * kKRegion;  // a K slot (the tile's keys over 128 dims) or
                                          // a V slot (64 of its keys over 256 dims)
static_assert(kSlotBytes == 4 * kVRegion, "K and V slots share one ring");
constexpr int kPRegion = kM * 128;   // 64 keys of the 128 P rows
constexpr int kPPart = 2 * kPRegion; // P (or its hi or lo part): the tile's 128 keys
constexpr int kOffP = 0;             // P, or P hi then P lo

// Shared-memory layout of each V mode: P, the ring (taken in the MMAs'
// order), the row-maximum exchange, the barriers.  The fp16 V mode's P is
// one part, and the 32 KB the lo part takes in the bf16 mode is a sixth
// ring slot: a slot is refilled six places after it was taken, which
// covers the about 2 us a slot's copy takes to land at the fp16 mode's
// pace (five slots left the MMA thread waiting about 0.3 us a tile).
template <bool kV16>
struct PLayout {
    static constexpr int slots = kV16 ? 6 : 5;
    static constexpr int off_ring = kOffP + (kV16 ? 1 : 2) * kPPart;
    static constexpr int off_red = off_ring + slots * kSlotBytes;  // [tile parity][half][row] floats
    static constexpr int off_bar = off_red + 2 * 2 * kM * 4;
    // barriers: a pair for each ring slot, one for each single buffer
    static constexpr int bar_full = 0, bar_empty = slots;
    static constexpr int bar_sfull = 2 * slots, bar_sempty = bar_sfull + 1, bar_pfull = bar_sfull + 2;
    static constexpr int bar_odone = bar_sfull + 3, bar_qfull = bar_sfull + 4, bar_red = bar_sfull + 5;
    static constexpr int num_bars = bar_red + 1;
    // no alignment slack: the dynamic shared memory is declared 1024-byte
    // aligned (checked at entry), and the ring leaves no room for it
    static constexpr size_t smem = off_bar + num_bars * 8 + 16;
    static_assert(smem <= 232448, "prefill shared memory above the 227 KB a CTA may hold");
};
constexpr float kScaleLog2 = 0.0625f * 1.4426950408889634f;  // log2(e) / sqrt(256)
constexpr float kRescale = 8.f;  // rescale O when the max grows by more than 2^8

// Instruction descriptor, kind::f16: D float32, A and B both bf16 or both
// fp16, A K-major, B K-major (S = Q K^T) or MN-major (O += P V), M = 128.
__host__ __device__ constexpr uint32_t mma_idesc(int n, bool b_mn_major, bool f16 = false) {
    return (1u << 4) | ((f16 ? 0u : 1u) << 7) | ((f16 ? 0u : 1u) << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kM >> 4) << 24);
}

// Two floats to an fp16 pair, round to nearest even, lo in the low half.
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    uint32_t h;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(hi), "f"(lo));
    return h;
}

// A bf16 pair to an fp16 pair (each bf16 value is exactly a float): exact
// for magnitudes 2^-14 to 65,280, rounded to fp16's 2^-24 grid below, and
// infinite above 65,504.
__device__ __forceinline__ uint32_t f16_of_bf16(uint32_t w) {
    return pack_f16(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// The fp16 V mode.  A launch whose streams each have a chunk of more than
// 32 queries and at least eight M-tiles a KV head reads V rows converted
// once a call by v16_gather into the workspace (each KV head's rows padded
// with zeros to a multiple of the key tile) instead of the cache's bf16
// rows: the PV product runs in fp16 on one P part, half the MMAs of the
// bf16 hi and lo parts (A and B of one MMA share a type, and P needs more
// than bf16's 8 significant bits).  The conversion costs a read and a write
// of the V rows; each M-tile's CTA would otherwise convert every V tile
// again.  Decode calls (at most 32 new rows a stream) never take it.
constexpr int kV16MinTiles = 8;
constexpr int kV16MinNew = 33;
__host__ __device__ inline int v16_stride(int len) { return (len + kN - 1) / kN * kN; }
// Rows of the launch's converted V (0: the launch reads bf16 V).
inline int64_t v16_rows(const Common &c) {
    int64_t rows = 0;
    for (int s = 0; s < c.n_seqs; ++s) {
        const SeqDev &d = c.seq[s];
        if (d.ncols == 0) continue;
        if (d.n_new < kV16MinNew || (d.ncols + kM - 1) / kM < kV16MinTiles) return 0;
        rows += (int64_t)c.n_kv_heads * v16_stride(d.len);
    }
    return rows <= ((int64_t)1 << 30) ? rows : 0;
}

// Shared-memory matrix descriptor, 128-byte swizzle: start address, leading
// byte offset (MN-major: between 64-element blocks), stride byte offset
// (between 8-row groups), the fixed version bits.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The same with A from TMEM (the TS form): a_tmem is the address of A's
// first column, 16 bf16 elements of each row in 8 consecutive 32-bit columns.
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 32 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
        "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 64 consecutive 32-bit TMEM columns of this thread's lane: one load and one
// wait for a whole S tile.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

struct PrefillArgs {
    const uint16_t *q;
    uint16_t *out;
    float *ws;
    // a decode call's new rows [token][KV head][256] (and [token][Di]), read
    // from here and stored into their pages by the kernel, or null
    const uint16_t *k_new, *v_new, *ik_new;
    // the fp16 V mode: the converted rows (in the workspace), their map, and
    // each stream's first row there (KV head 0; -1: the stream reads bf16 V)
    uint16_t *v16;
    int32_t v16_map;
    int32_t v16_row[PKV_MAX_SEQS];
};

// Byte offset of 16-byte chunk c (0..31) of row r in a 128-byte-swizzled
// operand made of 64-dim regions of `region` bytes.
__device__ __forceinline__ uint32_t swz128(int region, int r, int c) {
    return (c >> 3) * region + r * 128 + ((((c & 7) ^ (r & 7))) << 4);
}

template <bool kV16>
__global__ void __launch_bounds__(kPThreads, 1)
    prefill_partial(const __grid_constant__ Common c, const __grid_constant__ DecodeMaps maps,
                    const __grid_constant__ PrefillArgs a) {
    // the 128-byte swizzle of the TMA copies and the MMA operands repeats
    // every 1024 bytes from a 1024-byte boundary
    extern __shared__ __align__(1024) uint8_t smem[];
    using L = PLayout<kV16>;
    constexpr int kSlots = L::slots, kOffRing = L::off_ring, kOffRed = L::off_red;
    constexpr int kBarFull = L::bar_full, kBarEmpty = L::bar_empty, kBarSFull = L::bar_sfull;
    constexpr int kBarSEmpty = L::bar_sempty, kBarPFull = L::bar_pfull, kBarODone = L::bar_odone;
    constexpr int kBarQFull = L::bar_qfull, kBarRed = L::bar_red;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::off_bar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + L::num_bars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    {
        // the address as the hardware gives it (an asm result the compiler
        // cannot fold from the declared alignment)
        uint32_t base;
        asm volatile("mov.u32 %0, %1;" : "=r"(base) : "r"(smem_u32(smem)));
        if (base & 1023u) {  // uniform: every thread returns before any barrier
            if (tid == 0 && c.status) atomicOr(c.status, PKV_DEV_SMEM);
            return;
        }
    }
    const int H = c.n_kv_heads, G = c.group;
    // the stream whose block of work items holds this CTA (the blocks are
    // laid out longest CTA first, not in stream order)
    int s = 0;
    for (int t = 0; t < c.n_seqs; ++t) {
        const SeqDev &st = c.seq[t];
        const int items = H * ((st.ncols + kM - 1) / kM) * st.nsplit;
        if (st.ncols > 0 && (int)blockIdx.x >= st.work_off && (int)blockIdx.x < st.work_off + items) s = t;
    }
    const SeqDev &sd = c.seq[s];
    const int mtiles = (sd.ncols + kM - 1) / kM;
    // consecutive CTAs share a (KV head, split): the M-tiles that read the
    // same key range run in the same wave and find its tiles in L2.  The
    // M-tiles with the most keys (the last ones of a causal chunk) come
    // first, so that in a grid of several waves the SMs freed first take the
    // shortest CTAs of the last one (the serving mix's 2,048-query lane, 256
    // CTAs: 488 us against 506 in ascending order).  The order changes which
    // SM runs a CTA, never its result.
    const int item = blockIdx.x - sd.work_off;
    const int kvh = item / (mtiles * sd.nsplit);
    const int split = (item / mtiles) % sd.nsplit;
    const int mt = mtiles - 1 - item % mtiles;
    const int col0 = mt * kM;
    const int rows = min(kM, sd.ncols - col0);
    const int qbase = sd.len - sd.n_new;
    const int last_q = qbase + (col0 + rows - 1) / G;  // position of the tile's last query
    const int key0 = split * sd.split_len;
    const int key1 = min(min(sd.len, key0 + sd.split_len), last_q + 1);
    const int ntiles = key1 > key0 ? (key1 - key0 + kN - 1) / kN : 0;
    constexpr bool v16 = kV16;  // the PV product in fp16 on converted V rows

    if (tid == 0) {
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(&bars[kBarFull + i], 1);
            mbar_init(&bars[kBarEmpty + i], 1);
        }
        mbar_init(&bars[kBarSFull], 1);
        mbar_init(&bars[kBarSEmpty], kSoftThreads);
        mbar_init(&bars[kBarPFull], kSoftThreads);
        mbar_init(&bars[kBarODone], 1);
        mbar_init(&bars[kBarQFull], kSoftThreads);
        mbar_init(&bars[kBarRed], kSoftThreads);
        *abort_flag = 0;
        fence_mbar_init();
    }
    // tcgen05 alloc, dealloc, ld and st are warp-collective (.sync.aligned):
    // every one below follows a __syncwarp, because a CTA barrier does not
    // reconverge a warp whose lanes took different paths before it
    if (warp == kWarpMma) {
        __syncwarp();
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t sbase = smem_u32(smem);
    // the next kernel (the split combine, or the next call) may start once
    // every CTA is running: it waits for this grid before reading anything
    // this grid writes, except cached rows more than 32 positions below its
    // own new tokens, which the rows stored here (a decode call's at most 32
    // new rows a stream) are not
    if (tid == 0) pdl_trigger();

    if (warp < kSoftWarps) {
        // ------- softmax: row r (TMEM lane r) by two threads, keys 64 hf .. 64 hf + 63 of a tile -------
        pdl_wait();
        const int r = lane + 32 * (warp & 3);
        const int hf = warp >> 2;
        const int col = col0 + r;
        const bool row_ok = r < rows;
        const int j = row_ok ? col / G : 0;
        // rows past the M-tile's end take no mask: their Q rows are zero, so
        // their scores are finite, and their outputs are never written
        const int qpos = row_ok ? qbase + j : INT_MAX;
        const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        float *const red = reinterpret_cast<float *>(smem + kOffRed);
        // Q dims 128 hf .. 128 hf + 127 into TMEM columns 64 hf .. 64 hf + 63 (bf16 pairs)
        {
            const uint16_t *src =
                a.q + (((int64_t)sd.tok_off + j) * c.n_q_heads + kvh * G + (col - j * G)) * kHeadDim + 128 * hf;
#pragma unroll 1
            for (int h32 = 0; h32 < 2; ++h32) {
                uint32_t qv[32];
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    const uint4 v = row_ok ? __ldg(reinterpret_cast<const uint4 *>(src + 64 * h32 + 2 * i))
                                           : make_uint4(0, 0, 0, 0);
                    qv[i] = v.x;
                    qv[i + 1] = v.y;
                    qv[i + 2] = v.z;
                    qv[i + 3] = v.w;
                }
                __syncwarp();
                tmem_st32(lane_base + kQCol + 64 * hf + 32 * h32, qv);
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            tc_fence_before();
            mbar_arrive(&bars[kBarQFull]);
        }
        float m_used = -INFINITY, l = 0.f;
        uint8_t *const p_hi = smem + kOffP + hf * kPRegion, *const p_lo = p_hi + kPPart;
        for (int n = 0; n < ntiles; ++n) {
            // every exit is warp-uniform: the TMEM loads below are .sync.aligned
            if (!__all_sync(0xffffffffu, mbar_wait(&bars[kBarSFull], n & 1, c.status))) {
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            uint32_t sv[64];
            tmem_ld64(lane_base + kSCol + 64 * hf, sv);
            tc_fence_before();
            mbar_arrive(&bars[kBarSEmpty]);
            const int kt = key0 + n * kN + 64 * hf;  // this thread's first key
            // raw scores; the causal and split bounds cut into a tile only near
            // the diagonal and at the split's end
            float x[64];
            if (__all_sync(0xffffffffu, kt + 64 <= key1 && kt + 63 <= qpos)) {
#pragma unroll
                for (int i = 0; i < 64; ++i) x[i] = __uint_as_float(sv[i]);
            } else {
#pragma unroll
                for (int i = 0; i < 64; ++i) {
                    const int kp = kt + i;
                    x[i] = (kp < key1 && kp <= qpos) ? __uint_as_float(sv[i]) : -INFINITY;
                }
            }
            // this half's max as eight interleaved chains (exact in any order),
            // then the row's from the partner thread
            float m8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) m8[i] = x[i];
#pragma unroll
            for (int i = 8; i < 64; ++i) m8[i & 7] = fmaxf(m8[i & 7], x[i]);
            const float lmx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                    fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
            red[((n & 1) * 2 + hf) * kM + r] = lmx;
            mbar_arrive(&bars[kBarRed]);
            if (!__all_sync(0xffffffffu, mbar_wait(&bars[kBarRed], n & 1, c.status))) {
                *abort_flag = 1;
                break;
            }
            // in log2 units; -inf when the whole row of the tile is masked
            const float mx = fmaxf(lmx, red[((n & 1) * 2 + (hf ^ 1)) * kM + r]) * kScaleLog2;
            // both threads of a row see the same maximum, so they decide alike
            const bool grow = m_used != -INFINITY && mx > m_used + kRescale;
            if (__any_sync(0xffffffffu, grow)) {
                // correct this thread's half of O: the previous tile's products
                // must be in it first
                if (n > 0 && !__all_sync(0xffffffffu, mbar_wait(&bars[kBarODone], (n - 1) & 1, c.status))) {
                    *abort_flag = 1;
                    break;
                }
                tc_fence_after();
                const float m_new = fmaxf(m_used, mx);
                const float alpha = m_used == -INFINITY ? 0.f : ex2(m_used - m_new);
#pragma unroll 1
                for (int ch = 0; ch < 4; ++ch) {
                    uint32_t o[32];
                    tmem_ld32(lane_base + kOCol + 128 * hf + ch * 32, o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st32(lane_base + kOCol + 128 * hf + ch * 32, o);
                }
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                l *= alpha;
                m_used = m_new;
            } else if (m_used == -INFINITY) {
                m_used = mx;  // nothing accumulated yet: O is still zero
            }
            // p = 2^(s * scale - m); a masked score is -inf and gives 0 (the
            // offset is 0 while every score so far was masked)
            const float m_off = m_used == -INFINITY ? 0.f : m_used;
            float ps[4] = {0.f, 0.f, 0.f, 0.f};  // this half's sum as four chains
            uint32_t hi[32], lo[32];
            if (v16) {
                // P in fp16: 11 significant bits (weights at most 2^8 with the
                // lazy rescale; below 2^-14 on fp16's 2^-24 grid)
#pragma unroll
                for (int i = 0; i < 64; i += 2) {
                    const float p0 = ex2(fmaf(x[i], kScaleLog2, -m_off));
                    const float p1 = ex2(fmaf(x[i + 1], kScaleLog2, -m_off));
                    ps[(i >> 1) & 3] += p0 + p1;
                    hi[i / 2] = pack_f16(p0, p1);
                }
            } else {
#pragma unroll
                for (int i = 0; i < 64; i += 2) {
                    const float p0 = ex2(fmaf(x[i], kScaleLog2, -m_off));
                    const float p1 = ex2(fmaf(x[i + 1], kScaleLog2, -m_off));
                    ps[(i >> 1) & 3] += p0 + p1;
                    // p = hi + lo: hi is p's top 16 bits (exact), lo the top 16
                    // bits of the exact remainder, so hi + lo is p to 2^-15
                    // relative; bit selects keep the split off the conversion pipe
                    const uint32_t u0 = __float_as_uint(p0), u1 = __float_as_uint(p1);
                    hi[i / 2] = __byte_perm(u0, u1, 0x7632);
                    const float r0 = p0 - __uint_as_float(u0 & 0xffff0000u);
                    const float r1 = p1 - __uint_as_float(u1 & 0xffff0000u);
                    lo[i / 2] = __byte_perm(__float_as_uint(r0), __float_as_uint(r1), 0x7632);
                }
            }
            l += (ps[0] + ps[1]) + (ps[2] + ps[3]);
            // the P rows are free once the last tile's products are done
            if (n > 0 && !__all_sync(0xffffffffu, mbar_wait(&bars[kBarODone], (n - 1) & 1, c.status))) {
                *abort_flag = 1;
                break;
            }
            // row r of this half's P region: 64 keys = 128 bytes = chunks 0 .. 7
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                const uint32_t off = r * 128 + (((ch ^ (r & 7))) << 4);
                *reinterpret_cast<uint4 *>(p_hi + off) =
                    make_uint4(hi[4 * ch], hi[4 * ch + 1], hi[4 * ch + 2], hi[4 * ch + 3]);
                if (!v16)
                    *reinterpret_cast<uint4 *>(p_lo + off) =
                        make_uint4(lo[4 * ch], lo[4 * ch + 1], lo[4 * ch + 2], lo[4 * ch + 3]);
            }
            fence_async_smem();
            tc_fence_before();
            mbar_arrive(&bars[kBarPFull]);
        }
        // ---------------- epilogue ----------------
        bool ok = __all_sync(0xffffffffu, !*abort_flag);
        if (ok && ntiles > 0 &&
            !__all_sync(0xffffffffu, mbar_wait(&bars[kBarODone], (ntiles - 1) & 1, c.status))) {
            *abort_flag = 1;
            ok = false;
        }
        // the row's sum: this thread's keys and its partner's
        if (ok) {
            red[((ntiles & 1) * 2 + hf) * kM + r] = l;
            mbar_arrive(&bars[kBarRed]);
            if (!__all_sync(0xffffffffu, mbar_wait(&bars[kBarRed], ntiles & 1, c.status))) {
                *abort_flag = 1;
                ok = false;
            } else {
                l += red[((ntiles & 1) * 2 + (hf ^ 1)) * kM + r];
            }
        }
        tc_fence_after();
        if (ok) {
            const bool single = sd.nsplit == 1;
            float *part_acc = a.ws + sd.ws_off;
            float *part_ml = part_acc + (int64_t)H * sd.nsplit * sd.ncols * kHeadDim;
            const int64_t prow = ((int64_t)kvh * sd.nsplit + split) * sd.ncols + col;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            uint16_t *orow = a.out + (((int64_t)sd.tok_off + j) * c.n_q_heads + kvh * G + (col - j * G)) * kHeadDim;
            bool finite = true;  // a V entry beyond fp16's range makes O infinite or NaN
#pragma unroll 1
            for (int ch = 0; ch < 4; ++ch) {
                const int d0 = 128 * hf + 32 * ch;  // the chunk's first dim
                uint32_t o[32];
                __syncwarp();  // rows past the tile's end skipped the stores below
                if (ntiles > 0) {
                    tmem_ld32(lane_base + kOCol + d0, o);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0u;
                }
                if (!row_ok) continue;
#pragma unroll
                for (int i = 0; i < 32; ++i) finite &= fabsf(__uint_as_float(o[i])) <= 3.402823466e38f;
                if (single) {
#pragma unroll
                    for (int i = 0; i < 32; i += 8) {
                        uint4 v;
                        v.x = pack_bf16(__uint_as_float(o[i]) * inv, __uint_as_float(o[i + 1]) * inv);
                        v.y = pack_bf16(__uint_as_float(o[i + 2]) * inv, __uint_as_float(o[i + 3]) * inv);
                        v.z = pack_bf16(__uint_as_float(o[i + 4]) * inv, __uint_as_float(o[i + 5]) * inv);
                        v.w = pack_bf16(__uint_as_float(o[i + 6]) * inv, __uint_as_float(o[i + 7]) * inv);
                        *reinterpret_cast<uint4 *>(orow + d0 + i) = v;
                    }
                } else {
                    float *dst = part_acc + prow * kHeadDim + d0;
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        *reinterpret_cast<float4 *>(dst + i) =
                            make_float4(__uint_as_float(o[i]), __uint_as_float(o[i + 1]),
                                        __uint_as_float(o[i + 2]), __uint_as_float(o[i + 3]));
                }
            }
            if (row_ok && !single && hf == 0) {
                part_ml[prow * 2 + 0] = m_used;
                part_ml[prow * 2 + 1] = l;
            }
            if (!finite && c.status) atomicOr(c.status, PKV_DEV_RANGE);
        }
    } else if (warp >= kSoftWarps && warp != kWarpMma) {
        // ------- producers: K slots (warps 8, 11) and V slots (10, 12) of one ring -------
        // The MMAs take the slots in the order K(0) over dims 0-127 and
        // 128-255, then per tile m >= 1: K(m) halves, V(m-1) keys 0-63 and
        // 64-127 (the PV product of the tile before), and last V(ntiles-1).
        // Each producer takes one half (warps 8 and 10 the first, 11 and 12
        // the second) and knows its slots' places in that order, so the four
        // fill the ring side by side; a slot is refilled five (bf16 V) or six
        // (fp16 V) places after it was taken.
        pdl_wait();  // the chunk's rows are stored by the previous kernel
        const bool is_v = warp == 10 || warp == 12;
        const int hh = warp >= 11;  // which half of the tile's dims (K) or keys (V)
        // the stream's fields in registers: read from the launch parameters
        // with a per-CTA index, each costs a constant-cache round trip, and
        // the issue loop would reread them every slot
        const int ptok = sd.ptok, n_pages = sd.n_pages, n_table = sd.n_table, tok_off = sd.tok_off;
        const int32_t *const table = sd.table;
        const int64_t ps = sd.ps, layer_row = sd.layer_row;
        const uint16_t *const layer_base = sd.layer_base;
        const void *const map = sd.tma >= 0 ? &maps.map[sd.tma] : nullptr;          // 16 x 64 boxes
        const void *const map_k = sd.tma_k >= 0 ? &maps.map[sd.tma_k] : nullptr;    // a K slot
        const void *const map_v = sd.tma_v >= 0 ? &maps.map[sd.tma_v] : nullptr;    // a V slot
        const void *const map_t = is_v ? map_v : map_k;
        // fp16 V mode: each V slot is one copy of converted rows
        const bool v16v = v16 && is_v;
        const void *const map16 = v16v ? &maps.map[a.v16_map] : nullptr;
        const int y16 = v16v ? a.v16_row[s] + kvh * v16_stride(sd.len) : 0;
        const uint64_t pol = policy_evict_normal();  // every M-tile of the head reads these rows
        // V rows sit H * ptok rows after the K rows of the same page
        const int64_t gap = is_v ? (int64_t)H * ptok * kHeadDim : 0;
        const int vrows = is_v ? H * ptok : 0;
        const bool fuse = a.k_new != nullptr;
        const uint16_t *const new_rows = is_v ? a.v_new : a.k_new;
        const int nk = is_v ? 64 : kN;       // keys a slot
        const int region = is_v ? kVRegion : kKRegion;
        // page ids in registers: lane i holds pages win + i (cur) and
        // win + 32 + i (nxt); the window slides by 32 once a tile starts past
        // its first half, so the next half is loading long before it is read
        // and no table read waits in the issue loop (a tile of 128 keys spans
        // at most 33 pages, so its pages always lie in the 64-page window)
        auto page_id = [&](int p) -> int { return (table && p < n_table) ? __ldg(table + p) : 0; };
        int win = table ? key0 / ptok : 0;
        int cur = page_id(win + lane), nxt = page_id(win + 32 + lane);
        bool ok = true;
        for (int m = 0; m < ntiles && ok; ++m) {
            const int kt = key0 + m * kN;
            if (table) {
                const int first = min(kt, key1 - 1) / ptok;  // the tile's lowest page
                while (first >= win + 32) {
                    win += 32;
                    cur = nxt;
                    nxt = page_id(win + 32 + lane);
                }
            }
            // A whole cached tile in one page (pages of a multiple of 128)
            // needs only its first row (yt, the map row of its first K row);
            // a whole cached tile in pages of a multiple of 16 only the first
            // rows of its eight 16-row runs (lane i < 8: yrun, the map row of
            // run i, V's for the V producer).  Any other tile: the row offsets
            // of this lane's keys kt + 32 g + lane (clamped into the split),
            // and which of them had a bad page id.  The lookups come before
            // the slots' waits.
            const bool cached = kt + kN <= key1 && !(fuse && kt + kN > qbase);
            int yt = -1, yrun = -1;
            int64_t r[4] = {0, 0, 0, 0};
            uint32_t bm = 0;
            if (v16v) {
                // no lookups: the converted rows are contiguous
            } else if (cached && map != nullptr && !(map_k != nullptr && map_v != nullptr)) {
                const int key = kt + 16 * (lane & 7);
                int row = key;
                int64_t pg = 0;
                if (table) {
                    const int page = key / ptok;
                    row = key - page * ptok;
                    const int idx = page - win;  // 0 .. 63
                    const int a0 = __shfl_sync(0xffffffffu, cur, idx & 31);
                    const int a1 = __shfl_sync(0xffffffffu, nxt, idx & 31);
                    const int id = idx < 32 ? a0 : a1;
                    if (static_cast<uint32_t>(id) < static_cast<uint32_t>(n_pages)) {
                        pg = (int64_t)id * ps;
                    } else if (lane < 8 && !is_v && c.status) {
                        atomicOr(c.status, PKV_DEV_BAD_PAGE);
                    }
                }
                yrun = static_cast<int>(layer_row + (pg + off_k(ptok, kvh, row) + gap) / kHeadDim);
            } else if (cached && map_k != nullptr && map_v != nullptr) {
                int row = kt;
                int64_t pg = 0;
                if (table) {
                    const int page = kt / ptok;
                    row = kt - page * ptok;
                    const int id = __shfl_sync(0xffffffffu, cur, (page - win) & 31);  // page - win < 32
                    if (static_cast<uint32_t>(id) < static_cast<uint32_t>(n_pages)) {
                        pg = (int64_t)id * ps;
                    } else if (lane == 0 && !is_v && c.status) {
                        atomicOr(c.status, PKV_DEV_BAD_PAGE);
                    }
                }
                yt = static_cast<int>(layer_row + (pg + off_k(ptok, kvh, row)) / kHeadDim);
            } else {
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    if (is_v && (g >> 1) != hh) continue;  // a V slot holds two of the groups
                    const int key = min(kt + 32 * g + lane, key1 - 1);
                    int row = key;
                    int64_t pg = 0;
                    if (table) {
                        const int page = key / ptok;
                        row = key - page * ptok;
                        const int idx = page - win;  // 0 .. 63
                        const int a0 = __shfl_sync(0xffffffffu, cur, idx & 31);
                        const int a1 = __shfl_sync(0xffffffffu, nxt, idx & 31);
                        const int id = idx < 32 ? a0 : a1;
                        if (static_cast<uint32_t>(id) < static_cast<uint32_t>(n_pages)) {
                            pg = (int64_t)id * ps;
                        } else {
                            bm |= 1u << g;
                            if (c.status && !is_v) atomicOr(c.status, PKV_DEV_BAD_PAGE);
                        }
                    }
                    r[g] = pg + off_k(ptok, kvh, row) + gap;
                }
            }
            {
                // the slot's place in the MMAs' order
                const uint32_t q = is_v ? (m + 1 < ntiles ? 4 * m + 4 + hh : 4 * m + 2 + hh)
                                        : (m == 0 ? hh : 4 * m - 2 + hh);
                const int slot = q % kSlots;
                uint64_t *const full = &bars[kBarFull + slot];
                uint8_t *const dst = smem + kOffRing + slot * kSlotBytes;
                if (__any_sync(0xffffffffu, *abort_flag) ||
                    (q >= kSlots && !__all_sync(0xffffffffu, mbar_wait(&bars[kBarEmpty + slot],
                                                                         ((q / kSlots) - 1) & 1, c.status)))) {
                    *abort_flag = 1;
                    ok = false;
                    break;
                }
                if (v16v) {
                    if (lane == 0) {
                        mbar_arrive_expect_tx(full, kSlotBytes);
                        tma_load_3d(dst, map16, 0, y16 + kt + 64 * hh, 0, full, pol);
                    }
                    continue;
                }
                if (yt >= 0) {
                    // the tile lies in one page: the slot is one copy
                    if (lane == 0) {
                        mbar_arrive_expect_tx(full, kSlotBytes);
                        if (is_v)
                            tma_load_3d(dst, map_v, 0, yt + vrows + 64 * hh, 0, full, pol);
                        else
                            tma_load_3d(dst, map_k, 0, yt, 2 * hh, full, pol);
                    }
                    continue;
                }
                if (yrun >= 0) {  // uniform: every lane looked a run up
                    // 16-row page runs of a cached tile: a V slot in one page is
                    // one copy; else 8 (K) or 4 (V) runs of two or four chunks
                    const int rn0 = is_v ? 4 * hh : 0;
                    const int y0 = __shfl_sync(0xffffffffu, yrun, rn0);
                    if (is_v && map_v != nullptr) {
                        if (lane == 0) {
                            mbar_arrive_expect_tx(full, kSlotBytes);
                            tma_load_3d(dst, map_v, 0, y0, 0, full, pol);
                        }
                        continue;
                    }
                    int yr[8];
#pragma unroll
                    for (int rn = 0; rn < 8; ++rn) yr[rn] = __shfl_sync(0xffffffffu, yrun, (rn0 + rn) & 7);
                    if (lane == 0) {
                        mbar_arrive_expect_tx(full, kSlotBytes);
#pragma unroll
                        for (int rn = 0; rn < 8; ++rn) {
                            if (rn * 16 >= nk) break;
#pragma unroll
                            for (int ch = 0; ch < 4; ++ch) {
                                if (!is_v && ch >= 2) break;
                                tma_load_2d(dst + ch * region + rn * 2048, map, 64 * ((is_v ? 0 : 2 * hh) + ch),
                                            yr[rn], full, pol);
                            }
                        }
                    }
                    continue;
                }
                // the slot's keys: K, the tile's 128 (four groups of 32) over
                // dims 128 hh ..; V, keys 64 hh .. (two groups) over all dims
                const int kb = kt + (is_v ? 64 * hh : 0);
                const int g0 = is_v ? 2 * hh : 0;  // the slot's first key group
                const int64_t ra = is_v ? (hh ? r[2] : r[0]) : r[0];
                const int64_t rb = is_v ? (hh ? r[3] : r[1]) : r[1];
                const bool fresh = fuse && min(kb + nk, key1) > qbase;
                const bool whole = kb + nk <= key1 && !fresh;
                const int chunk0 = is_v ? 0 : 2 * hh;  // first 64-dim chunk of the slot
                if (whole && map_t != nullptr) {
                    // the slot's keys lie in one page: one copy
                    const int y0 = static_cast<int>(layer_row + shfl64(ra, 0) / kHeadDim);
                    if (lane == 0) {
                        mbar_arrive_expect_tx(full, kSlotBytes);
                        tma_load_3d(dst, map_t, 0, y0, chunk0, full, pol);
                    }
                } else if (whole && map != nullptr) {
                    // 16-row page runs: 8 (K) or 4 (V), two or four chunks each
                    int yr[8];
#pragma unroll
                    for (int rn = 0; rn < 8; ++rn) {
                        const int gg = rn >> 1;
                        const int64_t rg = is_v ? (gg == 0 ? ra : rb) : (gg == 0 ? r[0] : gg == 1 ? r[1] : gg == 2 ? r[2] : r[3]);
                        yr[rn] = static_cast<int>(layer_row + shfl64(rg, (rn & 1) * 16) / kHeadDim);
                    }
                    if (lane == 0) {
                        mbar_arrive_expect_tx(full, kSlotBytes);
#pragma unroll
                        for (int rn = 0; rn < 8; ++rn) {
                            if (rn * 16 >= nk) break;
#pragma unroll
                            for (int ch = 0; ch < 4; ++ch) {
                                if (!is_v && ch >= 2) break;
                                tma_load_2d(dst + ch * region + rn * 2048, map, 64 * (chunk0 + ch), yr[rn],
                                            full, pol);
                            }
                        }
                    }
                } else {
                    // key by key: each row's 16-byte chunks of the slot's dims
                    int64_t sp[4];
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        const int gk = g0 + g;  // key group within the tile
                        const int key = min(kt + 32 * gk + lane, key1 - 1);
                        const int64_t rg = gk == 0 ? r[0] : gk == 1 ? r[1] : gk == 2 ? r[2] : r[3];
                        const uint16_t *src = layer_base + rg;
                        if (fresh && key >= qbase)
                            src = new_rows + (((int64_t)tok_off + (key - qbase)) * H + kvh) * kHeadDim;
                        sp[g] = reinterpret_cast<int64_t>(src + 64 * chunk0);
                    }
                    if (is_v) {
                        // 64 rows of 32 chunks: a row a pass, a chunk a lane
#pragma unroll
                        for (int g = 0; g < 2; ++g)
#pragma unroll 8
                            for (int rr = 0; rr < 32; ++rr)
                                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                                                 smem_u32(dst + swz128(kVRegion, 32 * g + rr, lane))),
                                             "l"(reinterpret_cast<const uint16_t *>(shfl64(sp[g], rr)) + lane * 8)
                                             : "memory");
                    } else {
                        // 128 rows of 16 chunks: two rows a pass, a chunk a lane
                        const int hl = lane >> 4, cl = lane & 15;
#pragma unroll
                        for (int g = 0; g < 4; ++g)
#pragma unroll 4
                            for (int rr = 0; rr < 32; rr += 2)
                                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                                                 smem_u32(dst + swz128(kKRegion, 32 * g + rr + hl, cl))),
                                             "l"(reinterpret_cast<const uint16_t *>(shfl64(sp[g], rr + hl)) + cl * 8)
                                             : "memory");
                    }
                    // these are generic-proxy writes and the tensor cores read the
                    // slot through the async proxy: each lane waits for its own
                    // copies and fences the proxies before the warp's one arrival
                    // (an arrival made by the copies themselves would leave the
                    // writes unfenced)
                    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(full);
                    if (fresh && (is_v || hh == 0)) {
                        // store the slot's new rows (K or V of this KV head, and the
                        // indexer-key row once, with KV head 0) into their pages
                        for (int i = max(kb, qbase); i < min(kb + nk, key1); ++i) {
                            const int gk = (i - kt) >> 5, ln = (i - kt) & 31;
                            const int64_t rg = gk == 0 ? r[0] : gk == 1 ? r[1] : gk == 2 ? r[2] : r[3];
                            const int64_t kr = shfl64(rg, ln);
                            if ((bm >> gk) & 1u) continue;
                            const int64_t rw = (int64_t)tok_off + (i - qbase);
                            uint16_t *row = const_cast<uint16_t *>(layer_base) + kr;
                            reinterpret_cast<uint4 *>(row)[lane] =
                                __ldg(reinterpret_cast<const uint4 *>(new_rows + (rw * H + kvh) * kHeadDim) + lane);
                            if (!is_v && kvh == 0 && a.ik_new != nullptr && lane < c.idx_dim / 8) {
                                const int prow = table ? i % ptok : i;
                                const int64_t page_start = kr - (int64_t)prow * kHeadDim;
                                uint16_t *idst = const_cast<uint16_t *>(layer_base) + page_start +
                                                 off_ik(H, c.idx_dim, ptok, prow);
                                reinterpret_cast<uint4 *>(idst)[lane] =
                                    __ldg(reinterpret_cast<const uint4 *>(a.ik_new + rw * c.idx_dim) + lane);
                            }
                        }
                    }
                }
            }
        }
    } else if (warp == kWarpMma && lane == 0) {
        // ---------------- MMA issue ----------------
        // operands written by threads (Q, P, key-by-key slots) were fenced by
        // their writers before they arrived
        const uint32_t idesc_s = mma_idesc(kN, false);
        const uint32_t idesc_o = mma_idesc(kHeadDim, true, v16);
        bool ok = mbar_wait(&bars[kBarQFull], 0, c.status);
        tc_fence_after();
        uint32_t q = 0;  // slots taken, in the producer's order
        auto take = [&](uint32_t &addr) -> bool {
            const uint32_t slot = q % kSlots;
            if (!mbar_wait(&bars[kBarFull + slot], (q / kSlots) & 1, c.status)) return false;
            tc_fence_after();
            addr = sbase + kOffRing + slot * kSlotBytes;
            return true;
        };
        auto give = [&]() {
            tc_commit(&bars[kBarEmpty + q % kSlots]);  // free once these MMAs are done
            ++q;
        };
        // S = Q K^T: Q (A) from TMEM, 8 columns (16 dims) a step; K (B) from
        // the tile's two dim-half slots
        auto issue_s = [&](int n) -> bool {
            if (n > 0 && !mbar_wait(&bars[kBarSEmpty], (n - 1) & 1, c.status)) return false;
#pragma unroll 1
            for (int hh = 0; hh < 2; ++hh) {
                uint32_t kb;
                if (!take(kb)) return false;
#pragma unroll
                for (int k8 = 0; k8 < 8; ++k8) {
                    const uint32_t kbb = kb + (k8 >> 2) * kKRegion + (k8 & 3) * 32;
                    tc_mma_ts(tmem + kSCol, tmem + kQCol + (8 * hh + k8) * 8, smem_desc(kbb, 16, 1024),
                              idesc_s, (hh > 0 || k8 > 0) ? 1u : 0u);
                }
                give();
            }
            tc_commit(&bars[kBarSFull]);
            return true;
        };
        if (ok && ntiles > 0) ok = issue_s(0);
        for (int n = 0; ok && n < ntiles; ++n) {
            if (n + 1 < ntiles && !issue_s(n + 1)) {
                ok = false;
                break;
            }
            if (!mbar_wait(&bars[kBarPFull], n & 1, c.status)) {
                ok = false;
                break;
            }
            // O += P V over the tile's two key-half slots
#pragma unroll 1
            for (int hh = 0; hh < 2 && ok; ++hh) {
                uint32_t vb;
                if (!take(vb)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4) {
                    const uint32_t pa = sbase + kOffP + hh * kPRegion + k4 * 32;
                    const uint32_t va = vb + k4 * 2048;  // 16 keys = two 8-row groups
                    tc_mma(tmem + kOCol, smem_desc(pa, 16, 1024), smem_desc(va, kVRegion, 1024), idesc_o,
                           (n > 0 || hh > 0 || k4 > 0) ? 1u : 0u);
                    if (!v16)
                        tc_mma(tmem + kOCol, smem_desc(pa + kPPart, 16, 1024), smem_desc(va, kVRegion, 1024),
                               idesc_o, 1u);
                }
                give();
            }
            if (!ok) break;
            tc_commit(&bars[kBarODone]);
        }
        if (!ok) *abort_flag = 1;
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        __syncwarp();  // lane 0 issued the MMAs, lanes 1-31 went straight here
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
}

// The fp16 V mode's rows: a warp a run of 16 consecutive keys of one KV
// head of a stream, a lane 16 bytes of each row, the 16 loads issued before
// any store.  A run inside one page (pages of a multiple of 16 positions, or
// a contiguous stream) takes one page lookup, any other run one a row; keys
// past the stream's length are zeros.  The lookups come before the
// grid-dependency wait, the loads after it.  A table entry outside
// [0, n_pages) is reported and read as page 0, as the chunk kernel does.
constexpr int kV16Threads = 128;
constexpr int kV16RowsWarp = 16;
constexpr int kV16RowsBlock = kV16Threads / 32 * kV16RowsWarp;
static_assert(kN % kV16RowsBlock == 0, "a stream's rows fill whole blocks");

__global__ void __launch_bounds__(kV16Threads)
    v16_gather(const __grid_constant__ Common c, const __grid_constant__ PrefillArgs a) {
    const int lane = threadIdx.x & 31;
    const int row0 = (blockIdx.x * (kV16Threads / 32) + (threadIdx.x >> 5)) * kV16RowsWarp;
    // the stream holding these rows (a block's rows lie in one stream: each
    // stream's rows are a multiple of the key tile)
    int s = 0;
    for (int t = 0; t < c.n_seqs; ++t)
        if (a.v16_row[t] >= 0 && row0 >= a.v16_row[t]) s = t;
    const SeqDev &sd = c.seq[s];
    const int stride = v16_stride(sd.len);
    const int local = row0 - a.v16_row[s];
    const int kvh = local / stride, key0 = local - kvh * stride;
    pdl_trigger();  // the chunk kernel waits for this grid before it reads the rows
    const int n = min(kV16RowsWarp, sd.len - key0);  // rows with data (<= 0: none)
    const bool one = sd.table == nullptr || sd.ptok % kV16RowsWarp == 0;
    const uint4 *src[kV16RowsWarp];
    if (one) {
        // consecutive positions of one head in a page are consecutive rows
        const uint4 *r0 = n > 0 ? reinterpret_cast<const uint4 *>(v_row(sd, c.n_kv_heads, kvh, key0, c.status)) + lane
                                : nullptr;
#pragma unroll
        for (int i = 0; i < kV16RowsWarp; ++i) src[i] = i < n ? r0 + i * (kHeadDim / 8) : nullptr;
    } else {
#pragma unroll
        for (int i = 0; i < kV16RowsWarp; ++i)
            src[i] = i < n ? reinterpret_cast<const uint4 *>(v_row(sd, c.n_kv_heads, kvh, key0 + i, c.status)) + lane
                           : nullptr;
    }
    pdl_wait();  // the rows were stored by an earlier kernel
    uint4 v[kV16RowsWarp];
#pragma unroll
    for (int i = 0; i < kV16RowsWarp; ++i) {
        v[i] = make_uint4(0, 0, 0, 0);
        if (src[i])  // volatile: the loads stay ahead of the stores
            asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v[i].x), "=r"(v[i].y), "=r"(v[i].z), "=r"(v[i].w)
                         : "l"(src[i]));
    }
    asm volatile("" ::: "memory");
    // volatile too, so that no conversion (and the wait for its row) is
    // placed between the loads
    auto cvt = [](uint32_t w) {
        uint32_t h;
        asm volatile("cvt.rn.f16x2.f32 %0, %1, %2;"
                     : "=r"(h)
                     : "f"(__uint_as_float(w & 0xffff0000u)), "f"(__uint_as_float(w << 16)));
        return h;
    };
#pragma unroll
    for (int i = 0; i < kV16RowsWarp; ++i) {
        const uint4 h = make_uint4(cvt(v[i].x), cvt(v[i].y), cvt(v[i].z), cvt(v[i].w));
        reinterpret_cast<uint4 *>(a.v16 + (int64_t)(row0 + i) * kHeadDim)[lane] = h;
    }
}

}  // namespace

// Work items: (KV head, M-tile, split) per stream, splits fastest.  A stream
// is split only as far as filling the SMs needs, from its own shape alone.
// Split model of plan_prefill, in hundredths of a microsecond.
constexpr int64_t kTileCost = 220;   // a 128-key tile of one 128-row M-tile (bf16 V)
constexpr int64_t kTileCost16 = 175; // the same in the fp16 V mode
constexpr int64_t kCtaCost = 1200;   // a CTA's fixed cost
constexpr int64_t kPartialCost = 4;  // a (unit, split) partial written and read back
constexpr int kMaxPrefillSplits = 64;

int plan_prefill(Common &c, int nsm, DecodePlan *plan) {
    int32_t items = 0, comb = 0;
    int64_t floats = 0;
    const int H = c.n_kv_heads;
    for (int s = 0; s < c.n_seqs; ++s) c.seq[s].ncols = c.seq[s].n_new * c.group;
    const int64_t tile_cost = v16_rows(c) > 0 ? kTileCost16 : kTileCost;
    for (int s = 0; s < c.n_seqs; ++s) {
        SeqDev &d = c.seq[s];
        d.work_off = 0;
        d.comb_off = comb;
        d.ws_off = floats;
        d.ncols = d.n_new * c.group;
        if (d.ncols == 0) {
            d.nsplit = 1;
            d.split_len = kN;
            continue;
        }
        const int mtiles = (d.ncols + kM - 1) / kM;
        // Splits: the count with the least modelled time for this stream's
        // grid on nsm SMs, waves x (tiles a CTA x a tile's time + a CTA's
        // fixed cost) + the split partials' round trip through HBM.  The
        // costs are this kernel's on GB300: about 2.2 us a 128-key tile of
        // 128 rows (1.75 us in the fp16 V mode), 12 us a CTA (Q into TMEM,
        // pipeline fill, epilogue, the next CTA's entry) and 0.04 us a
        // (unit, split) partial of 128 rows written and read back.  For 512
        // queries at 31,000 (64 units) it picks 2 splits, one wave of 128
        // CTAs (bf16 V: 296 us; 7 splits, three nearly full waves, measured
        // the same, 3-6 and 8-19 splits 310-395 us).  For 2,048 queries at
        // 16,384 (256 units) it picks 1 split, 2 waves.
        // Only the stream's own length and rows and the SM count enter, so
        // paged and contiguous caches get the same splits.
        const int64_t units = (int64_t)H * mtiles, tiles = (d.len + kN - 1) / kN;
        const int max_ns = std::max(1, std::min(kMaxPrefillSplits, d.len / 256));  // 256 keys a split at least
        int ns = 1;
        int64_t best = INT64_MAX;
        for (int n = 1; n <= max_ns; ++n) {
            const int64_t waves = (units * n + nsm - 1) / nsm;
            const int64_t cost = waves * (((tiles + n - 1) / n) * tile_cost + kCtaCost) +
                                 (n > 1 ? n * units * kPartialCost : 0);
            if (cost < best) {
                best = cost;
                ns = n;
            }
        }
        int sl = (d.len + ns - 1) / ns;
        sl = (sl + kN - 1) / kN * kN;
        ns = (d.len + sl - 1) / sl;
        if (ns > 2048) return PKV_EINVAL;
        d.nsplit = ns;
        d.split_len = sl;
        if (ns > 1) {
            comb += H * d.ncols * comb_ctas(ns);
            floats += (int64_t)H * ns * d.ncols * (kHeadDim + 2);
            floats = (floats + 63) / 64 * 64;
        }
    }
    // Work-item blocks in the grid, longest CTA first (most key tiles a
    // split, ties in stream order): the SMs that take the long CTAs first are
    // refilled with short ones, instead of a long stream's CTAs starting last
    // and running alone at the end.  Only the launch order changes: each
    // stream's splits, and so its results, stay its own.
    int order[PKV_MAX_SEQS];
    for (int s = 0; s < c.n_seqs; ++s) order[s] = s;
    std::stable_sort(order, order + c.n_seqs, [&](int x, int y) {
        return c.seq[x].split_len > c.seq[y].split_len;
    });
    for (int k = 0; k < c.n_seqs; ++k) {
        SeqDev &d = c.seq[order[k]];
        if (d.ncols == 0) continue;
        d.work_off = items;
        items += H * ((d.ncols + kM - 1) / kM) * d.nsplit;
    }
    // the fp16 V mode's rows, after the partials
    const int64_t rows16 = v16_rows(c);
    plan->total_items = items;
    plan->total_comb = comb;
    plan->ws_bytes = static_cast<size_t>(floats) * 4 + static_cast<size_t>(rows16) * kHeadDim * 2;
    return PKV_OK;
}

int launch_prefill(const Common &c, const DecodePlan &plan, const DecodeMaps &maps,
                   const uint16_t *q, uint16_t *out, float *ws, const uint16_t *k_new,
                   const uint16_t *v_new, const uint16_t *ik_new, cudaStream_t stream) {
    static std::atomic<uint64_t> attr_done{0};
    if (once_per_device(attr_done, [] {
            const int rc = cuda_rc(cudaFuncSetAttribute(prefill_partial<false>,
                                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                        static_cast<int>(PLayout<false>::smem)));
            if (rc != PKV_OK) return rc;
            return cuda_rc(cudaFuncSetAttribute(prefill_partial<true>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                static_cast<int>(PLayout<true>::smem)));
        }) != PKV_OK)
        return PKV_ECUDA;
    PrefillArgs a{q, out, ws, k_new, v_new, ik_new, nullptr, -1, {}};
    for (int s = 0; s < PKV_MAX_SEQS; ++s) a.v16_row[s] = -1;
    // the fp16 V mode (chunks only: a decode call's new rows are not in
    // their pages yet): rows at the end of the workspace, as planned
    DecodeMaps m16 = maps;
    int64_t rows16 = k_new == nullptr ? v16_rows(c) : 0;
    const size_t bytes16 = static_cast<size_t>(rows16) * kHeadDim * 2;
    if (plan.ws_bytes < bytes16) rows16 = 0;
    for (int s = 0, r = 0; s < c.n_seqs && rows16 > 0; ++s)
        if (c.seq[s].ncols > 0) {
            a.v16_row[s] = r;
            r += c.n_kv_heads * v16_stride(c.seq[s].len);
        }
    if (rows16 > 0) {
        int n_maps = 0;
        for (int s = 0; s < c.n_seqs; ++s)
            n_maps = std::max(n_maps, std::max<int>(c.seq[s].tma, std::max<int>(c.seq[s].tma_k, c.seq[s].tma_v)) + 1);
        a.v16 = reinterpret_cast<uint16_t *>(reinterpret_cast<char *>(ws) + (plan.ws_bytes - bytes16));
        // the V slots' tile view (boxes of {64, 64, 4}) over the fp16 rows:
        // the map's element type is bf16, and a TMA copy moves the 2-byte
        // elements' bits unchanged, so fp16 rows come through as they are
        a.v16_map = row_map(m16, n_maps, a.v16, static_cast<uint64_t>(rows16), false, true, 64, 4);
        if (a.v16_map < 0) rows16 = 0;  // no map to be had: bf16 V
    }
    if (rows16 == 0) {
        a.v16 = nullptr;
        a.v16_map = -1;
        for (int s = 0; s < PKV_MAX_SEQS; ++s) a.v16_row[s] = -1;
    } else {
        cudaError_t e = launch_pdl(v16_gather, static_cast<unsigned>(rows16 / kV16RowsBlock), kV16Threads, 0,
                                   stream, c, a);
        if (e != cudaSuccess) return PKV_ECUDA;
    }
    cudaError_t e = rows16 > 0
                        ? launch_pdl(prefill_partial<true>, plan.total_items, kPThreads, PLayout<true>::smem,
                                     stream, c, m16, a)
                        : launch_pdl(prefill_partial<false>, plan.total_items, kPThreads, PLayout<false>::smem,
                                     stream, c, maps, a);
    if (e != cudaSuccess) return PKV_ECUDA;
    if (plan.total_comb > 0) return launch_combine(c, plan, q, out, ws, stream);
    return PKV_OK;
}

}  // namespace pkv
