// Decode attention over e4m3 K/V rows (#1170, commit 5c09685: a row's e4m3
// codes and float32 scale through the page table; the reference dequantizes
// code x scale).  Same work units, split plan and partial layout as the bf16
// decode, so the same combine kernel merges the splits, paged output equals
// contiguous output and a stream's output does not depend on its batch.
//
// A CTA is one (stream, KV head, split) unit of 8 warps.  The warps take the
// split's 16-key tiles round robin (one key slice per warp and column group)
// and each stages its own tiles, three deep: with codes at half the bytes of
// bf16 rows, a split of 256 keys is in flight before the grid-dependency
// wait.  A whole tile of a page whose size is a multiple of 16 is four 2D TMA
// boxes (16 code rows x 128 bytes, 128-byte swizzle) and two bulk copies of
// its 16 K and 16 V scales; a ragged tail is copied key by key, clamped into
// the split, so every staged row is a real row (a masked key's code must not
// be a NaN pattern).  Per tile a warp computes S^T = K Q^T and
// O^T += V^T P^T with mma.sync in f16 (an e4m3 code widens to f16 exactly;
// the queries are converted once), applies the K scale to S in float32,
// and keeps an online softmax per query column.  The V scale s = 2^E x mant
// (mant in [1, 2)) is folded into each key's weight: the sum of weights L
// keeps the logit's running maximum m, while O keeps a running maximum u of
// logit + E of its own, so the weight of the key that carries most of O is
// near 1 and every weight 2^(x + E - u) x mant lies in [0, 2), where f16 is
// precise whatever the spread of the row scales (a reference on the scales
// alone lets the weight of a large-scale key with a small softmax weight
// fall into f16's subnormals).  The weights are split into f16 hi + lo
// parts; O is brought back to m's reference once, at the end.  Dims are
// permuted inside the MMAs so
// every operand fragment comes from contiguous 16-byte shared-memory loads:
// in S thread group c (lane & 3) sums dims 64c .. 64c+63; in O^T row g of
// M-tile m is dim 32g + 2m and row g+8 is dim 32g + 2m + 1.
#include <cuda_fp16.h>

#include "pkv_dev.cuh"

namespace pkv {
namespace {

constexpr int kT8 = 16;                              // keys a tile
constexpr int kHalf8 = kT8 * 128;                    // 128-byte halves of 16 code rows (a TMA box)
constexpr int kCodes8 = 2 * kHalf8;                  // one tile's K (or V) codes, swizzled
constexpr int kTile8 = 2 * kCodes8;                  // K and V codes (a multiple of 1024 B)
constexpr int kWarps8 = 8;
constexpr int kThreads8 = kWarps8 * 32;
constexpr int kDepth8 = 3;                           // tiles in flight a warp
constexpr int kSlots8 = kWarps8 * kDepth8;
constexpr size_t kOffScl8 = (size_t)kSlots8 * kTile8;          // 16 K then 16 V scales a slot
constexpr size_t kOffBar8 = kOffScl8 + (size_t)kSlots8 * 128;  // a barrier a slot
constexpr size_t kSmem8 = 1024 + kOffBar8 + kSlots8 * 8 + 16;
// merge rows: dim d of a column at d + d / 32 (lanes that differ in g write
// different banks), columns kMS8 floats apart
constexpr int kMS8 = kHeadDim + 12;
constexpr float kScaleLog2 = 0.0625f * 1.4426950408889634f;  // log2(e) / sqrt(256)
static_assert(64 * kMS8 * 4 + 64 * 4 * 4 + 64 * 4 <= kOffScl8, "merge buffers reuse the stages");

// Byte offset of 16-byte chunk ch (0..15) of code row r (0..15) in a staged
// tile: two 128-byte halves, each 16 rows with chunk j at j ^ (r & 7).
__device__ __forceinline__ uint32_t sw8(int r, int ch) {
    return (ch >> 3) * kHalf8 + r * 128 + ((((ch & 7) ^ (r & 7))) << 4);
}

struct Decode8Args {
    const uint16_t *q;
    uint16_t *out;
    float *ws;
    const uint16_t *k_new;  // fused store of the new tokens (quantized here), or null
    const uint16_t *v_new;
    const uint16_t *ik_new;
};

// Two e4m3 codes (low byte first) to an f16 pair, exactly.
__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t two) {
    uint32_t r;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}"
        : "=r"(r)
        : "r"(two));
    return r;
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }

__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}


__device__ __forceinline__ float max_over_g(float v) {  // lanes sharing lane & 3
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
    return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
}

// s = 2^e x mant with mant in [1, 2); a zero or subnormal scale (a row of
// values below 2^-126 x 448) gives e = -inf, so its weight is 0.
__device__ __forceinline__ void pow2_split(float s, float &e, float &mant) {
    const uint32_t b = __float_as_uint(s);
    const int ex = static_cast<int>((b >> 23) & 0xffu);
    const bool normal = ex != 0 && ex != 0xff;
    e = normal ? static_cast<float>(ex - 127) : -INFINITY;
    mant = normal ? __uint_as_float((b & 0x007fffffu) | 0x3f800000u) : 0.f;
}

__device__ __forceinline__ float sum_over_g(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    v += __shfl_xor_sync(0xffffffffu, v, 8);
    return v + __shfl_xor_sync(0xffffffffu, v, 16);
}

__global__ void __maxnreg__(192)
    decode8_partial(const __grid_constant__ Common c, const __grid_constant__ DecodeMaps maps,
                    const Decode8Args a) {
    extern __shared__ uint8_t sm8_raw[];
    uint8_t *sm8 = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(sm8_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm8 + kOffBar8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + kSlots8);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, c4 = lane & 3;
    const int s = find_seq(c.n_seqs, blockIdx.x, [&](int t) { return c.seq[t].work_off; });
    const SeqDev &sd = c.seq[s];
    const int r = blockIdx.x - sd.work_off;
    const int kvh = r / sd.nsplit, split = r - kvh * sd.nsplit;
    const int H = c.n_kv_heads, G = c.group;
    const int key0 = split * sd.split_len, key1 = min(sd.len, key0 + sd.split_len);
    const int ntiles = (key1 - key0 + kT8 - 1) / kT8;
    const int ncols = sd.ncols, ncg = (ncols + 7) >> 3;
    const int ks_n = kWarps8 / ncg;  // key slices
    const int cg = warp % ncg, ks = warp / ncg;
    const bool active = ks < ks_n;
    const int qbase = sd.len - sd.n_new;
    const uint8_t *base = reinterpret_cast<const uint8_t *>(sd.layer_base);
    const int my_tiles = (active && ks < ntiles) ? (ntiles - ks + ks_n - 1) / ks_n : 0;
    const uint64_t pol = policy_evict_first();
    const void *map = sd.tma >= 0 ? &maps.map[sd.tma] : nullptr;

    if (tid == 0) {
        for (int i = 0; i < kSlots8; ++i) mbar_init(&bars[i], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    const bool fuse = a.k_new != nullptr;

    // Stage tile t of this warp's slice into its slot: lane i (and i + 16)
    // looks key i up once; 16 rows of K codes, 16 of V codes, 16 K and 16 V
    // scales, all completing on the slot's barrier.  With a fused store, the
    // rows of new positions are quantized here from k_new / v_new (the same
    // rule as pkv_store), written to the cache and to the stage directly.
    auto issue = [&](int t) {
        const int kt = key0 + (ks + t * ks_n) * kT8;
        const int slot = warp * kDepth8 + t % kDepth8;
        uint8_t *st = sm8 + (size_t)slot * kTile8;
        uint8_t *sc = sm8 + kOffScl8 + slot * 128;
        uint64_t *bar = &bars[slot];
        const int key = min(kt + (lane & 15), key1 - 1);
        int64_t pg = 0;
        int32_t row = key;
        bool bad = false;
        if (sd.table) {
            const int page = key / sd.ptok;
            row = key - page * sd.ptok;
            const int id = __ldg(sd.table + page);
            if (static_cast<uint32_t>(id) < static_cast<uint32_t>(sd.n_pages)) {
                pg = 2 * (int64_t)id * sd.ps;
            } else {
                bad = true;
                if (c.status && lane < 16) atomicOr(c.status, PKV_DEV_BAD_PAGE);
            }
        }
        const int64_t kc = pg + off8_code(false, H, sd.ptok, kvh, row);
        const int64_t vc = pg + off8_code(true, H, sd.ptok, kvh, row);
        if (fuse && min(kt + kT8, key1) - 1 >= qbase) {
            // a tile holding new positions: cached rows copied key by key,
            // new rows quantized by the whole warp, one row at a time
            const bool fresh = key >= qbase;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int item = lane + 32 * i, rr = item >> 4, ch = item & 15;
                const int64_t krr = shfl64(kc, rr), vrr = shfl64(vc, rr);
                const bool frr = __shfl_sync(0xffffffffu, fresh, rr);
                if (!frr) {
                    cp_async16(st + sw8(rr, ch), base + krr + 16 * ch, pol);
                    cp_async16(st + kCodes8 + sw8(rr, ch), base + vrr + 16 * ch, pol);
                }
            }
            if (!fresh) cp_async4(sc + 4 * lane, base + pg + off8_scale(lane >= 16, H, sd.ptok, kvh, row));
            // rows past the split's end repeat its last key, masked in the
            // softmax: zero codes and scales keep them finite without work
            const unsigned past = __ballot_sync(0xffffffffu, lane < 16 && kt + lane >= key1);
            unsigned todo = __ballot_sync(0xffffffffu, fresh && lane < 16) & ~past;
            if (past) {
                for (int rr = __ffs(past) - 1; rr < kT8; ++rr) {
                    *reinterpret_cast<uint2 *>(st + sw8(rr, lane >> 1) + (lane & 1) * 8) = make_uint2(0u, 0u);
                    *reinterpret_cast<uint2 *>(st + kCodes8 + sw8(rr, lane >> 1) + (lane & 1) * 8) = make_uint2(0u, 0u);
                }
                if (lane < 16 && ((past >> lane) & 1u)) {
                    reinterpret_cast<float *>(sc)[lane] = 0.f;
                    reinterpret_cast<float *>(sc)[16 + lane] = 0.f;
                }
            }
            while (todo) {
                const int rr = __ffs(todo) - 1;
                todo &= todo - 1;
                const int p = kt + rr;                           // its position
                const bool write = !__shfl_sync(0xffffffffu, bad, rr);
                const int64_t tr = (int64_t)sd.tok_off + (p - qbase);  // its packed input row
                const int64_t pg_rr = shfl64(pg, rr);
                const int row_rr = __shfl_sync(0xffffffffu, row, rr);
                const bool ik_row = write && kvh == 0 && a.ik_new != nullptr && lane < c.idx_dim / 8;
                // the row's inputs load together: one round trip
                const uint4 in_k = __ldg(reinterpret_cast<const uint4 *>(a.k_new + (tr * H + kvh) * kHeadDim) + lane);
                const uint4 in_v = __ldg(reinterpret_cast<const uint4 *>(a.v_new + (tr * H + kvh) * kHeadDim) + lane);
                const uint4 in_ik = ik_row ? __ldg(reinterpret_cast<const uint4 *>(a.ik_new + tr * c.idx_dim) + lane)
                                           : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int v = 0; v < 2; ++v) {
                    uint2 codes;
                    const float scale = quantize_row8(v ? in_v : in_k, &codes);
                    *reinterpret_cast<uint2 *>(st + (v ? kCodes8 : 0) + sw8(rr, lane >> 1) + (lane & 1) * 8) = codes;
                    if (lane == 0) reinterpret_cast<float *>(sc)[16 * v + rr] = scale;
                    if (write) {
                        uint8_t *lb = const_cast<uint8_t *>(base) + pg_rr;
                        *reinterpret_cast<uint2 *>(lb + off8_code(v, H, sd.ptok, kvh, row_rr) + 8 * lane) = codes;
                        if (lane == 0) *reinterpret_cast<float *>(lb + off8_scale(v, H, sd.ptok, kvh, row_rr)) = scale;
                    }
                }
                if (ik_row) {
                    // the indexer-key row of the position, written once (KV head 0)
                    uint8_t *idst = const_cast<uint8_t *>(base) + pg_rr + 2 * off_ik_f(true, H, c.idx_dim, sd.ptok, row_rr);
                    reinterpret_cast<uint4 *>(idst)[lane] = in_ik;
                }
            }
            cp_async_mbar_arrive(bar);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar);
        } else if (map != nullptr && kt + kT8 <= key1) {
            // one page holds the 16 keys (page size a multiple of 16, tiles
            // start on 16): their code rows and scales are contiguous runs
            const int yk = static_cast<int>(sd.layer_row + shfl64(kc, 0) / 256);
            const int yv = static_cast<int>(sd.layer_row + shfl64(vc, 0) / 256);
            const int64_t s0 = shfl64(pg, 0) + off8_scale(false, H, sd.ptok, kvh, __shfl_sync(0xffffffffu, row, 0));
            const int64_t s1 = shfl64(pg, 0) + off8_scale(true, H, sd.ptok, kvh, __shfl_sync(0xffffffffu, row, 0));
            if (lane == 0) {
                mbar_arrive_expect_tx(bar, kTile8 + 128);
                tma_load_2d(st, map, 0, yk, bar, pol);
                tma_load_2d(st + kHalf8, map, 128, yk, bar, pol);
                tma_load_2d(st + kCodes8, map, 0, yv, bar, pol);
                tma_load_2d(st + kCodes8 + kHalf8, map, 128, yv, bar, pol);
                bulk_g2s(sc, base + s0, 64, bar, pol);
                bulk_g2s(sc + 64, base + s1, 64, bar, pol);
            }
        } else {
            // key rr's rows from lane rr's lookup, in the same swizzled layout
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int item = lane + 32 * i, rr = item >> 4, ch = item & 15;
                cp_async16(st + sw8(rr, ch), base + shfl64(kc, rr) + 16 * ch, pol);
                cp_async16(st + kCodes8 + sw8(rr, ch), base + shfl64(vc, rr) + 16 * ch, pol);
            }
            cp_async4(sc + 4 * lane, base + pg + off8_scale(lane >= 16, H, sd.ptok, kvh, row));
            cp_async_mbar_arrive(bar);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar);
        }
    };

    // nothing this CTA writes is read by the next kernel before its own wait
    // (a decode reads no row within 32 positions of its new tokens early)
    if (tid == 0) pdl_trigger();
    // rows of cached positions more than 32 below the new tokens stream
    // before the grid-dependency wait; later tiles (a decode of the same
    // stream queued just before may still be storing the rows right below
    // the new tokens) wait for it
    int issued = 0;
    for (; issued < kDepth8 && issued < my_tiles; ++issued) {
        const int kt = key0 + (ks + issued * ks_n) * kT8;
        if (kt + kT8 > qbase - 32) break;
        issue(issued);
    }
    // the query row's address from the launch parameters before the wait
    // (an asm use the compiler cannot move past it): only its load waits
    const uint16_t *qr = nullptr;
    {
        const int col = cg * 8 + g;
        if (active && col < ncols) {
            const int j = col / G;
            qr = a.q + (((int64_t)sd.tok_off + j) * c.n_q_heads + kvh * G + (col - j * G)) * kHeadDim;
        }
    }
    asm volatile("" ::"l"(qr));
    pdl_wait();
    __syncthreads();
    for (; issued < kDepth8 && issued < my_tiles; ++issued) issue(issued);

    // the queries of this thread's B-operand column, in the permuted dim order
    uint32_t qf[16][2];
    {
        // dims 64 c4 .. 64 c4 + 63 of the row: eight 16-byte loads, two steps each
        uint4 u[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            u[i] = qr ? __ldg(reinterpret_cast<const uint4 *>(qr + 64 * c4) + i) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            qf[2 * i][0] = h2_bits(__floats2half2_rn(bf16_lo(u[i].x), bf16_hi(u[i].x)));
            qf[2 * i][1] = h2_bits(__floats2half2_rn(bf16_lo(u[i].y), bf16_hi(u[i].y)));
            qf[2 * i + 1][0] = h2_bits(__floats2half2_rn(bf16_lo(u[i].z), bf16_hi(u[i].z)));
            qf[2 * i + 1][1] = h2_bits(__floats2half2_rn(bf16_lo(u[i].w), bf16_hi(u[i].w)));
        }
    }
    const int colA = cg * 8 + 2 * c4, colB = colA + 1;
    const int limA = colA < ncols ? qbase + colA / G : -1;
    const int limB = colB < ncols ? qbase + colB / G : -1;

    float acc[16][4];
#pragma unroll
    for (int m = 0; m < 16; ++m) acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0.f;
    float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
    float uA = -INFINITY, uB = -INFINITY;  // running max of logit + V-scale exponent (O's reference)

    for (int t = 0; t < my_tiles; ++t) {
        const int slot = warp * kDepth8 + t % kDepth8;
        // every lane waits (the barrier makes the async copies visible to it);
        // a wait that runs out leaves the loop on every lane together
        if (!__all_sync(0xffffffffu, mbar_wait(&bars[slot], (t / kDepth8) & 1, c.status))) {
            *abort_flag = 1;
            break;
        }
        const uint8_t *st = sm8 + (size_t)slot * kTile8;
        const float *scl = reinterpret_cast<const float *>(sm8 + kOffScl8 + slot * 128);
        const int kt = key0 + (ks + t * ks_n) * kT8;

        // ---- S^T = K Q^T: rows keys g and g + 8, columns colA and colB ----
        float sacc[4] = {0.f, 0.f, 0.f, 0.f};
        {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 w0 = *reinterpret_cast<const uint4 *>(st + sw8(g, 4 * c4 + i));
                const uint4 w1 = *reinterpret_cast<const uint4 *>(st + sw8(g + 8, 4 * c4 + i));
                const uint32_t x0[4] = {w0.x, w0.y, w0.z, w0.w}, x1[4] = {w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    mma_f16(sacc, e4m3x2_f16x2(x0[j] & 0xffffu), e4m3x2_f16x2(x1[j] & 0xffffu),
                            e4m3x2_f16x2(x0[j] >> 16), e4m3x2_f16x2(x1[j] >> 16), qf[4 * i + j][0],
                            qf[4 * i + j][1]);
            }
        }
        // ---- K scale, causal and split bounds, online softmax ----
        const int ka = kt + g, kb = kt + g + 8;
        const float ska = scl[g] * kScaleLog2, skb = scl[g + 8] * kScaleLog2;
        float x[4];
        x[0] = (ka < key1 && ka <= limA) ? sacc[0] * ska : -INFINITY;
        x[1] = (ka < key1 && ka <= limB) ? sacc[1] * ska : -INFINITY;
        x[2] = (kb < key1 && kb <= limA) ? sacc[2] * skb : -INFINITY;
        x[3] = (kb < key1 && kb <= limB) ? sacc[3] * skb : -INFINITY;
        const float nA = fmaxf(mA, max_over_g(fmaxf(x[0], x[2])));
        const float nB = fmaxf(mB, max_over_g(fmaxf(x[1], x[3])));
        const float oA = nA == -INFINITY ? 0.f : nA, oB = nB == -INFINITY ? 0.f : nB;
        const float alA = ex2(mA - oA), alB = ex2(mB - oB);  // 0 while nothing was accumulated
        float p[4];
        p[0] = ex2(x[0] - oA);
        p[1] = ex2(x[1] - oB);
        p[2] = ex2(x[2] - oA);
        p[3] = ex2(x[3] - oB);
        lA = lA * alA + sum_over_g(p[0] + p[2]);
        lB = lB * alB + sum_over_g(p[1] + p[3]);
        mA = nA;
        mB = nB;
        // ---- weights of O: 2^(x + E - u) x mant for the V scale 2^E x mant ----
        float ea, ma, eb, mb;
        pow2_split(scl[16 + g], ea, ma);
        pow2_split(scl[16 + g + 8], eb, mb);
        const float y0 = x[0] + ea, y1 = x[1] + ea, y2 = x[2] + eb, y3 = x[3] + eb;
        const float nuA = fmaxf(uA, max_over_g(fmaxf(y0, y2)));
        const float nuB = fmaxf(uB, max_over_g(fmaxf(y1, y3)));
        const float vA = nuA == -INFINITY ? 0.f : nuA, vB = nuB == -INFINITY ? 0.f : nuB;
        const float beA = ex2(uA - vA), beB = ex2(uB - vB);  // 0 while nothing was accumulated
        uA = nuA;
        uB = nuB;
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            acc[m][0] *= beA;
            acc[m][1] *= beB;
            acc[m][2] *= beA;
            acc[m][3] *= beB;
        }
        // ---- the weights as f16 hi + lo, to the B-operand layout ----
        const float q0 = ex2(y0 - vA) * ma, q1 = ex2(y1 - vB) * ma;
        const float q2 = ex2(y2 - vA) * mb, q3 = ex2(y3 - vB) * mb;
        const __half2 h01 = __floats2half2_rn(q0, q1), h23 = __floats2half2_rn(q2, q3);
        const __half2 l01 = __floats2half2_rn(q0 - __low2float(h01), q1 - __high2float(h01));
        const __half2 l23 = __floats2half2_rn(q2 - __low2float(h23), q3 - __high2float(h23));
        const uint32_t b0h = movmatrix_t(h2_bits(h01)), b1h = movmatrix_t(h2_bits(h23));
        const uint32_t b0l = movmatrix_t(h2_bits(l01)), b1l = movmatrix_t(h2_bits(l23));
        // ---- O^T += V^T P'^T: V codes of keys 2c, 2c+1, 2c+8, 2c+9, dims 32g .. 32g+31 ----
        uint32_t w[4][8];
        {
            const uint8_t *vb = st + kCodes8;
            const int kr[4] = {2 * c4, 2 * c4 + 1, 2 * c4 + 8, 2 * c4 + 9};
#pragma unroll
            for (int x4 = 0; x4 < 4; ++x4) {
                const uint4 u0 = *reinterpret_cast<const uint4 *>(vb + sw8(kr[x4], 2 * g));
                const uint4 u1 = *reinterpret_cast<const uint4 *>(vb + sw8(kr[x4], 2 * g + 1));
                w[x4][0] = u0.x;
                w[x4][1] = u0.y;
                w[x4][2] = u0.z;
                w[x4][3] = u0.w;
                w[x4][4] = u1.x;
                w[x4][5] = u1.y;
                w[x4][6] = u1.z;
                w[x4][7] = u1.w;
            }
        }
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            const int wi = m >> 1, b = 2 * (m & 1);
            const uint32_t sel0 = b | ((4 + b) << 4), sel1 = (b + 1) | ((5 + b) << 4);
            const uint32_t a0 = e4m3x2_f16x2(__byte_perm(w[0][wi], w[1][wi], sel0));
            const uint32_t a1 = e4m3x2_f16x2(__byte_perm(w[0][wi], w[1][wi], sel1));
            const uint32_t a2 = e4m3x2_f16x2(__byte_perm(w[2][wi], w[3][wi], sel0));
            const uint32_t a3 = e4m3x2_f16x2(__byte_perm(w[2][wi], w[3][wi], sel1));
            mma_f16(acc[m], a0, a1, a2, a3, b0h, b1h);
            mma_f16(acc[m], a0, a1, a2, a3, b0l, b1l);
        }
        __syncwarp();  // every lane is done with the stage before it is refilled
        if (issued < my_tiles) {
            fence_proxy_async_smem();  // these reads come before the next copies' writes
            issue(issued);
            ++issued;
        }
    }

    // ---- merge the key slices of each column group in a fixed order ----
    __syncthreads();
    const int NC = ncg * 8;
    float *mbuf = reinterpret_cast<float *>(sm8);  // [ks][NC][kMS8]
    float *mlb = mbuf + ks_n * NC * kMS8;          // [ks][NC][2]
    if (active) {
        // O from its own reference u back to the logits' m: 2^(u - m)
        const float fA = uA == -INFINITY ? 0.f : ex2(uA - mA);
        const float fB = uB == -INFINITY ? 0.f : ex2(uB - mB);
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            const int d0 = 33 * g + 2 * m;  // dim 32 g + 2 m, skewed by g
            mbuf[(ks * NC + colA) * kMS8 + d0] = acc[m][0] * fA;
            mbuf[(ks * NC + colB) * kMS8 + d0] = acc[m][1] * fB;
            mbuf[(ks * NC + colA) * kMS8 + d0 + 1] = acc[m][2] * fA;
            mbuf[(ks * NC + colB) * kMS8 + d0 + 1] = acc[m][3] * fB;
        }
        if (g == 0) {
            mlb[(ks * NC + colA) * 2 + 0] = mA;
            mlb[(ks * NC + colA) * 2 + 1] = lA;
            mlb[(ks * NC + colB) * 2 + 0] = mB;
            mlb[(ks * NC + colB) * 2 + 1] = lB;
        }
    }
    __syncthreads();
    const bool single = sd.nsplit == 1;
    float *part_acc = a.ws + sd.ws_off;
    float *part_ml = part_acc + (int64_t)H * sd.nsplit * ncols * kHeadDim;
    const int64_t pidx = ((int64_t)kvh * sd.nsplit + split) * ncols;
    for (int idx = tid; idx < ncols * (kHeadDim / 4); idx += kThreads8) {
        const int col = idx / (kHeadDim / 4), d = 4 * (idx - col * (kHeadDim / 4));
        // the slices' weights of the column (each thread of a column computes them)
        float M = -INFINITY;
        for (int k = 0; k < ks_n; ++k) M = fmaxf(M, mlb[(k * NC + col) * 2]);
        float L = 0.f;
        float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
        const int sd0 = d + (d >> 5);  // the four dims share one skew
        for (int k = 0; k < ks_n; ++k) {
            const float wk = M == -INFINITY ? 0.f : ex2(mlb[(k * NC + col) * 2] - M);
            L += wk * mlb[(k * NC + col) * 2 + 1];
            const float *v = mbuf + (k * NC + col) * kMS8 + sd0;
            O.x += wk * v[0];
            O.y += wk * v[1];
            O.z += wk * v[2];
            O.w += wk * v[3];
        }
        if (single) {
            const float inv = L > 0.f ? 1.f / L : 0.f;
            const int j = col / G;
            uint2 pk;
            pk.x = pack_bf16(O.x * inv, O.y * inv);
            pk.y = pack_bf16(O.z * inv, O.w * inv);
            *reinterpret_cast<uint2 *>(
                a.out + (((int64_t)sd.tok_off + j) * c.n_q_heads + kvh * G + (col - j * G)) * kHeadDim + d) = pk;
        } else {
            *reinterpret_cast<float4 *>(part_acc + (pidx + col) * kHeadDim + d) = O;
            if (d == 0) {
                part_ml[(pidx + col) * 2 + 0] = M;
                part_ml[(pidx + col) * 2 + 1] = L;
            }
        }
    }
}

}  // namespace

int launch_decode8(const Common &c, const DecodePlan &plan, const DecodeMaps &maps,
                   const uint16_t *q, uint16_t *out, float *ws, const uint16_t *k_new,
                   const uint16_t *v_new, const uint16_t *ik_new, cudaStream_t stream) {
    static std::atomic<uint64_t> attr_done{0};
    if (once_per_device(attr_done, [] {
            if (cudaFuncSetAttribute(decode8_partial, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kSmem8)) != cudaSuccess)
                return PKV_ECUDA;
            return cuda_rc(cudaFuncSetAttribute(decode8_partial,
                                                cudaFuncAttributePreferredSharedMemoryCarveout,
                                                cudaSharedmemCarveoutMaxShared));
        }) != PKV_OK)
        return PKV_ECUDA;
    Decode8Args a{q, out, ws, k_new, v_new, ik_new};
    cudaError_t e =
        launch_pdl(decode8_partial, plan.total_items, kThreads8, kSmem8, stream, c, maps, a);
    if (e != cudaSuccess) return PKV_ECUDA;
    if (plan.total_comb > 0) return launch_combine(c, plan, q, out, ws, stream);
    return PKV_OK;
}

}  // namespace pkv
