// Block scores over pooled rows and top-k block selection.
//
// Scores: each (head, block) score is the float32 chain
// acc = fmaf(qi[d], P[b][d], acc), d = 0 .. Di-1, run by one thread (the
// order is part of the result: a top-k decision downstream must see the same
// bits on any cache layout); a thread runs two such chains side by side, and
// a CTA takes 32 blocks, so a stream of 2,250 blocks spreads over 71 CTAs.
// Pooled rows are looked up once per block (pg_at on its first position) and
// staged in shared memory with 16-byte loads.
//
// Top-k: one CTA per (stream, head) finds the k-th largest score on
// order-preserving keys (held in shared memory when the row fits): one
// histogram of the keys' top 11 bits locates the bin holding it; when that
// bin holds at most 64 keys one warp sorts them, when it holds at most 512
// the k-th largest is found by ranking them directly, and otherwise an 8-bit
// radix select over all 32 bits finds it (each pass's digit found by one warp
// in parallel).  The selected block ids are written
// in ascending order by an ordered compaction; an exact tie at the threshold
// goes to the lower ids.
#include <algorithm>

#include "pkv_dev.cuh"

namespace pkv {
namespace {

constexpr int kScoreBlocks = 32;   // blocks a CTA: a lane each
constexpr int kScoreThreads = 256;
constexpr int kPStride = kIdxDim + 1;  // float stride of a staged pooled row
constexpr int kMaxQHeads = 64;

__global__ void __launch_bounds__(kScoreThreads)
    scores_kernel(const __grid_constant__ Common c, const uint16_t *__restrict__ qi,
                  float *__restrict__ scores, int32_t ld, int32_t tiles_per_seq) {
    __shared__ float ps[kScoreBlocks * kPStride];
    __shared__ int64_t prow[kScoreBlocks];  // each block's pooled row (-1 past the end)
    extern __shared__ float qs[];  // [n_q_heads][Di]
    pdl_wait();
    pdl_trigger();
    const int s = blockIdx.x / tiles_per_seq;
    const int b0 = (blockIdx.x - s * tiles_per_seq) * kScoreBlocks;
    const SeqDev &sd = c.seq[s];
    const int nb = sd.len / 4;
    const int H = c.n_kv_heads, Di = c.idx_dim, Hq = c.n_q_heads;
    const int tid = threadIdx.x;
    // pooled rows of blocks b0 .. b0+63: one lookup per block, then the rows
    if (tid < kScoreBlocks) {
        const int b = b0 + tid;
        int64_t off = -1;
        if (b < nb) {
            int32_t row;
            const int64_t page = page_start(sd, 4 * b, &row, c.status);
            off = page + off_p_f(c.kv_fp8, H, Di, sd.ptok, row / 4);
        }
        prow[tid] = off;
    }
    // indexer queries of this stream's one decode token, 8 a thread and load
    {
        const uint4 *src = reinterpret_cast<const uint4 *>(qi + (int64_t)sd.tok_off * Hq * Di);
        for (int i = tid; i < Hq * Di / 8; i += kScoreThreads) {
            const uint4 w = __ldg(src + i);
            const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 8; ++e)
                qs[8 * i + e] = __uint_as_float((e & 1) ? (u[e / 2] & 0xffff0000u) : (u[e / 2] << 16));
        }
    }
    __syncthreads();
    // the 64 pooled rows, 16 bytes a load and every load in flight at once
    constexpr int kLoads = kScoreBlocks * (kIdxDim / 8) / kScoreThreads;  // 2
    uint4 w[kLoads];
#pragma unroll
    for (int it = 0; it < kLoads; ++it) {
        const int i = tid + it * kScoreThreads, bl = i >> 4, c16 = i & 15;
        const int64_t off = prow[bl];
        w[it] = off >= 0 ? __ldg(reinterpret_cast<const uint4 *>(sd.layer_base + off) + c16)
                         : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int it = 0; it < kLoads; ++it) {
        const int i = tid + it * kScoreThreads, bl = i >> 4, c16 = i & 15;
        const uint32_t u[4] = {w[it].x, w[it].y, w[it].z, w[it].w};
#pragma unroll
        for (int e = 0; e < 8; ++e)
            ps[bl * kPStride + 8 * c16 + e] =
                __uint_as_float((e & 1) ? (u[e / 2] & 0xffff0000u) : (u[e / 2] << 16));
    }
    __syncthreads();
    const int lane = tid & 31, warp = tid >> 5;
    // a warp takes heads h and h + 8, each lane block lane of the tile: two
    // chains side by side, each still summed in d order
    const float *pa = ps + lane * kPStride;
    for (int h = warp; h < Hq; h += 2 * (kScoreThreads / 32)) {
        const int h2 = h + kScoreThreads / 32;
        const bool two = h2 < Hq;
        const float *qa = qs + h * Di, *qb = qs + (two ? h2 : h) * Di;
        float a0 = 0.f, a1 = 0.f;
#pragma unroll 8
        for (int d = 0; d < kIdxDim; ++d) {
            const float u = pa[d];
            a0 = __fmaf_rn(qa[d], u, a0);
            a1 = __fmaf_rn(qb[d], u, a1);
        }
        const int ba = b0 + lane;
        if (ba < ld) {
            scores[((int64_t)s * Hq + h) * ld + ba] = ba < nb ? a0 : -INFINITY;
            if (two) scores[((int64_t)s * Hq + h2) * ld + ba] = ba < nb ? a1 : -INFINITY;
        }
    }
}

constexpr int kTopThreads = 256;
constexpr int kTopSmemKeys = 12288;  // order keys of a row held in shared memory (48 KB)
constexpr int kTopBins = 2048;       // the first histogram: the keys' top 11 bits
constexpr int kTopCand = 512;        // keys of the threshold bin ranked directly
static_assert(kTopBins % kTopThreads == 0, "a thread sums whole groups of bins");

__device__ __forceinline__ uint32_t order_key(float x) {
    uint32_t u = __float_as_uint(x);
    if (u == 0x80000000u) u = 0;  // -0 ranks with +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide exclusive prefix sum of one value per thread; returns the total.
__device__ __forceinline__ int block_exclusive_scan(int v, int *excl, int *warp_tot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int t = lane < kTopThreads / 32 ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        if (lane < kTopThreads / 32) warp_tot[lane] = t;  // inclusive
    }
    __syncthreads();
    const int before = warp ? warp_tot[warp - 1] : 0;
    *excl = before + x - v;
    const int total = warp_tot[kTopThreads / 32 - 1];
    __syncthreads();
    return total;
}

// The same for two values a thread at once (one pass of barriers).
__device__ __forceinline__ void block_exclusive_scan2(int v0, int v1, int *excl0, int *excl1,
                                                      int2 *warp_tot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x0 = v0, x1 = v1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y0 = __shfl_up_sync(0xffffffffu, x0, o);
        const int y1 = __shfl_up_sync(0xffffffffu, x1, o);
        if (lane >= o) {
            x0 += y0;
            x1 += y1;
        }
    }
    if (lane == 31) warp_tot[warp] = make_int2(x0, x1);
    __syncthreads();
    if (warp == 0) {
        int2 t = lane < kTopThreads / 32 ? warp_tot[lane] : make_int2(0, 0);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y0 = __shfl_up_sync(0xffffffffu, t.x, o);
            const int y1 = __shfl_up_sync(0xffffffffu, t.y, o);
            if (lane >= o) {
                t.x += y0;
                t.y += y1;
            }
        }
        if (lane < kTopThreads / 32) warp_tot[lane] = t;  // inclusive
    }
    __syncthreads();
    const int2 before = warp ? warp_tot[warp - 1] : make_int2(0, 0);
    *excl0 = before.x + x0 - v0;
    *excl1 = before.y + x1 - v1;
}

__global__ void __launch_bounds__(kTopThreads)
    topk_kernel(const __grid_constant__ Common c, const float *__restrict__ scores, int32_t ld,
                int32_t k, int32_t *__restrict__ ids, int32_t keys_in_smem) {
    __shared__ int hist[256];
    __shared__ int hist11[kTopBins];      // counts of the keys' top 11 bits
    __shared__ uint32_t cand[kTopCand];   // keys of the threshold bin
    __shared__ int warp_tot[kTopThreads / 32];
    __shared__ int2 warp_tot2[kTopThreads / 32];
    __shared__ uint32_t sh_prefix;
    __shared__ int sh_need, sh_m, sh_cnt;
    extern __shared__ uint32_t skeys[];  // the row's order keys, when it fits
    pdl_wait();
    pdl_trigger();
    const int s = blockIdx.x / c.n_q_heads, h = blockIdx.x - s * c.n_q_heads;
    const int nb = c.seq[s].len / 4;
    const int kk = min(k, nb);
    const float *row = scores + ((int64_t)s * c.n_q_heads + h) * ld;
    int32_t *out = ids + ((int64_t)s * c.n_q_heads + h) * k;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool in_smem = keys_in_smem != 0;  // the launch sized the array for every row
    auto key_of = [&](int b) -> uint32_t { return in_smem ? skeys[b] : order_key(row[b]); };

    // The threshold key T with count(key > T) < kk <= count(key >= T), and
    // `need`, the number of keys equal to T to take.  First the top 11 bits:
    // one histogram and a block-wide suffix count find the bin holding T;
    // when that bin holds at most kTopCand keys, T is the one of them with
    // the right rank among them.  Otherwise an 8-bit radix select over all
    // 32 bits finds it.
    uint32_t prefix = 0, mask = 0;
    int need = kk;  // selected elements still to find inside the current prefix
    bool found = false;
    if (kk > 0) {
        for (int i = tid; i < kTopBins; i += kTopThreads) hist11[i] = 0;
        if (tid == 0) sh_cnt = 0;
        __syncthreads();
        // the row's order keys (kept when they fit) and their histogram; a
        // 16-byte-aligned row is read four scores a load, a thread's loads of
        // a pass all in flight before the first is used
        auto take = [&](int b, float x) {
            const uint32_t key = order_key(x);
            if (in_smem) skeys[b] = key;
            atomicAdd(&hist11[key >> 21], 1);
        };
        const int n4 = (reinterpret_cast<uintptr_t>(row) & 15u) == 0 ? nb >> 2 : 0;
        const float4 *row4 = reinterpret_cast<const float4 *>(row);
        constexpr int kLoads = 4;
        for (int i0 = 0; i0 < n4; i0 += kLoads * kTopThreads) {
            float4 v[kLoads];
#pragma unroll
            for (int u = 0; u < kLoads; ++u) {
                const int i = i0 + u * kTopThreads + tid;
                v[u] = i < n4 ? row4[i] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < kLoads; ++u) {
                const int i = i0 + u * kTopThreads + tid;
                if (i < n4) {
                    take(4 * i, v[u].x);
                    take(4 * i + 1, v[u].y);
                    take(4 * i + 2, v[u].z);
                    take(4 * i + 3, v[u].w);
                }
            }
        }
        for (int b = 4 * n4 + tid; b < nb; b += kTopThreads) take(b, row[b]);
        __syncthreads();
        // thread t: bins 2047 - 8t down to 2040 - 8t (descending keys)
        constexpr int per = kTopBins / kTopThreads;
        int own = 0;
#pragma unroll
        for (int i = 0; i < per; ++i) own += hist11[kTopBins - 1 - (per * tid + i)];
        int above;  // keys in higher bins
        block_exclusive_scan(own, &above, warp_tot);
        if (above < need && need <= above + own) {  // the threshold bin is one of this thread's
            int acc = above;
            for (int i = 0; i < per; ++i) {
                const int bin = kTopBins - 1 - (per * tid + i);
                if (acc + hist11[bin] >= need) {
                    sh_prefix = static_cast<uint32_t>(bin);
                    sh_need = need - acc;
                    sh_m = hist11[bin];
                    break;
                }
                acc += hist11[bin];
            }
        }
        __syncthreads();
        const uint32_t bin = sh_prefix;
        const int need1 = sh_need, m = sh_m;
        if (m <= kTopCand) {
            for (int b = tid; b < nb; b += kTopThreads) {
                const uint32_t key = key_of(b);
                if ((key >> 21) == bin) cand[atomicAdd(&sh_cnt, 1)] = key;
            }
            __syncthreads();
            if (m <= 64) {
                // one warp sorts the bin's keys, two a lane, into descending
                // order (a bitonic network; padding 0 sorts below every key or
                // equals it), then T is the need1-th
                if (warp == 0) {
                    uint32_t v[2] = {lane < m ? cand[lane] : 0u, lane + 32 < m ? cand[lane + 32] : 0u};
#pragma unroll
                    for (int k2 = 2; k2 <= 64; k2 <<= 1) {
#pragma unroll
                        for (int j = k2 >> 1; j > 0; j >>= 1) {
                            uint32_t p[2];
#pragma unroll
                            for (int r = 0; r < 2; ++r)
                                p[r] = j == 32 ? v[1 - r] : __shfl_xor_sync(0xffffffffu, v[r], j);
#pragma unroll
                            for (int r = 0; r < 2; ++r) {
                                const int i = lane + 32 * r;
                                const bool keep_min = ((i & k2) == 0) != ((i & j) == 0);
                                v[r] = keep_min ? min(v[r], p[r]) : max(v[r], p[r]);
                            }
                        }
                    }
                    const int at = need1 - 1;  // 0 .. m-1
                    const uint32_t t = __shfl_sync(0xffffffffu, at < 32 ? v[0] : v[1], at & 31);
                    const int gt = __popc(__ballot_sync(0xffffffffu, v[0] > t)) +
                                   __popc(__ballot_sync(0xffffffffu, v[1] > t));
                    if (lane == 0) {
                        sh_prefix = t;
                        sh_need = need1 - gt;
                    }
                }
            } else {
                // T: the candidate with fewer than need1 larger candidates and at
                // least need1 at or above it (equal keys write the same values)
                for (int i = tid; i < m; i += kTopThreads) {
                    const uint32_t x = cand[i];
                    int gt = 0, ge = 0;
                    for (int j = 0; j < m; ++j) {
                        const uint32_t y = cand[j];
                        gt += y > x;
                        ge += y >= x;
                    }
                    if (gt < need1 && need1 <= ge) {
                        sh_prefix = x;
                        sh_need = need1 - gt;
                    }
                }
            }
            __syncthreads();
            prefix = sh_prefix;
            need = sh_need;
            found = true;
        }
        __syncthreads();  // every thread has read sh_prefix and sh_need
    }
    if (kk > 0 && !found) {
        for (int shift = 24; shift >= 0; shift -= 8) {
            for (int i = tid; i < 256; i += kTopThreads) hist[i] = 0;
            __syncthreads();
            for (int b = tid; b < nb; b += kTopThreads) {
                const uint32_t key = key_of(b);
                if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
            }
            __syncthreads();
            if (warp == 0) {
                // lane l holds digits 8l .. 8l+7; counts above each lane by a suffix sum
                int own = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) own += hist[8 * lane + i];
                int incl = own;  // keys with a digit >= 8 * lane
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_down_sync(0xffffffffu, incl, o);
                    if (lane + o < 32) incl += y;
                }
                const int above = incl - own;
                if (above < need && need <= incl) {  // the threshold digit is this lane's
                    int acc = above, digit = 8 * lane + 7;
                    for (; digit > 8 * lane; --digit) {
                        if (acc + hist[digit] >= need) break;
                        acc += hist[digit];
                    }
                    sh_prefix = prefix | (static_cast<uint32_t>(digit) << shift);
                    sh_need = need - acc;
                }
            }
            __syncthreads();
            prefix = sh_prefix;
            need = sh_need;
            mask |= 255u << shift;
            __syncthreads();
        }
    }
    const uint32_t T = prefix;  // threshold key; `need` of the keys equal to T are taken
    // ordered compaction over ids: thread t owns the contiguous ids [t*chunk, ..)
    const int chunk = (nb + kTopThreads - 1) / kTopThreads;
    const int lo = min(nb, tid * chunk), hi = min(nb, lo + chunk);
    int eq = 0, gt = 0;
    if (kk > 0)
        for (int b = lo; b < hi; ++b) {
            const uint32_t key = key_of(b);
            eq += key == T;
            gt += key > T;
        }
    // keys equal to T are taken in id order, so the threads before this one
    // took min(eq_before, need) of them
    int eq_before, gt_before;
    block_exclusive_scan2(eq, gt, &eq_before, &gt_before, warp_tot2);
    if (kk > 0) {
        int e = eq_before, o = gt_before + min(eq_before, need);
        for (int b = lo; b < hi; ++b) {
            const uint32_t key = key_of(b);
            if (key > T) out[o++] = b;
            else if (key == T && e++ < need) out[o++] = b;
        }
    }
    for (int i = kk + tid; i < k; i += kTopThreads) out[i] = -1;
}

}  // namespace

int launch_scores(const Common &c, float *scores, int32_t ld, const uint16_t *qi, int32_t max_nb,
                  cudaStream_t stream) {
    if (c.n_q_heads > kMaxQHeads) return PKV_EINVAL;
    (void)max_nb;
    const int tiles = (ld + kScoreBlocks - 1) / kScoreBlocks;
    const size_t dyn = static_cast<size_t>(c.n_q_heads) * c.idx_dim * sizeof(float);
    static std::atomic<uint64_t> attr_done{0};
    if (once_per_device(attr_done, [] {
            return cuda_rc(cudaFuncSetAttribute(
                scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                kMaxQHeads * kIdxDim * static_cast<int>(sizeof(float))));
        }) != PKV_OK)
        return PKV_ECUDA;
    return launch_status(launch_pdl(scores_kernel, c.n_seqs * tiles, kScoreThreads, dyn, stream,
                                    c, qi, scores, ld, tiles));
}

int launch_topk(const Common &c, const float *scores, int32_t ld, int32_t k, int32_t *ids,
                cudaStream_t stream) {
    int max_nb = 0;
    for (int s = 0; s < c.n_seqs; ++s) max_nb = std::max(max_nb, c.seq[s].len / 4);
    const bool in_smem = max_nb <= kTopSmemKeys;
    const size_t dyn = in_smem ? static_cast<size_t>(max_nb) * 4 : 0;
    static std::atomic<uint64_t> attr_done{0};
    if (once_per_device(attr_done, [] {
            return cuda_rc(cudaFuncSetAttribute(topk_kernel,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                kTopSmemKeys * 4));
        }) != PKV_OK)
        return PKV_ECUDA;
    return launch_status(launch_pdl(topk_kernel, c.n_seqs * c.n_q_heads, kTopThreads, dyn, stream,
                                    c, scores, ld, k, ids, static_cast<int32_t>(in_smem)));
}

}  // namespace pkv
