// Block-wide top-k selection of one row of block scores, for a block of
// kTopThreads threads and shared memory the caller provides.
//
// The k-th largest order key T is found first (one histogram of the keys'
// top 11 bits locates the bin holding it; when that bin holds at most 64 keys
// one warp sorts them, at most 512 all threads rank them, and otherwise an
// 8-bit radix select over all 32 bits finds it); then the keys above T and
// the first keys equal to T, in id order, are written in ascending id order
// by one ordered compaction.  Exact ties therefore go to the lower ids.
#pragma once

#include "pkv_dev.cuh"

namespace pkv {

#ifndef PKV_TOPK_THREADS
#define PKV_TOPK_THREADS 512
#endif
constexpr int kTopThreads = PKV_TOPK_THREADS;
static_assert(kTopThreads % 32 == 0 && kTopThreads <= 1024, "whole warps, at most 32 of them");
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

// The shared memory one selection works in.
struct TopkSmem {
    int *hist;         // [256]
    int *hist11;       // [kTopBins]
    uint32_t *cand;    // [kTopCand]
    int *warp_tot;     // [kTopThreads / 32]
    int2 *warp_tot2;   // [kTopThreads / 32]
    int *vars;         // [4]: threshold bits, keys still to take, bin size, candidates found
    uint32_t *skeys;   // [nb]: the row's order keys, or null to read the row on every pass
};

// Writes the min(k, nb) selected ids of row[0 .. nb-1], ascending, to
// out[0 ..], then -1 up to out[k-1].  Every thread of the block calls it; it
// ends with the writes to `out` issued, not with a barrier.
__device__ __forceinline__ void topk_block(const float *row, int nb, int k, int32_t *out,
                                           const TopkSmem &sm) {
    int *const hist = sm.hist;
    int *const hist11 = sm.hist11;
    uint32_t *const cand = sm.cand;
    int *const warp_tot = sm.warp_tot;
    int2 *const warp_tot2 = sm.warp_tot2;
    uint32_t *const skeys = sm.skeys;
    uint32_t &sh_prefix = reinterpret_cast<uint32_t &>(sm.vars[0]);
    int &sh_need = sm.vars[1];
    int &sh_m = sm.vars[2];
    int &sh_cnt = sm.vars[3];
    const int kk = min(k, nb);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool in_smem = skeys != nullptr;
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

}  // namespace pkv
