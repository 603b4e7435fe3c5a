// Block scores over pooled rows and top-k block selection.
//
// Scores: one thread per (head, block) runs the float32 chain
// acc = fmaf(qi[d], P[b][d], acc), d = 0 .. Di-1 (the order is part of the
// result: a top-k decision downstream must see the same bits on any cache
// layout).  Pooled rows are looked up once per block (pg_at on its first
// position) and staged in shared memory.
//
// Top-k: one CTA per (stream, head) finds the k-th largest score by an 8-bit
// radix select on order-preserving keys, then writes the selected block ids
// in ascending order with an ordered compaction; an exact tie at the
// threshold goes to the lower ids.
#include "pkv_dev.cuh"

namespace pkv {
namespace {

constexpr int kScoreBlocks = 64;   // blocks a CTA
constexpr int kScoreThreads = 256;
constexpr int kPStride = kIdxDim + 1;  // float stride of a staged pooled row
constexpr int kMaxQHeads = 64;

__global__ void __launch_bounds__(kScoreThreads)
    scores_kernel(const __grid_constant__ Common c, const uint16_t *__restrict__ qi,
                  float *__restrict__ scores, int32_t ld, int32_t tiles_per_seq) {
    __shared__ float ps[kScoreBlocks * kPStride];
    extern __shared__ float qs[];  // [n_q_heads][Di]
    pdl_wait();
    pdl_trigger();
    const int s = blockIdx.x / tiles_per_seq;
    const int b0 = (blockIdx.x - s * tiles_per_seq) * kScoreBlocks;
    const SeqDev &sd = c.seq[s];
    const int nb = sd.len / 4;
    const int H = c.n_kv_heads, Di = c.idx_dim, Hq = c.n_q_heads;
    const int tid = threadIdx.x;
    // indexer queries of this stream's one decode token
    for (int i = tid; i < Hq * Di; i += kScoreThreads)
        qs[i] = __uint_as_float(static_cast<uint32_t>(qi[(int64_t)sd.tok_off * Hq * Di + i]) << 16);
    // pooled rows of blocks b0 .. b0+63: one lookup per block
    for (int i = tid; i < kScoreBlocks * (kIdxDim / 2); i += kScoreThreads) {
        const int bl = i / (kIdxDim / 2), d2 = i - bl * (kIdxDim / 2);
        const int b = b0 + bl;
        float lo = 0.f, hi = 0.f;
        if (b < nb) {
            int32_t row;
            const int64_t page = page_start(sd, 4 * b, &row, c.status);
            const uint32_t w = *reinterpret_cast<const uint32_t *>(
                sd.layer_base + page + off_p_f(c.kv_fp8, H, Di, sd.ptok, row / 4) + 2 * d2);
            lo = __uint_as_float(w << 16);
            hi = __uint_as_float(w & 0xffff0000u);
        }
        ps[bl * kPStride + 2 * d2] = lo;
        ps[bl * kPStride + 2 * d2 + 1] = hi;
    }
    __syncthreads();
    const int lane = tid & 31, warp = tid >> 5;
    // warps walk heads; each lane owns blocks lane and lane + 32 of the tile
    for (int h = warp; h < Hq; h += kScoreThreads / 32) {
        const float *q = qs + h * Di;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int bl = lane + 32 * half;
            const int b = b0 + bl;
            if (b >= ld) continue;
            float acc = 0.f;
            const float *p = ps + bl * kPStride;
            for (int d = 0; d < kIdxDim; ++d) acc = __fmaf_rn(q[d], p[d], acc);
            scores[((int64_t)s * Hq + h) * ld + b] = b < nb ? acc : -INFINITY;
        }
    }
}

constexpr int kTopThreads = 256;

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

__global__ void __launch_bounds__(kTopThreads)
    topk_kernel(const __grid_constant__ Common c, const float *__restrict__ scores, int32_t ld,
                int32_t k, int32_t *__restrict__ ids) {
    __shared__ int hist[256];
    __shared__ int warp_tot[kTopThreads / 32];
    __shared__ uint32_t sh_prefix;
    __shared__ int sh_need;
    pdl_wait();
    pdl_trigger();
    const int s = blockIdx.x / c.n_q_heads, h = blockIdx.x - s * c.n_q_heads;
    const int nb = c.seq[s].len / 4;
    const int kk = min(k, nb);
    const float *row = scores + ((int64_t)s * c.n_q_heads + h) * ld;
    int32_t *out = ids + ((int64_t)s * c.n_q_heads + h) * k;
    const int tid = threadIdx.x;

    // radix select: the key T with count(key > T) < kk <= count(key >= T)
    uint32_t prefix = 0, mask = 0;
    int need = kk;  // selected elements still to find inside the current prefix
    if (kk > 0) {
        for (int shift = 24; shift >= 0; shift -= 8) {
            for (int i = tid; i < 256; i += kTopThreads) hist[i] = 0;
            __syncthreads();
            for (int b = tid; b < nb; b += kTopThreads) {
                const uint32_t key = order_key(row[b]);
                if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
            }
            __syncthreads();
            if (tid == 0) {
                int acc = 0, digit = 255;
                for (; digit > 0; --digit) {
                    if (acc + hist[digit] >= need) break;
                    acc += hist[digit];
                }
                sh_prefix = prefix | (static_cast<uint32_t>(digit) << shift);
                sh_need = need - acc;
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
    int eq = 0;
    if (kk > 0)
        for (int b = lo; b < hi; ++b) eq += order_key(row[b]) == T;
    int eq_before;
    block_exclusive_scan(eq, &eq_before, warp_tot);
    int sel = 0;
    if (kk > 0) {
        int e = eq_before;
        for (int b = lo; b < hi; ++b) {
            const uint32_t key = order_key(row[b]);
            if (key > T) ++sel;
            else if (key == T && e++ < need) ++sel;
        }
    }
    int sel_before;
    block_exclusive_scan(sel, &sel_before, warp_tot);
    if (kk > 0) {
        int e = eq_before, o = sel_before;
        for (int b = lo; b < hi; ++b) {
            const uint32_t key = order_key(row[b]);
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
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kMaxQHeads * kIdxDim * static_cast<int>(sizeof(float))) !=
            cudaSuccess)
            return PKV_ECUDA;
        attr_set = true;
    }
    return launch_status(launch_pdl(scores_kernel, c.n_seqs * tiles, kScoreThreads, dyn, stream,
                                    c, qi, scores, ld, tiles));
}

int launch_topk(const Common &c, const float *scores, int32_t ld, int32_t k, int32_t *ids,
                cudaStream_t stream) {
    return launch_status(launch_pdl(topk_kernel, c.n_seqs * c.n_q_heads, kTopThreads, 0, stream,
                                    c, scores, ld, k, ids));
}

}  // namespace pkv
