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
// Top-k: one CTA per (stream, head) runs the block-wide selection of
// pkv_topk.cuh (a threshold by histogram, sort, ranking or radix select, then
// an ordered compaction; exact ties go to the lower ids), with the row's
// order keys in shared memory when the longest row fits.
#include <algorithm>

#include "pkv_dev.cuh"
#include "pkv_topk.cuh"

namespace pkv {
namespace {

constexpr int kScoreBlocks = 32;   // blocks a CTA: a lane each
constexpr int kScoreThreads = 256;
// float stride of a staged pooled row: 16-byte rows whose lanes' 16-byte
// loads spread over the banks (528 B apart)
constexpr int kPStride = kIdxDim + 4;
constexpr int kMaxQHeads = 64;

// Four bf16 values (two packed words, low half first) as floats: exact.
__device__ __forceinline__ float4 bf16x4_to_float4(uint32_t u0, uint32_t u1) {
    return make_float4(__uint_as_float(u0 << 16), __uint_as_float(u0 & 0xffff0000u),
                       __uint_as_float(u1 << 16), __uint_as_float(u1 & 0xffff0000u));
}

__global__ void __launch_bounds__(kScoreThreads, 1)
    scores_kernel(const __grid_constant__ Common c, const uint16_t *__restrict__ qi,
                  float *__restrict__ scores, int32_t ld, int32_t tiles_per_seq) {
    __shared__ __align__(16) float ps[kScoreBlocks * kPStride];
    __shared__ int64_t prow[kScoreBlocks];  // each block's pooled row (-1 past the end)
    extern __shared__ float4 qs4[];  // [n_q_heads][Di / 4]
    const int s = blockIdx.x / tiles_per_seq;
    const int b0 = (blockIdx.x - s * tiles_per_seq) * kScoreBlocks;
    const SeqDev &sd = c.seq[s];
    const int nb = sd.len / 4;
    const int H = c.n_kv_heads, Di = c.idx_dim, Hq = c.n_q_heads;
    const int tid = threadIdx.x;
    // pooled rows of blocks b0 .. b0+63: one lookup per block.  The launch
    // parameters and the page table are not written by the kernels before
    // this one, so the lookups run before the grid-dependency wait; the
    // pooled rows and the queries (which those kernels write) after it.
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
    pdl_wait();
    pdl_trigger();
    // indexer queries of this stream's one decode token, 8 a thread and load
    {
        const uint4 *src = reinterpret_cast<const uint4 *>(qi + (int64_t)sd.tok_off * Hq * Di);
        for (int i = tid; i < Hq * Di / 8; i += kScoreThreads) {
            const uint4 w = __ldg(src + i);
            qs4[2 * i] = bf16x4_to_float4(w.x, w.y);
            qs4[2 * i + 1] = bf16x4_to_float4(w.z, w.w);
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
        float4 *dst = reinterpret_cast<float4 *>(ps + bl * kPStride + 8 * c16);
        dst[0] = bf16x4_to_float4(w[it].x, w[it].y);
        dst[1] = bf16x4_to_float4(w[it].z, w[it].w);
    }
    __syncthreads();
    const int lane = tid & 31, warp = tid >> 5;
    // a warp takes heads h and h + 8, each lane block lane of the tile: two
    // chains side by side, each still summed in d order
    // (four dims a shared-memory load, each chain still taken in d order)
    const float4 *pa = reinterpret_cast<const float4 *>(ps + lane * kPStride);
    for (int h = warp; h < Hq; h += 2 * (kScoreThreads / 32)) {
        const int h2 = h + kScoreThreads / 32;
        const bool two = h2 < Hq;
        const float4 *qa = qs4 + h * (kIdxDim / 4), *qb = qs4 + (two ? h2 : h) * (kIdxDim / 4);
        float a0 = 0.f, a1 = 0.f;
#pragma unroll 4
        for (int d4 = 0; d4 < kIdxDim / 4; ++d4) {
            const float4 u = pa[d4], x = qa[d4], y = qb[d4];
            a0 = __fmaf_rn(x.x, u.x, a0);
            a1 = __fmaf_rn(y.x, u.x, a1);
            a0 = __fmaf_rn(x.y, u.y, a0);
            a1 = __fmaf_rn(y.y, u.y, a1);
            a0 = __fmaf_rn(x.z, u.z, a0);
            a1 = __fmaf_rn(y.z, u.z, a1);
            a0 = __fmaf_rn(x.w, u.w, a0);
            a1 = __fmaf_rn(y.w, u.w, a1);
        }
        const int ba = b0 + lane;
        if (ba < ld) {
            scores[((int64_t)s * Hq + h) * ld + ba] = ba < nb ? a0 : -INFINITY;
            if (two) scores[((int64_t)s * Hq + h2) * ld + ba] = ba < nb ? a1 : -INFINITY;
        }
    }
}

constexpr int kTopSmemKeys = 12288;  // order keys of a row held in shared memory (48 KB)

__global__ void __launch_bounds__(kTopThreads)
    topk_kernel(const __grid_constant__ Common c, const float *__restrict__ scores, int32_t ld,
                int32_t k, int32_t *__restrict__ ids, int32_t keys_in_smem) {
    __shared__ int hist[256];
    __shared__ int hist11[kTopBins];
    __shared__ uint32_t cand[kTopCand];
    __shared__ int warp_tot[kTopThreads / 32];
    __shared__ int2 warp_tot2[kTopThreads / 32];
    __shared__ int vars[4];
    extern __shared__ uint32_t skeys[];  // the row's order keys, when it fits
    // the row and its length from the launch parameters before the wait (an
    // asm use the compiler cannot move past it): only the scores wait
    const int s = blockIdx.x / c.n_q_heads, h = blockIdx.x - s * c.n_q_heads;
    const int nb = c.seq[s].len / 4;
    const float *row = scores + ((int64_t)s * c.n_q_heads + h) * ld;
    int32_t *out = ids + ((int64_t)s * c.n_q_heads + h) * k;
    asm volatile("" ::"r"(nb), "l"(row), "l"(out));
    pdl_wait();
    pdl_trigger();
    // the launch sized the key array for every row, or gave it none
    const TopkSmem sm{hist, hist11, cand, warp_tot, warp_tot2, vars,
                      keys_in_smem != 0 ? skeys : nullptr};
    topk_block(row, nb, k, out, sm);
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
