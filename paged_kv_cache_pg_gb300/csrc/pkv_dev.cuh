// Device helpers: pg_at row translation, inline-PTX wrappers for sm_103a
// (mbarrier, bulk async copies, ldmatrix, warp MMA, movmatrix), bounded
// waits and programmatic dependent launch control.
#pragma once

#include <cstdint>
#include <utility>

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "pkv_internal.h"

namespace pkv {

// ---- pg_at (#1169 What this changes; #1170 commit ce5b78d) -----------------
// With no table the old contiguous expression; with a table the start of the
// page holding the position plus the row inside that page.  The branch is
// uniform for a stream, taken once per key per tile by the caller, never per
// load.  A table entry outside [0, n_pages) is reported and replaced by page
// 0, so the read stays inside the arena.
__device__ __forceinline__ int64_t page_start(const SeqDev &s, int32_t pos, int32_t *row,
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
        id = 0;
    }
    return (int64_t)id * s.ps;
}

__device__ __forceinline__ const uint16_t *k_row(const SeqDev &s, int32_t h_kv, int32_t head,
                                                 int32_t pos, uint32_t *status) {
    int32_t row;
    int64_t p = page_start(s, pos, &row, status);
    return s.layer_base + p + off_k(s.ptok, head, row);
}

__device__ __forceinline__ const uint16_t *v_row(const SeqDev &s, int32_t h_kv, int32_t head,
                                                 int32_t pos, uint32_t *status) {
    int32_t row;
    int64_t p = page_start(s, pos, &row, status);
    return s.layer_base + p + off_v(h_kv, s.ptok, head, row);
}

// ---- small PTX wrappers -----------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// A wait that gives up after about a second: it reports PKV_DEV_TIMEOUT and
// returns false instead of hanging the GPU.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t *status) {
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = global_ns();
    for (uint32_t spin = 0;; ++spin) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((spin & 255u) == 255u && global_ns() - t0 > kWaitLimitNs) {
            if (status) atomicOr(status, PKV_DEV_TIMEOUT);
            return false;
        }
    }
}

// Orders this thread's earlier shared-memory accesses before later
// async-proxy (bulk copy, TMA) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// One bulk async copy global -> shared, completing on `bar` (bytes % 16 == 0,
// both addresses 16-byte aligned).  Streamed rows are read once: evict first.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Bulk prefetch of [src, src + bytes) into L2 (bytes % 16 == 0, src 16-byte
// aligned); nothing lands in shared memory and nothing waits on it.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// One 2D TMA tile (64 x 16 bf16 box, 128-byte swizzle) global -> shared.
__device__ __forceinline__ void tma_load_2d(void *dst, const void *map, int x, int y,
                                            uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// One 3D tensor-map box (x, y, z) -> shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(void *dst, const void *map, int x, int y, int z,
                                            uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// 16-byte asynchronous copy global -> shared (L1 bypassed).
__device__ __forceinline__ void cp_async16(void *dst, const void *src, uint64_t policy) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)),
                 "l"(src), "l"(policy)
                 : "memory");
}

// Arrive on `bar` once this thread's earlier cp.async copies have landed
// (the barrier's pending count is raised by one first).
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &a0, uint32_t &a1, uint32_t &a2,
                                        uint32_t &a3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &a0, uint32_t &a1,
                                          uint32_t &a2, uint32_t &a3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                 : "r"(addr));
}

// D (16x8 f32) += A (16x16 bf16, row) * B (16x8 bf16, col)
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float bf16_lo(uint32_t packed) { return __uint_as_float(packed << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t packed) {
    return __uint_as_float(packed & 0xffff0000u);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// e4m3 quantization of one 256-element bf16 row spread over a warp, eight
// elements a lane in row order (#1170, commit 5c09685: a row's e4m3 codes and
// float32 scale; the scale rule is the plainest reading): scale = max|x| / 448,
// code = the e4m3 value nearest x / scale (float32 division with IEEE
// rounding, ties to even, saturating); an all-zero row has scale 0 and codes 0.
// Returns the scale (the same on every lane); *codes gets the lane's 8 codes,
// low byte first.
__device__ __forceinline__ float quantize_row8(const uint4 u, uint2 *codes) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    float x[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
        x[e] = __uint_as_float((e & 1) ? (w[e / 2] & 0xffff0000u) : (w[e / 2] << 16));
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
    for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale = __fdiv_rn(amax, 448.f);
    uint32_t packed[2] = {0u, 0u};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const float q = scale > 0.f ? __fdiv_rn(x[e], scale) : 0.f;
        const uint32_t code = __nv_cvt_float_to_fp8(q, __NV_SATFINITE, __NV_E4M3);
        packed[e / 4] |= code << (8 * (e & 3));
    }
    *codes = make_uint2(packed[0], packed[1]);
    return scale;
}

// Programmatic dependent launch: wait for the previous grid's results, and
// let the next grid start its prologue early.
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Let the next kernel start once this thread's writes are visible device
// wide: for kernels writing cache rows, which the next kernel may read
// before its grid-dependency wait.
__device__ __forceinline__ void pdl_trigger_after_writes() {
    __threadfence();
    pdl_trigger();
}

// A 64-bit value from lane `src` of the warp.
__device__ __forceinline__ int64_t shfl64(int64_t v, int src) {
    const int lo = __shfl_sync(0xffffffffu, static_cast<int>(v), src);
    const int hi = __shfl_sync(0xffffffffu, static_cast<int>(v >> 32), src);
    return (static_cast<int64_t>(hi) << 32) | static_cast<uint32_t>(lo);
}

// Stream of the work item / token: the last s with off(s) <= i.
template <typename F>
__device__ __forceinline__ int find_seq(int n, int32_t i, F off) {
    // four streams' offsets are loaded before any is compared: read from the
    // launch parameters with a computed index, their constant-cache misses
    // then overlap instead of following one another
    int s = 0;
    for (int t0 = 1; t0 < n; t0 += 4) {
        int32_t v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = t0 + k < n ? off(t0 + k) : INT32_MAX;
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (v[k] <= i) s = t0 + k;
    }
    return s;
}

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel on the stream drains; it calls pdl_wait() before
// touching memory that kernel writes.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace pkv
