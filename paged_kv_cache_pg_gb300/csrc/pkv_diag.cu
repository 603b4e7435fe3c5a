// Diagnostics: pipeline waits that run out.  One warp waits on a shared
// memory barrier that nothing arrives on, with the same bounded wait every
// kernel of the library uses: it gives up after its time limit, ORs
// PKV_DEV_TIMEOUT into the status word and returns, so the GPU and the
// context stay usable.  A second launch does the same inside a whole CTA
// with the decode's stage barriers, where one slice's copy never lands.
#include "pkv_dev.cuh"

namespace pkv {
namespace {

__global__ void wait_runs_out_kernel(uint32_t *status) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    mbar_wait(&bar, 0, threadIdx.x == 0 ? status : nullptr);  // nothing arrives on `bar`
}

// A whole CTA shaped like the decode's partial CTA: eight warps in four key
// slices of two warps, twelve stage slots (three a slice) with a full and an
// empty barrier each.  A slice's lead warp "stages" a tile by arriving on its
// full barrier (an arrival stands for a landed copy; nothing is copied), both
// warps of the slice wait on it, release the slot on its empty barrier, and
// the lead warp refills the slot once both released it, for eight tiles a
// slice.  The lead warp of slice `withheld` never arrives for that slice's
// second tile.  Its two warps' waits run out (PKV_DEV_TIMEOUT), they set the
// CTA's abort flag and leave their loop; the other slices finish theirs; the
// whole CTA then meets at the barrier the decode meets at after its loop
// and returns.
__global__ void __launch_bounds__(256) cta_wait_runs_out_kernel(uint32_t *status, int withheld) {
    constexpr int kS = 3, kSlices = 4, kTiles = 8;
    __shared__ uint64_t full[kS * kSlices], empty[kS * kSlices];
    __shared__ volatile int abort_flag;
    const int tid = threadIdx.x, lane = tid & 31;
    const int dh = (tid >> 5) & 1, ks = tid >> 6;
    const bool leader = dh == 0;
    if (tid == 0) {
        for (int i = 0; i < kS * kSlices; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 2);
        }
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    auto stage = [&](int j) {
        if (lane == 0 && !(ks == withheld && j == 1)) mbar_arrive(&full[ks * kS + j % kS]);
    };
    int issued = 0;
    if (leader)
        for (; issued < kS; ++issued) stage(issued);
    for (int j = 0; j < kTiles; ++j) {
        const int slot = ks * kS + j % kS;
        if (!mbar_wait(&full[slot], (j / kS) & 1, status)) {
            abort_flag = 1;
            break;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        if (leader && issued < kTiles) {
            if (!mbar_wait(&empty[slot], (j / kS) & 1, status)) {
                abort_flag = 1;
                break;
            }
            stage(issued);
            ++issued;
        }
    }
    __syncthreads();
    if (abort_flag) return;
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_diag_cta_wait_runs_out(int32_t *dev_status, int32_t withheld_slice,
                                          cudaStream_t stream) {
    if (!dev_status || withheld_slice < 0 || withheld_slice > 3) return PKV_EINVAL;
    pkv::cta_wait_runs_out_kernel<<<1, 256, 0, stream>>>(reinterpret_cast<uint32_t *>(dev_status),
                                                         withheld_slice);
    return pkv::launch_status(cudaGetLastError());
}

extern "C" int pkv_diag_wait_runs_out(int32_t *dev_status, cudaStream_t stream) {
    if (!dev_status) return PKV_EINVAL;
    pkv::wait_runs_out_kernel<<<1, 32, 0, stream>>>(reinterpret_cast<uint32_t *>(dev_status));
    return pkv::launch_status(cudaGetLastError());
}
