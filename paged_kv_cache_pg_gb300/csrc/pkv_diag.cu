// Diagnostics: a pipeline wait that runs out.  One warp waits on a shared
// memory barrier that nothing arrives on, with the same bounded wait every
// kernel of the library uses: it gives up after its time limit, ORs
// PKV_DEV_TIMEOUT into the status word and returns, so the GPU and the
// context stay usable.
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

}  // namespace
}  // namespace pkv

extern "C" int pkv_diag_wait_runs_out(int32_t *dev_status, cudaStream_t stream) {
    if (!dev_status) return PKV_EINVAL;
    pkv::wait_runs_out_kernel<<<1, 32, 0, stream>>>(reinterpret_cast<uint32_t *>(dev_status));
    return pkv::launch_status(cudaGetLastError());
}
