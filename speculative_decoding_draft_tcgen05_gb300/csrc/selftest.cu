// Self-test of the bounded pipeline wait that every tcgen05/TMA kernel of the
// library uses: a one-warp kernel waits on an mbarrier that nothing will ever
// complete, gives up after the wait's time bound, and reports it in the same
// device error bits the kernels latch. The host can check that the wait ends,
// that the bit arrives and that the context stays usable, without a broken
// pipeline and without faulting the GPU.
#include "common.cuh"
#include "dflash_select.h"
#include "kernels.h"

namespace dfl {
dflash_status host_fail(dflash_status st, const char *msg);
}  // namespace dfl

namespace {

__global__ void wait_timeout_kernel(int *status)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        dfl::mbar_init(dfl::smem_u32(&bar), 1);  // expects one arrival; none is ever made
        abort_flag = 0;
        dfl::fence_mbar_init();
    }
    __syncwarp();
    if (threadIdx.x == 0 && !dfl::mbar_wait(dfl::smem_u32(&bar), 0, &abort_flag)) atomicOr(status, dfl::DEV_ERR_TIMEOUT);
}

}  // namespace

extern "C" dflash_status dflash_selftest_wait_timeout(int32_t *device_status, void *stream)
{
    if (!device_status) return dfl::host_fail(DFLASH_ERR_INVALID_ARG, "device_status must not be NULL");
    wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(device_status);
    if (cudaGetLastError() != cudaSuccess) return dfl::host_fail(DFLASH_ERR_CUDA, "self-test launch failed");
    return DFLASH_OK;
}
