// Failure-detection self-test of the bounded wait used by every role of the
// attention kernels (device side of vitfp8_selftest_bounded_wait).
#include <cstdint>
#include <cuda_runtime.h>

#include "attn_common.cuh"
#include "internal.cuh"
#include "ptx.cuh"

namespace vitfp8 {

// Self-test of the bounded wait every role of the attention kernels uses:
// one warp waits on an mbarrier that nothing ever arrives on.  The wait must
// give up after its limit (about half a second), record
// VITFP8_ERR_DEVICE_TIMEOUT in the workspace error word and return, leaving
// the context usable -- the failure is detected, not a hang or a fault.
__global__ void selftest_wait_kernel(WsHeader* ws) {
    __shared__ alignas(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        ws->error = 0;
        abort_flag = 0;
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
    }
    __syncthreads();
    bwait(smem_u32(&bar), 0, &abort_flag, &ws->error);
}

cudaError_t launch_selftest_wait(void* ws, cudaStream_t s) {
    selftest_wait_kernel<<<1, 32, 0, s>>>(static_cast<WsHeader*>(ws));
    return cudaGetLastError();
}

}  // namespace vitfp8
