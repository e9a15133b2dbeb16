// Failure-detection self-tests: the bounded wait used by every role of the
// attention kernels (device side of vitfp8_selftest_bounded_wait), and the
// checked build's bounds check (vitfp8_selftest_bounds_check).
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

// Self-test of the checked build's bounds check: one thread asks VF_IN
// whether element 16 of a 16-element buffer may be accessed.  The buffer is
// only named, never touched: in the checked build the check refuses and
// records VITFP8_ERR_DEVICE_BOUNDS, so the access it guards is skipped; in
// the normal build the check is compiled away and nothing is recorded.
__global__ void selftest_bounds_kernel(WsHeader* ws) {
    ws->error = 0;
    const int64_t n = 16;
    (void)n;   // the normal build compiles the checks away
    if (VF_IN(n, 1, n, &ws->error)) {
        // The access a failed check would skip (none here).
    }
    if (VF_IN(0, 1, n, &ws->error)) {
        // In range: nothing is recorded.
    }
}

cudaError_t launch_selftest_bounds(void* ws, cudaStream_t s) {
    selftest_bounds_kernel<<<1, 1, 0, s>>>(static_cast<WsHeader*>(ws));
    return cudaGetLastError();
}

}  // namespace vitfp8
