// selftest.cu -- a kernel for testing failure handling without a GPU fault.
//
// One thread waits, through the same bounded wait every attention kernel
// uses (attn::wait_bar), on a shared-memory barrier that nothing ever
// completes.  After the wait limit it records ATTN_ERR_TIMEOUT in the device
// status word and returns, as a stalled attention kernel's waits would: no
// trap, no fault, and the context stays usable.
#include "kernels.h"
#include "ptx.cuh"

namespace attn {

namespace {

__global__ void __launch_bounds__(32) selftest_timeout_kernel(unsigned* status) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        bar_init(&bar, 1);
        abort_flag = 0;
        bar_init_fence();
    }
    __syncwarp();
    if (threadIdx.x == 0) (void)wait_bar(&bar, 0u, &abort_flag, status);  // phase 0 never completes
}

}  // namespace

cudaError_t launch_selftest_timeout(unsigned* status, cudaStream_t stream) {
    selftest_timeout_kernel<<<1, 32, 0, stream>>>(status);
    return cudaGetLastError();
}

}  // namespace attn
