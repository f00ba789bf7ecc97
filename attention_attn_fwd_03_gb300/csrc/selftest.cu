// selftest.cu -- two small kernels that check the device rather than compute
// attention.
//
// selftest_timeout_kernel: failure handling without a GPU fault.  One thread
// waits, through the same bounded wait every attention kernel uses
// (attn::wait_bar), on a shared-memory barrier that nothing ever completes.
// After the wait limit it records ATTN_ERR_TIMEOUT in the device status word
// and returns, as a stalled attention kernel's waits would: no trap, no
// fault, and the context stays usable.
//
// selftest_mma_rate_kernel: the dense tensor-core rate per SM, measured.  One
// CTA per SM; one thread issues a stream of 128x128x16 bf16 tcgen05.mma
// (both operands in shared memory, the fp32 accumulator in tensor memory,
// every MMA accumulating into it -- the pattern of the attention kernels'
// S = Q K^T) and times them with the SM cycle counter.  SMs x FLOP per SM
// cycle x SM clock is the dense bf16 peak the attention kernels are held to.
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

constexpr int kRateSmem = 120 * 1024;  // more than half an SM's shared memory: one CTA per SM
constexpr int kRatePanel = 128 * 128;  // 128 rows x 128 B, one 128-byte-swizzled operand panel

__global__ void __launch_bounds__(128, 1) selftest_mma_rate_kernel(int n_groups, unsigned long long* cycles,
                                                                   unsigned* status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t done;
    __shared__ uint32_t tmem_holder;
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5;
    // operands: A and B panels of bf16 values in [1, 2) (any finite values do)
    for (int i = threadIdx.x; i < 2 * kRatePanel / 4; i += blockDim.x)
        reinterpret_cast<uint32_t*>(smem)[i] = 0x3F803F80u + ((uint32_t)(i * 2654435761u) & 0x007F007Fu);
    fence_async_smem();
    if (threadIdx.x == 0) {
        bar_init(&done, 1);
        abort_flag = 0;
        bar_init_fence();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_holder, 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_holder;
    if (threadIdx.x == 0) {
        const uint32_t base = smem_u32(smem);
        const uint64_t a = sdesc_sw128(base, 16, 1024);
        const uint64_t b = sdesc_sw128(base + kRatePanel, 16, 1024);
        constexpr uint32_t idesc = idesc_make(128, 128, 1u, false, false);
        // warm-up: 64 MMAs, completed before the clock starts
        for (int g = 0; g < 16; ++g) mma4_ss<2, 4, 6, 2, 4, 6, false>(tmem, a, b, idesc, g > 0 ? 1u : 0u);
        tc_commit(&done);
        bool ok = wait_bar(&done, 0u, &abort_flag, status);
        const unsigned long long t0 = clock64();
        for (int g = 0; ok && g < n_groups; ++g) mma4_ss<2, 4, 6, 2, 4, 6, false>(tmem, a, b, idesc, 1u);
        tc_commit(&done);
        ok = ok && wait_bar(&done, 1u, &abort_flag, status);
        const unsigned long long t1 = clock64();
        cycles[blockIdx.x] = ok ? t1 - t0 : 0ull;
        if (!ok) drain_wait(&done, 1u, status);  // every MMA done before tensor memory is freed
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 128);
    }
}

}  // namespace

cudaError_t launch_selftest_timeout(unsigned* status, cudaStream_t stream) {
    selftest_timeout_kernel<<<1, 32, 0, stream>>>(status);
    return cudaGetLastError();
}

cudaError_t launch_selftest_mma_rate(int n_ctas, int n_groups, unsigned long long* cycles, unsigned* status,
                                     cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(selftest_mma_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kRateSmem + 1024);
    if (e != cudaSuccess) return e;
    selftest_mma_rate_kernel<<<n_ctas, 128, kRateSmem + 1024, stream>>>(n_groups, cycles, status);
    return cudaGetLastError();
}

}  // namespace attn
