// selftest.cu -- exercises the bounded device-side wait the kernels use for
// every mbarrier, without faulting or hanging the GPU: one wait on a phase
// that nothing completes (it must give up after the time limit and report a
// timeout), one wait on a phase that completes (it must succeed).
#include "pfkv_internal.cuh"

namespace pfkv {
namespace {

__global__ void selftest_wait_kernel(uint32_t *result) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    // phase 0 of `bar` never completes: no thread arrives
    const bool first = mbar_wait_bounded(&bar, 0);
    __syncwarp();
    // now complete phase 0 and wait for it
    if (threadIdx.x == 0)
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&bar)) : "memory");
    const bool second = mbar_wait_bounded(&bar, 0);
    __syncwarp();
    if (threadIdx.x == 0) *result = (first ? 0u : kStatusTimeout) | (second ? 0x100u : 0u);
}

}  // namespace
}  // namespace pfkv

extern "C" pfkv_status pfkv_selftest_bounded_wait(uint32_t *result, void *stream) {
    if (!result) return PFKV_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(result) & 3u) return PFKV_ERR_ALIGNMENT;
    pfkv::selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(result);
    if (cudaGetLastError() != cudaSuccess) return PFKV_ERR_CUDA;
    return PFKV_OK;
}
