// stage.cu -- pfkv_stage_copy's kernel: a copy in 16-byte words by every SM,
// for per-step inputs a caller keeps in host memory (see include/pfkv.h).
#include "pfkv_internal.cuh"

namespace pfkv {
namespace {

constexpr int kStageThreads = 256;

// Waits for the previous kernel (a caller's kernel may still be writing src
// or reading dst), then lets the next kernel of the stream launch: this
// library's kernels wait for this one to complete before they read dst.
__global__ void __launch_bounds__(kStageThreads) stage_copy_kernel(uint4 *dst, const uint4 *src,
                                                                   long long n16) {
    pdl_enter();
    for (long long i = blockIdx.x * (long long)kStageThreads + threadIdx.x; i < n16;
         i += (long long)gridDim.x * kStageThreads)
        dst[i] = src[i];
}

}  // namespace

cudaError_t launch_stage_copy(void *dst, const void *src, size_t bytes, int num_sms, cudaStream_t s) {
    const long long n16 = (long long)(bytes / 16);
    const long long need = (n16 + kStageThreads - 1) / kStageThreads;
    const long long grid = need < 4LL * num_sms ? need : 4LL * num_sms;
    return launch_pdl(stage_copy_kernel, dim3((unsigned)grid), dim3(kStageThreads), 0, s,
                      static_cast<uint4 *>(dst), static_cast<const uint4 *>(src), n16);
}

cudaError_t preload_stage() { return preload_kernel(stage_copy_kernel); }

}  // namespace pfkv
