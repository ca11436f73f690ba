// decode_noalloc.cu -- pfkv_paged_decode_attn for callers that cannot
// allocate device memory.
//
// Some callers cannot hand this library a workspace: an inference engine that
// has already divided all GPU memory between weights and its KV page pool, a
// plugin whose host framework owns every device allocation, or a decode loop
// that must not call cudaMalloc/cudaFree because those calls can synchronise
// the device.  For them the workspace lives in a fixed-size array in the
// library's own device memory, reserved when the library is loaded onto a GPU
// and kept until the process exits.
#include <atomic>

#include "pfkv_internal.cuh"

namespace {

// The shared workspace.  Its name is only a host-side stand-in for the device
// array: kernels receive the device address from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_workspace[PFKV_NOALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void *> g_workspace_addr[kMaxDevices];

// Device address of the array on the current device, looked up on the first
// call made with that device current.
pfkv_status workspace_address(void **addr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return PFKV_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return PFKV_ERR_UNSUPPORTED;
    void *p = g_workspace_addr[dev].load(std::memory_order_acquire);
    if (!p) {
        if (cudaGetSymbolAddress(&p, g_noalloc_workspace) != cudaSuccess || !p) {
            cudaGetLastError();
            return PFKV_ERR_CUDA;
        }
        g_workspace_addr[dev].store(p, std::memory_order_release);
    }
    *addr = p;
    return PFKV_OK;
}

}  // namespace

extern "C" pfkv_status pfkv_paged_decode_attn_noalloc(const pfkv_cache *cache,
                                                      const pfkv_pages *pages, const void *q,
                                                      int32_t num_q_heads, float sm_scale,
                                                      int32_t split_tokens, int32_t max_seq_len,
                                                      void *out, uint8_t *flags, void *stream) {
    size_t need = 0;
    pfkv_status st = pfkv_decode_workspace_size(cache, pages, num_q_heads, split_tokens,
                                                max_seq_len, &need);
    if (st != PFKV_OK) return st;
    if (need > (size_t)PFKV_NOALLOC_WORKSPACE_BYTES) return PFKV_ERR_WORKSPACE;
    void *ws = nullptr;
    st = workspace_address(&ws);
    if (st != PFKV_OK) return st;
    return pfkv_paged_decode_attn(cache, pages, q, num_q_heads, sm_scale, split_tokens,
                                  max_seq_len, ws, (size_t)PFKV_NOALLOC_WORKSPACE_BYTES, out, flags,
                                  stream);
}
