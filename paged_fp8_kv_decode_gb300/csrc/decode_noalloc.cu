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
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "pfkv_internal.cuh"

namespace {

// The shared workspace.  Its name is only a host-side stand-in for the device
// array: kernels receive the device address from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_workspace[PFKV_NOALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;

// The address of the array in the context that was current when it was
// looked up, keyed by the context's unique id.  A module is loaded once per
// context, so another context on the same device (a plugin host's own, or the
// primary context re-created after cudaDeviceReset) holds the array at
// another address; a new context never reuses an id, where it may reuse a
// handle.
struct Cached {
    unsigned long long ctx_id;
    void *addr;
};
std::mutex g_mutex;
Cached g_cached[kMaxDevices];

// Driver entry points through the runtime (no link against the driver
// library).
template <typename Fn>
Fn driver_fn(const char *name, int version) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion(name, &p, version, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<Fn>(p);
}

// Unique id of the current context; 0 if none is current.
bool current_context_id(unsigned long long *id) {
    static const PFN_cuCtxGetCurrent_v4000 get_ctx =
        driver_fn<PFN_cuCtxGetCurrent_v4000>("cuCtxGetCurrent", 4000);
    static const PFN_cuCtxGetId_v12000 get_id = driver_fn<PFN_cuCtxGetId_v12000>("cuCtxGetId", 12000);
    CUcontext ctx = nullptr;
    if (!get_ctx || !get_id || get_ctx(&ctx) != CUDA_SUCCESS) return false;
    *id = 0;
    return ctx == nullptr || get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the array in the current context, looked up on the first
// call made with that context current (cudaGetSymbolAddress, which also makes
// the runtime's context current if none is).
pfkv_status workspace_address(void **addr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return PFKV_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return PFKV_ERR_UNSUPPORTED;
    unsigned long long id = 0;
    if (!current_context_id(&id)) return PFKV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    Cached &c = g_cached[dev];
    if (id == 0 || c.ctx_id != id || c.addr == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_workspace) != cudaSuccess || !p) {
            cudaGetLastError();
            return PFKV_ERR_CUDA;
        }
        // the lookup made the runtime's context current if none was
        if (!current_context_id(&id) || id == 0) return PFKV_ERR_CUDA;
        c.ctx_id = id;
        c.addr = p;
    }
    *addr = c.addr;
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
