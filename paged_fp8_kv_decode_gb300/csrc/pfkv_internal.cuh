// pfkv_internal.cuh -- device primitives and launch plans shared by the
// kernels of libpfkv.so (sm_103a).  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "../../include/pfkv.h"

namespace pfkv {

constexpr int kPage = PFKV_PAGE_SIZE;

// per-(request, kv head, chunk) status bits written by the split kernel
constexpr uint32_t kStatusBadPage = PFKV_FLAG_BAD_PAGE;
constexpr uint32_t kStatusTimeout = PFKV_FLAG_DEVICE_TIMEOUT;
// validation: a CTA checks kValTile live entries of one table row, each of its
// kValThreads threads kValPer of them with all loads issued before any is used
constexpr int kValThreads = 256;
constexpr int kValPer = 8;
constexpr int kValTile = kValThreads * kValPer;

// persistent split kernel: the largest segment and request counts its
// shared-memory tables hold (the combine kernels size their own tables from
// the same numbers)
constexpr int kPersMaxSegments = 4096;
constexpr int kPersMaxRequests = 4096;

// A bounded wait gives up after this many nanoseconds of %globaltimer.
constexpr unsigned long long kWaitLimitNs = 100ull * 1000ull * 1000ull;

// --------------------------------------------------------------------------
// Launch plan of one paged_decode_attn call (computed on the host; the same
// numbers size the workspace).
// --------------------------------------------------------------------------
struct DecodePlan {
    int B, Hkv, Hq, G, D, dtype;
    int chunk_tokens;   // tokens per split-KV chunk (multiple of 16)
    int nchunks;        // ceil(max_seq_len / chunk_tokens), >= 1
    bool tags;
    // kind 0: one CTA per (request, kv head, chunk), workspace rows indexed
    //         [b][hq][chunk];
    // kind 1: persistent balanced workers (FP8 or BF16, head_dim 128 or 64,
    //         G <= 8), rows indexed segment + worker, pers_ctas CTAs
    int kind;
    int pers_ctas, workers;
    int htiles;         // validation tiles per table row: ceil(max_pages / kValTile)
    // workspace layout (byte offsets, 256-aligned)
    size_t off_hflags, off_status, off_lse, off_o, off_prefix, total;
    bool mass;
    size_t off_mscore, off_lsefin, off_rflags;
    int Breq, kq;       // requests and query tokens per request (B = Breq * kq)
    // persistent kind: the batch runs as ngroups launches of up to greq
    // requests each (split then combine per group), so that one launch's
    // segments and requests fit the kernels' shared-memory tables
    int greq, ngroups;
};

struct DecodeArgs {
    // pool
    const void *k_pages, *v_pages;
    const float *k_scale, *v_scale;
    const uint32_t *page_tags;
    int num_pages;
    // batch
    const int32_t *block_tables;
    long long bt_sb, bt_sh;
    const int32_t *seq_lens;
    long long len_sb, len_sh;
    const uint32_t *expected_tags;
    int max_pages, max_seq_len;
    // query / output
    const __nv_bfloat16 *q;
    __nv_bfloat16 *out;
    uint8_t *flags;
    float q_scale;      // sm_scale * log2(e): scores are kept in log2 units
    // workspace
    uint32_t *hflags;   // [B][Hkv][htiles] tag/bounds bits from the validation kernel
    int htiles;
    int fuse_tags;      // compare tags where the split kernels load page ids
    // query tokens per request (multi-query verify; 1 for plain decode).  The
    // split and combine kernels see B * kq "virtual requests" v: request
    // v / kq, query token v % kq, attending to the first n - kq + 1 + v % kq
    // tokens of each head; q, out and the partial rows are indexed by v.
    int kq;
    // attention mass (null unless requested)
    float *mscore;      // [B][Hkv][mlen][G] final scores (log2 units) of live tokens
    int mlen;           // = max_seq_len
    float *lse_fin;     // [B][Hq] log2-sum-exp over all of a head's tokens
    uint8_t *rflags;    // [B] request flags, written by the combine
    float *mass;        // caller's running totals, mass[b*mass_sb + h*mass_sh + j]
    long long mass_sb, mass_sh;
    uint32_t *status;   // [B][Hkv][nchunks]
    float *lse;         // [B][Hq][nchunks]  log2-sum-exp of the chunk
    float *o;           // [B][Hq][nchunks][D] chunk output (normalised)
    int *ws_prefix;     // persistent kind: exclusive unit prefix per segment
    // The kernel just before the split kernel in the stream is this library's
    // validation kernel, launched by the same call.  That kernel waits for its
    // own predecessors before it lets the split kernel start, so the call's
    // inputs are final when the split kernel starts.
    int early;
};

struct AppendArgs {
    void *k_pages, *v_pages;
    float *k_scale, *v_scale;
    const uint32_t *page_tags;
    int num_pages, Hkv, D, dtype;
    const int32_t *block_tables;
    long long bt_sb, bt_sh;
    const uint32_t *expected_tags;
    int max_pages;
    const int32_t *positions, *new_lens;
    long long len_sb, len_sh;
    int T;
    const __nv_bfloat16 *k_new, *v_new;
    uint8_t *flags;
};

// Launch with programmatic dependent launch allowed: the kernel may be
// scheduled while the previous kernel in the stream still runs.  Every kernel
// of this library starts with pdl_enter(), which waits for the previous
// kernel's completion and memory before anything else, so the overlap is
// limited to launch latency and is safe whatever precedes it in the stream.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Tokens of kv head h that virtual request v attends to (see DecodeArgs::kq),
// or -1 when the request's length is invalid (it is then flagged BAD_LENGTH).
__device__ __forceinline__ int query_len(const DecodeArgs &a, int v, int h) {
    const int b = a.kq == 1 ? v : v / a.kq;
    const int n = a.seq_lens[(long long)b * a.len_sb + (long long)h * a.len_sh];
    if (n < 0 || (long long)n > (long long)a.max_pages * kPage || n > a.max_seq_len) return -1;
    return max(0, n - a.kq + 1 + (v - b * a.kq));
}

// First block-table entry of kv head h of virtual request v.
__device__ __forceinline__ long long table_row(const DecodeArgs &a, int v, int h) {
    return (long long)(a.kq == 1 ? v : v / a.kq) * a.bt_sb + (long long)h * a.bt_sh;
}

// Status bits of table entry bt_index naming page `id` of kv head h: BAD_PAGE
// for an id outside the pool, TAG_MISMATCH (fused check only) for a pool tag
// that differs from the expected one.  Zero: the unit may be read.
__device__ __forceinline__ uint32_t entry_bits(const DecodeArgs &a, int id, int h, int Hkv,
                                               long long bt_index) {
    if (id < 0 || id >= a.num_pages) return PFKV_FLAG_BAD_PAGE;
    if (a.fuse_tags && a.page_tags[(long long)id * Hkv + h] != a.expected_tags[bt_index])
        return PFKV_FLAG_TAG_MISMATCH;
    return 0u;
}

// Persistent layout: the worker of global unit x when U units are shared by W
// workers (worker w takes units [ceil(wU/W), ceil((w+1)U/W))).
// 16-token units of chunk c (chunk_tokens tokens each) of a head with n
// tokens; none for a flagged length (n < 0).  The persistent split kernel and
// its combine count units with this one function.
__device__ __forceinline__ int segment_units(int n, int c, int chunk_tokens) {
    if (n < 0) return 0;
    const int pages = (n + kPage - 1) / kPage;
    const int cp = chunk_tokens / kPage;
    return max(0, min(pages, (c + 1) * cp) - c * cp);
}

__device__ __forceinline__ int pers_worker_of(long long x, long long U, int W) {
    return (int)((x * W) / U);
}

// Final scores of one token for the attention-mass pass (a.mscore set).
template <int G>
__device__ __forceinline__ void store_scores(const DecodeArgs &a, int bh, int tok,
                                             const float (&sc)[G]) {
    float *dst = a.mscore + ((long long)bh * a.mlen + tok) * G;
    if constexpr (G == 8) {
        reinterpret_cast<float4 *>(dst)[0] = make_float4(sc[0], sc[1], sc[2], sc[3]);
        reinterpret_cast<float4 *>(dst)[1] = make_float4(sc[4], sc[5], sc[6], sc[7]);
    } else if constexpr (G == 4) {
        *reinterpret_cast<float4 *>(dst) = make_float4(sc[0], sc[1], sc[2], sc[3]);
    } else if constexpr (G == 2) {
        *reinterpret_cast<float2 *>(dst) = make_float2(sc[0], sc[1]);
    } else {
        dst[0] = sc[0];
    }
}

// Whether the validation kernel flagged request b (any kv head, any tile).
// Computed by the whole CTA: every thread must call it.
__device__ __forceinline__ bool request_rejected_cta(const DecodeArgs &a, int b, int Hkv) {
    int f = 0;
    if (a.hflags) {
        const int n = Hkv * a.htiles;
        const uint32_t *src = a.hflags + (long long)b * n;
        for (int i = threadIdx.x; i < n; i += blockDim.x) f |= src[i] != 0u;
    }
    return __syncthreads_or(f) != 0;
}

// launchers (defined in the .cu files)
cudaError_t launch_kv_append(const AppendArgs &a, int B, cudaStream_t s);
cudaError_t launch_validate(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s);
cudaError_t launch_append_validate(const AppendArgs &ap, int B, const DecodeArgs &a, const DecodePlan &p,
                                   cudaStream_t s);
cudaError_t launch_split(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s);
cudaError_t launch_mass(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s);
bool pers_supported(const DecodePlan &p);
int pers_workers_for(long long units_bound, int num_sms);
cudaError_t launch_split_pers(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s);
cudaError_t launch_split_pers_d64(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s);
cudaError_t launch_combine_pers(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s);
cudaError_t launch_combine(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s);
cudaError_t launch_e4m3_encode(const float *x, int64_t n, uint8_t *out, cudaStream_t s);
cudaError_t launch_e4m3_decode(const uint8_t *c, int64_t n, float *out, cudaStream_t s);

// Load every kernel of one source file onto the current device (and set the
// shared-memory opt-ins its launches need), so that no later launch pays for
// lazy module loading.  Called once per device, on its first use.
cudaError_t preload_append();
cudaError_t preload_split_pers();
cudaError_t preload_split_pers_d64();
cudaError_t preload_combine_pers();
cudaError_t preload_split_generic();
cudaError_t preload_mass();
cudaError_t preload_stage();
cudaError_t launch_stage_copy(void *dst, const void *src, size_t bytes, int num_sms, cudaStream_t s);

// Loads one kernel (a no-op if it is loaded already).
template <typename F>
cudaError_t preload_kernel(F *kernel) {
    cudaFuncAttributes attr;
    return cudaFuncGetAttributes(&attr, kernel);
}

// --------------------------------------------------------------------------
// device helpers
// --------------------------------------------------------------------------
#if defined(__CUDACC__)

// Wait for the previous kernel in the stream (completion and memory), then
// let the next one launch.  A no-op without programmatic dependent launch.
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of `bar` to complete; false if the bounded wait
// gave up (the caller records a timeout and stops issuing work).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    unsigned long long t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// 1-D bulk copy global -> shared (this CTA), completing `bytes` of tx on bar.
// dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Two e4m3 codes (low byte first) -> two exact fp32 values, via the hardware
// e4m3x2 -> f16x2 conversion (every e4m3 value is exact in f16).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t two) {
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two), __NV_E4M3);
    return __half22float2(*reinterpret_cast<__half2 *>(&h));
}

// bf16 pair packed in a 32-bit word (low half first) -> two exact fp32 values.
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// fp32 -> e4m3, round to nearest even, saturating to +-448 (NaN -> 0x7F).
__device__ __forceinline__ uint8_t float_to_e4m3(float x) {
    return static_cast<uint8_t>(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3));
}

// OR `bits` into byte `idx` of a byte array through its aligned 32-bit word.
__device__ __forceinline__ void atomic_or_byte(uint8_t *base, int idx, uint32_t bits) {
    uintptr_t addr = reinterpret_cast<uintptr_t>(base + idx);
    unsigned int *word = reinterpret_cast<unsigned int *>(addr & ~uintptr_t(3));
    atomicOr(word, bits << (8 * (addr & 3)));
}

#endif  // __CUDACC__

}  // namespace pfkv
