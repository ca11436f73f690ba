// api.cu -- the C ABI of libpfkv.so (declared in include/pfkv.h): argument
// validation, launch planning and dispatch.  No allocation, no host
// synchronisation; every launch goes to the caller's stream.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "pfkv_internal.cuh"

namespace pfkv {
namespace {

constexpr int kMaxDevices = 64;
// per-device: 0 = unknown, 1 = supported (sm_103), 2 = unsupported; SM count
std::atomic<int> g_dev_state[kMaxDevices];
std::atomic<int> g_dev_sms[kMaxDevices];

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Checks that the current device is an sm_103 GPU; returns its SM count.
pfkv_status device_check(int *num_sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return PFKV_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return PFKV_ERR_UNSUPPORTED;
    int st = g_dev_state[dev].load(std::memory_order_acquire);
    if (st == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return PFKV_ERR_CUDA;
        }
        g_dev_sms[dev].store(sms, std::memory_order_relaxed);
        st = (major == 10 && minor == 3) ? 1 : 2;
        if (st == 1) {
            // load every kernel now, so that no launch of a later call, maybe
            // inside a timed or captured region, pays for lazy module loading
            cudaError_t e = preload_append();
            if (e == cudaSuccess) e = preload_split_pers();
            if (e == cudaSuccess) e = preload_combine_pers();
            if (e == cudaSuccess) e = preload_split_generic();
            if (e == cudaSuccess) e = preload_mass();
            if (e == cudaSuccess) e = preload_stage();
            if (e != cudaSuccess) {
                cudaGetLastError();
                return PFKV_ERR_CUDA;
            }
        }
        g_dev_state[dev].store(st, std::memory_order_release);
    }
    if (st != 1) return PFKV_ERR_UNSUPPORTED;
    if (num_sms) *num_sms = g_dev_sms[dev].load(std::memory_order_relaxed);
    return PFKV_OK;
}

pfkv_status check_cache(const pfkv_cache *c) {
    if (!c) return PFKV_ERR_INVALID_ARG;
    if (c->page_size != kPage) return PFKV_ERR_UNSUPPORTED;
    if (c->head_dim != 64 && c->head_dim != 128) return PFKV_ERR_UNSUPPORTED;
    if (c->dtype != PFKV_KV_BF16 && c->dtype != PFKV_KV_FP8_E4M3) return PFKV_ERR_INVALID_ARG;
    if (c->num_pages <= 0 || c->num_kv_heads <= 0) return PFKV_ERR_INVALID_ARG;
    // unit indices page * num_kv_heads + h are 32-bit in the kernels
    if ((long long)c->num_pages * c->num_kv_heads > 0x7fffffffLL) return PFKV_ERR_UNSUPPORTED;
    if (!c->k_pages || !c->v_pages) return PFKV_ERR_INVALID_ARG;
    if (c->dtype == PFKV_KV_FP8_E4M3 && (!c->k_scale || !c->v_scale)) return PFKV_ERR_INVALID_ARG;
    if (!aligned(c->k_pages, 16) || !aligned(c->v_pages, 16)) return PFKV_ERR_ALIGNMENT;
    if (c->dtype == PFKV_KV_FP8_E4M3 && (!aligned(c->k_scale, 4) || !aligned(c->v_scale, 4)))
        return PFKV_ERR_ALIGNMENT;
    if (c->page_tags && !aligned(c->page_tags, 4)) return PFKV_ERR_ALIGNMENT;
    return PFKV_OK;
}

pfkv_status check_pages(const pfkv_cache *c, const pfkv_pages *p) {
    if (!p) return PFKV_ERR_INVALID_ARG;
    if (p->batch < 0 || p->max_pages <= 0) return PFKV_ERR_INVALID_ARG;
    if (p->batch == 0) return PFKV_OK;
    if (!p->block_tables || !p->seq_lens) return PFKV_ERR_INVALID_ARG;
    if (p->bt_stride_b < 0 || p->bt_stride_h < 0 || p->len_stride_b < 0 || p->len_stride_h < 0)
        return PFKV_ERR_INVALID_ARG;
    // a table row must hold max_pages entries without running into the next
    if (p->bt_stride_h == 0 && p->batch > 1 && p->bt_stride_b < p->max_pages)
        return PFKV_ERR_INVALID_ARG;
    if ((c->page_tags == nullptr) != (p->expected_tags == nullptr)) return PFKV_ERR_INVALID_ARG;
    if (!aligned(p->block_tables, 4) || !aligned(p->seq_lens, 4)) return PFKV_ERR_ALIGNMENT;
    if (p->expected_tags && !aligned(p->expected_tags, 4)) return PFKV_ERR_ALIGNMENT;
    return PFKV_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int auto_chunk_tokens(int B, int Hkv, int max_seq_len, int num_sms) {
    // aim for about eight chunks per SM if every head had max_seq_len tokens
    const long long work = (long long)B * Hkv * (max_seq_len > 0 ? max_seq_len : 1);
    long long per = (work + 8LL * num_sms - 1) / (8LL * num_sms);
    per = (per + 255) / 256 * 256;
    if (per < 256) per = 256;
    if (per > 4096) per = 4096;
    return (int)per;
}

// Host-visible checks of the attention arguments (no CUDA call).
pfkv_status check_decode_args(const pfkv_cache *c, int32_t num_q_heads, int32_t split_tokens,
                              int32_t max_seq_len) {
    if (num_q_heads <= 0 || num_q_heads % c->num_kv_heads != 0) return PFKV_ERR_INVALID_ARG;
    const int G = num_q_heads / c->num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return PFKV_ERR_UNSUPPORTED;
    if (max_seq_len < 0) return PFKV_ERR_INVALID_ARG;
    if (split_tokens < 0 || split_tokens % kPage != 0) return PFKV_ERR_INVALID_ARG;
    if (split_tokens > 8192) return PFKV_ERR_UNSUPPORTED;
    return PFKV_OK;
}

// Arguments of a kv_append call, checked (no launch).  PFKV_OK with an empty
// batch means there is nothing to do.
pfkv_status append_args(const pfkv_cache *cache, const pfkv_pages *pages, const int32_t *positions,
                        const int32_t *new_lens, int32_t num_new_tokens, const void *k_new,
                        const void *v_new, uint8_t *flags, AppendArgs *out) {
    pfkv_status st = check_cache(cache);
    if (st != PFKV_OK) return st;
    st = check_pages(cache, pages);
    if (st != PFKV_OK) return st;
    if (num_new_tokens <= 0) return PFKV_ERR_INVALID_ARG;
    if (pages->batch == 0) return PFKV_OK;
    if (!positions || !k_new || !v_new) return PFKV_ERR_INVALID_ARG;
    if (!aligned(positions, 4) || (new_lens && !aligned(new_lens, 4))) return PFKV_ERR_ALIGNMENT;
    if (!aligned(k_new, 16) || !aligned(v_new, 16)) return PFKV_ERR_ALIGNMENT;
    if (flags && !aligned(flags, 4)) return PFKV_ERR_ALIGNMENT;
    const long long units = ((long long)num_new_tokens + 30) / kPage;
    if ((units + 3) / 4 > 65535) return PFKV_ERR_UNSUPPORTED;
    if ((long long)pages->batch * cache->num_kv_heads > 0x7fffffffLL) return PFKV_ERR_UNSUPPORTED;
    AppendArgs a{};
    a.k_pages = cache->k_pages;
    a.v_pages = cache->v_pages;
    a.k_scale = cache->k_scale;
    a.v_scale = cache->v_scale;
    a.page_tags = cache->page_tags;
    a.num_pages = cache->num_pages;
    a.Hkv = cache->num_kv_heads;
    a.D = cache->head_dim;
    a.dtype = cache->dtype;
    a.block_tables = pages->block_tables;
    a.bt_sb = pages->bt_stride_b;
    a.bt_sh = pages->bt_stride_h;
    a.expected_tags = pages->expected_tags;
    a.max_pages = pages->max_pages;
    a.positions = positions;
    a.new_lens = new_lens;
    a.len_sb = pages->len_stride_b;
    a.len_sh = pages->len_stride_h;
    a.T = num_new_tokens;
    a.k_new = static_cast<const __nv_bfloat16 *>(k_new);
    a.v_new = static_cast<const __nv_bfloat16 *>(v_new);
    a.flags = flags;
    *out = a;
    return PFKV_OK;
}

pfkv_status make_plan(const pfkv_cache *c, const pfkv_pages *p, int32_t num_q_heads,
                      int32_t split_tokens, int32_t max_seq_len, int num_sms, DecodePlan *plan,
                      bool mass = false, int32_t kq = 1, bool cuda_cores = false) {
    const pfkv_status st = check_decode_args(c, num_q_heads, split_tokens, max_seq_len);
    if (st != PFKV_OK) return st;
    if (kq < 1 || (long long)p->batch * kq > 0x7fffffffLL) return PFKV_ERR_INVALID_ARG;
    const int G = num_q_heads / c->num_kv_heads;
    DecodePlan q{};
    q.Breq = p->batch;
    q.kq = kq;
    q.B = p->batch * kq;  // virtual requests: one per (request, query token)
    q.Hkv = c->num_kv_heads;
    q.Hq = num_q_heads;
    q.G = G;
    q.D = c->head_dim;
    q.dtype = c->dtype;
    q.tags = c->page_tags != nullptr;
    // Persistent balanced path (head_dim 128): one segment per (request, kv
    // head) unless the caller fixes the split size.  Only the output is
    // contracted, not the split: the split size is coarsened (a multiple of
    // the caller's) when a launch's segments would not fit the kernels'
    // tables, and a batch whose (request, kv head) pairs alone would not fit
    // runs as several launches of whole requests.
    q.kind = !cuda_cores && pers_supported(q) && (long long)kq * q.Hkv <= kPersMaxSegments ? 1 : 0;
    if (q.kind == 1) {
        q.greq = (int)min((long long)q.Breq,
                          min((long long)kPersMaxRequests, (long long)(kPersMaxSegments / (kq * q.Hkv))));
        q.greq = max(q.greq, 1);
        q.ngroups = (q.Breq + q.greq - 1) / q.greq;
        const long long pages = max_seq_len > 0 ? (max_seq_len + kPage - 1) / kPage : 1;
        long long chunk_pages = split_tokens > 0 ? split_tokens / kPage : pages;
        const long long max_chunks = kPersMaxSegments / ((long long)q.greq * kq * q.Hkv);
        if ((pages + chunk_pages - 1) / chunk_pages > max_chunks)
            chunk_pages = (pages + max_chunks - 1) / max_chunks;
        if (chunk_pages > 0x7fffffffLL / kPage) return PFKV_ERR_UNSUPPORTED;
        q.chunk_tokens = (int)(chunk_pages * kPage);
        q.nchunks = (int)((pages + chunk_pages - 1) / chunk_pages);
        q.pers_ctas = num_sms;
        // every (virtual request, kv head) at max_seq_len: an upper bound on the units
        const long long units_bound = (long long)q.B * q.Hkv * pages;
        q.workers = num_sms * pers_workers_for(units_bound, num_sms);
    } else {
        q.greq = q.Breq;
        q.ngroups = 1;
        q.chunk_tokens = split_tokens > 0 ? split_tokens
                                          : auto_chunk_tokens(q.B, q.Hkv, max_seq_len, num_sms);
        q.nchunks = max_seq_len > 0 ? (max_seq_len + q.chunk_tokens - 1) / q.chunk_tokens : 1;
        q.pers_ctas = q.workers = 0;
    }
    q.htiles = max(1, (p->max_pages + kValTile - 1) / kValTile);
    // segments of one launch (one request group for the persistent kind)
    const long long Bl = q.kind == 1 ? (long long)min(q.greq, q.Breq) * kq : q.B;
    const long long items = Bl * q.Hkv * q.nchunks;
    if (items > 0x7fffffffLL || (long long)q.B * q.Hq > 0x7fffffffLL) return PFKV_ERR_UNSUPPORTED;
    // rows of partial results: one per (b, hq, chunk), or segment + worker
    const size_t rows_kv = q.kind == 1 ? (size_t)items + q.workers : (size_t)items;
    size_t off = 0;
    q.off_hflags = off;
    off = align256(off + (q.tags ? sizeof(uint32_t) * q.Breq * q.Hkv * q.htiles : 0));
    q.off_prefix = off;
    off = align256(off + (q.kind == 1 ? sizeof(int) * ((size_t)items + 1) : 0));
    q.off_status = off;
    off = align256(off + sizeof(uint32_t) * rows_kv);
    q.off_lse = off;
    off = align256(off + sizeof(float) * rows_kv * q.G);
    q.off_o = off;
    off = align256(off + sizeof(float) * rows_kv * q.G * q.D);
    // attention mass: every live token's G final scores, each head's final
    // log2-sum-exp and the request flags
    q.mass = mass;
    q.off_mscore = off;
    off = align256(off + (mass ? sizeof(float) * q.B * q.Hkv * (size_t)max_seq_len * q.G : 0));
    q.off_lsefin = off;
    off = align256(off + (mass ? sizeof(float) * q.B * q.Hq : 0));
    q.off_rflags = off;
    off = align256(off + (mass ? (size_t)q.B : 0));
    q.total = off;
    *plan = q;
    return PFKV_OK;
}

}  // namespace
}  // namespace pfkv

using namespace pfkv;

extern "C" {

const char *pfkv_status_string(pfkv_status s) {
    switch (s) {
        case PFKV_OK: return "ok";
        case PFKV_ERR_INVALID_ARG: return "invalid argument";
        case PFKV_ERR_UNSUPPORTED: return "unsupported configuration or device";
        case PFKV_ERR_ALIGNMENT: return "misaligned pointer";
        case PFKV_ERR_WORKSPACE: return "workspace missing or too small";
        case PFKV_ERR_CUDA: return "CUDA error";
        case PFKV_ERR_DEVICE: return "a device-side wait gave up";
    }
    return "unknown status";
}

int32_t pfkv_abi_version(void) { return PFKV_ABI_VERSION; }

pfkv_status pfkv_flags_status(const uint8_t *flags, int32_t batch) {
    if (batch < 0 || (batch > 0 && !flags)) return PFKV_ERR_INVALID_ARG;
    for (int32_t b = 0; b < batch; ++b)
        if (flags[b] & PFKV_FLAG_DEVICE_TIMEOUT) return PFKV_ERR_DEVICE;
    return PFKV_OK;
}

pfkv_status pfkv_kv_append(const pfkv_cache *cache, const pfkv_pages *pages,
                           const int32_t *positions, const int32_t *new_lens,
                           int32_t num_new_tokens, const void *k_new, const void *v_new,
                           uint8_t *flags, void *stream) {
    AppendArgs a{};
    pfkv_status st = append_args(cache, pages, positions, new_lens, num_new_tokens, k_new, v_new,
                                       flags, &a);
    if (st != PFKV_OK || pages->batch == 0) return st;
    st = device_check(nullptr);
    if (st != PFKV_OK) return st;
    if (launch_kv_append(a, pages->batch, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return PFKV_ERR_CUDA;
    return PFKV_OK;
}

pfkv_status pfkv_decode_workspace_size(const pfkv_cache *cache, const pfkv_pages *pages,
                                       int32_t num_q_heads, int32_t split_tokens,
                                       int32_t max_seq_len, size_t *bytes) {
    if (!bytes) return PFKV_ERR_INVALID_ARG;
    pfkv_status st = check_cache(cache);
    if (st != PFKV_OK) return st;
    st = check_pages(cache, pages);
    if (st != PFKV_OK) return st;
    st = check_decode_args(cache, num_q_heads, split_tokens, max_seq_len);
    if (st != PFKV_OK) return st;
    int sms = 0;
    st = device_check(&sms);
    if (st != PFKV_OK) return st;
    DecodePlan plan;
    st = make_plan(cache, pages, num_q_heads, split_tokens, max_seq_len, sms, &plan);
    if (st != PFKV_OK) return st;
    *bytes = plan.total;
    return PFKV_OK;
}

}  // extern "C"

namespace {

// The arguments of the request group starting at request r0: every
// per-request pointer moved to the group's first request.
DecodeArgs group_args(const DecodeArgs &a, const DecodePlan &p, int r0) {
    DecodeArgs g = a;
    const long long v0 = (long long)r0 * p.kq;  // first virtual request
    g.q = a.q + v0 * p.Hq * p.D;
    g.out = a.out + v0 * p.Hq * p.D;
    if (a.flags) g.flags = a.flags + r0;
    g.block_tables = a.block_tables + (long long)r0 * a.bt_sb;
    g.seq_lens = a.seq_lens + (long long)r0 * a.len_sb;
    if (a.expected_tags) g.expected_tags = a.expected_tags + (long long)r0 * a.bt_sb;
    if (a.hflags) g.hflags = a.hflags + (long long)r0 * p.Hkv * p.htiles;
    if (a.mscore) g.mscore = a.mscore + v0 * p.Hkv * (long long)a.mlen * p.G;
    if (a.lse_fin) g.lse_fin = a.lse_fin + v0 * p.Hq;
    if (a.rflags) g.rflags = a.rflags + r0;
    return g;
}

struct MassOut {
    float *mass;
    int64_t sb, sh;
};

// The attention call: the stages named in `stages`, plus the attention-mass
// pass when `mass` is given.  With `app` (checked arguments of a kv_append
// for the same pages), the append runs first, in the same launch as the
// validation when that stage runs.
pfkv_status attn_impl(const pfkv_cache *cache, const pfkv_pages *pages, const void *q,
                      int32_t num_q_heads, float sm_scale, int32_t split_tokens,
                      int32_t max_seq_len, void *workspace, size_t workspace_bytes, void *out,
                      uint8_t *flags, uint32_t stages, const MassOut *mass, void *stream,
                      int32_t kq = 1, const AppendArgs *app = nullptr) {
    if (kq < 1 || (mass && kq != 1)) return kq < 1 ? PFKV_ERR_INVALID_ARG : PFKV_ERR_UNSUPPORTED;
    if ((stages & PFKV_STAGE_ALL) == 0 ||
        (stages & ~(PFKV_STAGE_ALL | PFKV_STAGE_FUSED_TAGS | PFKV_STAGE_CUDA_CORES)))
        return PFKV_ERR_INVALID_ARG;
    const bool fused = (stages & PFKV_STAGE_FUSED_TAGS) != 0;
    pfkv_status st = check_cache(cache);
    if (st != PFKV_OK) return st;
    st = check_pages(cache, pages);
    if (st != PFKV_OK) return st;
    if (!(sm_scale == sm_scale) || std::isinf(sm_scale)) return PFKV_ERR_INVALID_ARG;
    if (pages->batch == 0) return PFKV_OK;
    if (!q || !out) return PFKV_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(out, 16)) return PFKV_ERR_ALIGNMENT;
    if (flags && !aligned(flags, 4)) return PFKV_ERR_ALIGNMENT;
    st = check_decode_args(cache, num_q_heads, split_tokens, max_seq_len);
    if (st != PFKV_OK) return st;
    if (!workspace) return PFKV_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return PFKV_ERR_ALIGNMENT;
    int sms = 0;
    st = device_check(&sms);
    if (st != PFKV_OK) return st;
    DecodePlan plan;
    st = make_plan(cache, pages, num_q_heads, split_tokens, max_seq_len, sms, &plan,
                   mass != nullptr, kq, (stages & PFKV_STAGE_CUDA_CORES) != 0);
    if (st != PFKV_OK) return st;
    if (workspace_bytes < plan.total) return PFKV_ERR_WORKSPACE;

    DecodeArgs a{};
    a.k_pages = cache->k_pages;
    a.v_pages = cache->v_pages;
    a.k_scale = cache->k_scale;
    a.v_scale = cache->v_scale;
    a.page_tags = cache->page_tags;
    a.num_pages = cache->num_pages;
    a.block_tables = pages->block_tables;
    a.bt_sb = pages->bt_stride_b;
    a.bt_sh = pages->bt_stride_h;
    a.seq_lens = pages->seq_lens;
    a.len_sb = pages->len_stride_b;
    a.len_sh = pages->len_stride_h;
    a.expected_tags = pages->expected_tags;
    a.max_pages = pages->max_pages;
    a.max_seq_len = max_seq_len;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.flags = flags;
    a.q_scale = sm_scale * 1.4426950408889634f;  // log2(e): scores in log2 units
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    a.hflags = plan.tags && !fused ? reinterpret_cast<uint32_t *>(ws + plan.off_hflags) : nullptr;
    a.htiles = plan.htiles;
    a.fuse_tags = plan.tags && fused ? 1 : 0;
    a.kq = plan.kq;
    a.status = reinterpret_cast<uint32_t *>(ws + plan.off_status);
    a.lse = reinterpret_cast<float *>(ws + plan.off_lse);
    a.o = reinterpret_cast<float *>(ws + plan.off_o);
    a.ws_prefix = reinterpret_cast<int *>(ws + plan.off_prefix);
    if (mass) {
        a.mscore = reinterpret_cast<float *>(ws + plan.off_mscore);
        a.mlen = max_seq_len;
        a.lse_fin = reinterpret_cast<float *>(ws + plan.off_lsefin);
        a.rflags = ws + plan.off_rflags;
        a.mass = mass->mass;
        a.mass_sb = mass->sb;
        a.mass_sh = mass->sh;
    }

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool validate = (stages & PFKV_STAGE_VALIDATE) && plan.tags && !fused;
    a.early = validate ? 1 : 0;
    if (app && validate) {
        if (launch_append_validate(*app, pages->batch, a, plan, s) != cudaSuccess) return PFKV_ERR_CUDA;
    } else {
        if (app && launch_kv_append(*app, pages->batch, s) != cudaSuccess) return PFKV_ERR_CUDA;
        if (validate && launch_validate(a, plan, s) != cudaSuccess) return PFKV_ERR_CUDA;
    }
    if (plan.ngroups > 1) {
        // Request groups, each split then combine on its own slice of the
        // batch: the workspace rows are reused from group to group, so the two
        // stages run in the same call.
        if (((stages & PFKV_STAGE_SPLIT) != 0) != ((stages & PFKV_STAGE_COMBINE) != 0))
            return PFKV_ERR_UNSUPPORTED;
        if (stages & PFKV_STAGE_SPLIT) {
            for (int g = 0; g < plan.ngroups; ++g) {
                const int r0 = g * plan.greq, gr = min(plan.greq, plan.Breq - r0);
                DecodePlan pg = plan;
                pg.Breq = gr;
                pg.B = gr * plan.kq;
                DecodeArgs ag = group_args(a, plan, r0);
                // after the first group the kernel before each split is the
                // previous group's combine, which waits for its own
                // predecessors first and writes none of the call's inputs
                if (g > 0) ag.early = 1;
                if (launch_split(ag, pg, s) != cudaSuccess || launch_combine(ag, pg, s) != cudaSuccess)
                    return PFKV_ERR_CUDA;
            }
        }
    } else {
        if ((stages & PFKV_STAGE_SPLIT) && launch_split(a, plan, s) != cudaSuccess) return PFKV_ERR_CUDA;
        if ((stages & PFKV_STAGE_COMBINE) && launch_combine(a, plan, s) != cudaSuccess)
            return PFKV_ERR_CUDA;
    }
    if (mass && launch_mass(a, plan, s) != cudaSuccess) return PFKV_ERR_CUDA;
    return PFKV_OK;
}

}  // namespace

extern "C" {

pfkv_status pfkv_stage_copy(void *dst, const void *src, size_t bytes, void *stream) {
    if (bytes == 0) return PFKV_OK;
    if (!dst || !src) return PFKV_ERR_INVALID_ARG;
    if (!aligned(dst, 16) || !aligned(src, 16) || (bytes & 15u)) return PFKV_ERR_ALIGNMENT;
    const uintptr_t d = reinterpret_cast<uintptr_t>(dst), r = reinterpret_cast<uintptr_t>(src);
    if (d < r + bytes && r < d + bytes) return PFKV_ERR_INVALID_ARG;  // overlapping ranges
    int sms = 0;
    const pfkv_status st = device_check(&sms);
    if (st != PFKV_OK) return st;
    return launch_stage_copy(dst, src, bytes, sms, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PFKV_OK
               : PFKV_ERR_CUDA;
}

pfkv_status pfkv_decode_step(const pfkv_cache *cache, const pfkv_pages *pages,
                             const int32_t *positions, const int32_t *new_lens, int32_t num_new_tokens,
                             const void *k_new, const void *v_new, uint8_t *append_flags,
                             const void *q, int32_t num_q_heads, float sm_scale, int32_t split_tokens,
                             int32_t max_seq_len, void *workspace, size_t workspace_bytes, void *out,
                             uint8_t *flags, uint32_t options, void *stream) {
    if (options & ~PFKV_STAGE_FUSED_TAGS) return PFKV_ERR_INVALID_ARG;
    AppendArgs ap{};
    const pfkv_status st = append_args(cache, pages, positions, new_lens, num_new_tokens, k_new, v_new,
                                       append_flags, &ap);
    if (st != PFKV_OK || pages->batch == 0) return st;
    return attn_impl(cache, pages, q, num_q_heads, sm_scale, split_tokens, max_seq_len, workspace,
                     workspace_bytes, out, flags, PFKV_STAGE_ALL | options, nullptr, stream, 1, &ap);
}

pfkv_status pfkv_paged_decode_attn_stages(const pfkv_cache *cache, const pfkv_pages *pages,
                                          const void *q, int32_t num_q_heads, float sm_scale,
                                          int32_t split_tokens, int32_t max_seq_len,
                                          void *workspace, size_t workspace_bytes, void *out,
                                          uint8_t *flags, uint32_t stages, void *stream) {
    return attn_impl(cache, pages, q, num_q_heads, sm_scale, split_tokens, max_seq_len,
                     workspace, workspace_bytes, out, flags, stages, nullptr, stream);
}

pfkv_status pfkv_decode_multi_workspace_size(const pfkv_cache *cache, const pfkv_pages *pages,
                                             int32_t num_q_heads, int32_t num_query_tokens,
                                             int32_t split_tokens, int32_t max_seq_len,
                                             size_t *bytes) {
    if (!bytes) return PFKV_ERR_INVALID_ARG;
    pfkv_status st = check_cache(cache);
    if (st != PFKV_OK) return st;
    st = check_pages(cache, pages);
    if (st != PFKV_OK) return st;
    st = check_decode_args(cache, num_q_heads, split_tokens, max_seq_len);
    if (st != PFKV_OK) return st;
    if (num_query_tokens < 1) return PFKV_ERR_INVALID_ARG;
    int sms = 0;
    st = device_check(&sms);
    if (st != PFKV_OK) return st;
    DecodePlan plan;
    st = make_plan(cache, pages, num_q_heads, split_tokens, max_seq_len, sms, &plan, false,
                   num_query_tokens);
    if (st != PFKV_OK) return st;
    *bytes = plan.total;
    return PFKV_OK;
}

pfkv_status pfkv_paged_decode_attn_multi(const pfkv_cache *cache, const pfkv_pages *pages,
                                         const void *q, int32_t num_q_heads,
                                         int32_t num_query_tokens, float sm_scale,
                                         int32_t split_tokens, int32_t max_seq_len,
                                         void *workspace, size_t workspace_bytes, void *out,
                                         uint8_t *flags, uint32_t options, void *stream) {
    if (options & ~PFKV_STAGE_FUSED_TAGS) return PFKV_ERR_INVALID_ARG;
    if (num_query_tokens < 1) return PFKV_ERR_INVALID_ARG;
    return attn_impl(cache, pages, q, num_q_heads, sm_scale, split_tokens, max_seq_len,
                     workspace, workspace_bytes, out, flags, PFKV_STAGE_ALL | options, nullptr,
                     stream, num_query_tokens);
}

pfkv_status pfkv_decode_mass_workspace_size(const pfkv_cache *cache, const pfkv_pages *pages,
                                            int32_t num_q_heads, int32_t split_tokens,
                                            int32_t max_seq_len, size_t *bytes) {
    if (!bytes) return PFKV_ERR_INVALID_ARG;
    pfkv_status st = check_cache(cache);
    if (st != PFKV_OK) return st;
    st = check_pages(cache, pages);
    if (st != PFKV_OK) return st;
    st = check_decode_args(cache, num_q_heads, split_tokens, max_seq_len);
    if (st != PFKV_OK) return st;
    int sms = 0;
    st = device_check(&sms);
    if (st != PFKV_OK) return st;
    DecodePlan plan;
    st = make_plan(cache, pages, num_q_heads, split_tokens, max_seq_len, sms, &plan, true);
    if (st != PFKV_OK) return st;
    *bytes = plan.total;
    return PFKV_OK;
}

pfkv_status pfkv_paged_decode_attn_mass(const pfkv_cache *cache, const pfkv_pages *pages,
                                        const void *q, int32_t num_q_heads, float sm_scale,
                                        int32_t split_tokens, int32_t max_seq_len,
                                        void *workspace, size_t workspace_bytes, void *out,
                                        uint8_t *flags, float *attn_mass, int64_t mass_stride_b,
                                        int64_t mass_stride_h, uint32_t options, void *stream) {
    if (options & ~PFKV_STAGE_FUSED_TAGS) return PFKV_ERR_INVALID_ARG;
    if (mass_stride_b < 0 || mass_stride_h < 0) return PFKV_ERR_INVALID_ARG;
    if (pages && pages->batch > 0) {
        if (!attn_mass) return PFKV_ERR_INVALID_ARG;
        if (!aligned(attn_mass, 4)) return PFKV_ERR_ALIGNMENT;
    }
    const MassOut m{attn_mass, mass_stride_b, mass_stride_h};
    return attn_impl(cache, pages, q, num_q_heads, sm_scale, split_tokens, max_seq_len,
                     workspace, workspace_bytes, out, flags, PFKV_STAGE_ALL | options, &m, stream);
}

pfkv_status pfkv_paged_decode_attn(const pfkv_cache *cache, const pfkv_pages *pages,
                                   const void *q, int32_t num_q_heads, float sm_scale,
                                   int32_t split_tokens, int32_t max_seq_len, void *workspace,
                                   size_t workspace_bytes, void *out, uint8_t *flags,
                                   void *stream) {
    return pfkv_paged_decode_attn_stages(cache, pages, q, num_q_heads, sm_scale, split_tokens,
                                         max_seq_len, workspace, workspace_bytes, out, flags,
                                         PFKV_STAGE_ALL, stream);
}

pfkv_status pfkv_paged_decode_attn_fused_tags(const pfkv_cache *cache, const pfkv_pages *pages,
                                              const void *q, int32_t num_q_heads, float sm_scale,
                                              int32_t split_tokens, int32_t max_seq_len,
                                              void *workspace, size_t workspace_bytes, void *out,
                                              uint8_t *flags, void *stream) {
    return pfkv_paged_decode_attn_stages(cache, pages, q, num_q_heads, sm_scale, split_tokens,
                                         max_seq_len, workspace, workspace_bytes, out, flags,
                                         PFKV_STAGE_ALL | PFKV_STAGE_FUSED_TAGS, stream);
}

pfkv_status pfkv_e4m3_encode(const float *x, int64_t n, uint8_t *out, void *stream) {
    if (n < 0) return PFKV_ERR_INVALID_ARG;
    if (n == 0) return PFKV_OK;
    if (!x || !out) return PFKV_ERR_INVALID_ARG;
    if (!aligned(x, 4)) return PFKV_ERR_ALIGNMENT;
    pfkv_status st = device_check(nullptr);
    if (st != PFKV_OK) return st;
    return launch_e4m3_encode(x, n, out, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PFKV_OK
               : PFKV_ERR_CUDA;
}

pfkv_status pfkv_e4m3_decode(const uint8_t *codes, int64_t n, float *out, void *stream) {
    if (n < 0) return PFKV_ERR_INVALID_ARG;
    if (n == 0) return PFKV_OK;
    if (!codes || !out) return PFKV_ERR_INVALID_ARG;
    if (!aligned(out, 4)) return PFKV_ERR_ALIGNMENT;
    pfkv_status st = device_check(nullptr);
    if (st != PFKV_OK) return st;
    return launch_e4m3_decode(codes, n, out, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PFKV_OK
               : PFKV_ERR_CUDA;
}

}  // extern "C"
