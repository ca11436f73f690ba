// append.cu -- kv_append (write/quantise new tokens into page slots), the
// separate integrity/bounds validation that runs before attention, and the
// e4m3 conversion utilities.
//
// FP8 e4m3 cache instead of BF16: "Cloudflare quantizes Kimi and GLM caches
// for 41% faster inference", 2nd paragraph.  Tag check as a separate batch
// validation before decode reads: same page, 4th paragraph.
#include <type_traits>

#include "pfkv_internal.cuh"

namespace pfkv {

// --------------------------------------------------------------------------
// kv_append: one warp per (request, kv head, k-th unit touched by the call).
// A warp owns every token of the call that falls into its unit, so the unit
// scale (absmax over those tokens / 448) is a warp reduction, and the rows it
// writes are whole 16-token page slabs or their parts.
// --------------------------------------------------------------------------
constexpr int kAppendWarps = 4;

// The k-th unit touched by the call for (request, kv head) bh, by one warp.
template <int D, bool FP8>
__device__ __forceinline__ void append_unit(const AppendArgs &a, int bh, int k, int lane) {
    constexpr int EPL = D / 32;  // elements per lane per row (4 or 2)
    using Vec = typename std::conditional<EPL == 4, uint2, uint32_t>::type;
    const int b = bh / a.Hkv, h = bh - b * a.Hkv;
    // A decode step appends one token: then unit 0 is the only one written, and
    // its row (row bh of k_new / v_new) does not depend on the position, so it
    // loads while the position and the page id are fetched.
    const bool one = a.T == 1;
    Vec kpre{}, vpre{};
    if (one && k == 0) {
        kpre = *reinterpret_cast<const Vec *>(a.k_new + (long long)bh * D + lane * EPL);
        vpre = *reinterpret_cast<const Vec *>(a.v_new + (long long)bh * D + lane * EPL);
    }

    const long long li = (long long)b * a.len_sb + (long long)h * a.len_sh;
    const int p0 = a.positions[li];
    int n = a.new_lens ? a.new_lens[li] : a.T;
    n = min(n, a.T);
    if (n <= 0) return;
    if (p0 < 0) {
        if (k == 0 && lane == 0 && a.flags) atomic_or_byte(a.flags, b, PFKV_FLAG_BAD_LENGTH);
        return;
    }
    const long long lp = (long long)(p0 / kPage) + k;  // logical page of this unit
    const long long tb = max((long long)p0, lp * kPage) - p0;
    const long long te = min((long long)p0 + n, (lp + 1) * kPage) - p0;
    if (tb >= te) return;  // the call writes nothing into this unit
    if (lp >= a.max_pages) {
        if (lane == 0 && a.flags) atomic_or_byte(a.flags, b, PFKV_FLAG_BAD_LENGTH);
        return;
    }
    const long long bi = (long long)b * a.bt_sb + (long long)h * a.bt_sh + lp;
    const int phys = a.block_tables[bi];
    if (phys < 0 || phys >= a.num_pages) {
        if (lane == 0 && a.flags) atomic_or_byte(a.flags, b, PFKV_FLAG_BAD_PAGE);
        return;
    }
    const long long u = (long long)phys * a.Hkv + h;
    const int slot0 = (int)((p0 + tb) % kPage);
    // the unit's stored scales (used when this call does not open the unit)
    // load in the same round as its tag
    float kscale_st = 1.f, vscale_st = 1.f;
    if (FP8 && slot0 != 0) {
        kscale_st = a.k_scale[u];
        vscale_st = a.v_scale[u];
    }
    if (a.page_tags && a.expected_tags && a.page_tags[u] != a.expected_tags[bi]) {
        if (lane == 0 && a.flags) atomic_or_byte(a.flags, b, PFKV_FLAG_TAG_MISMATCH);
        return;
    }
    const int cnt = (int)(te - tb);
    const long long src_row0 = ((long long)(b * a.Hkv + h) * a.T + tb);
    const __nv_bfloat16 *ksrc = a.k_new + src_row0 * D + lane * EPL;
    const __nv_bfloat16 *vsrc = a.v_new + src_row0 * D + lane * EPL;
    const long long dst_row0 = u * kPage + slot0;

    // element e of this lane's part of row j of the new tokens (K or V)
    auto elem = [&](const __nv_bfloat16 *src, const Vec &pre, int j, int e) {
        if (one) {  // the preloaded row (j is 0)
            uint32_t w;
            if constexpr (EPL == 4) w = e < 2 ? pre.x : pre.y;
            else w = pre;
            return (e & 1) ? __uint_as_float(w & 0xFFFF0000u) : __uint_as_float(w << 16);
        }
        return __bfloat162float(src[(long long)j * D + e]);
    };
    if constexpr (!FP8) {
        Vec *kd = reinterpret_cast<Vec *>(static_cast<__nv_bfloat16 *>(a.k_pages) + dst_row0 * D) + lane;
        Vec *vd = reinterpret_cast<Vec *>(static_cast<__nv_bfloat16 *>(a.v_pages) + dst_row0 * D) + lane;
        if (one) {
            kd[0] = kpre;
            vd[0] = vpre;
        } else {
            for (int j = 0; j < cnt; ++j) {
                kd[j * (D / EPL)] = *reinterpret_cast<const Vec *>(ksrc + (long long)j * D);
                vd[j * (D / EPL)] = *reinterpret_cast<const Vec *>(vsrc + (long long)j * D);
            }
        }
    } else {
        float kscale, vscale;
        if (slot0 == 0) {
            // this call opens the unit: scale from its own tokens in the unit
            float ka = 0.f, va = 0.f;
            for (int j = 0; j < cnt; ++j) {
#pragma unroll
                for (int e = 0; e < EPL; ++e) {
                    ka = fmaxf(ka, fabsf(elem(ksrc, kpre, j, e)));
                    va = fmaxf(va, fabsf(elem(vsrc, vpre, j, e)));
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                ka = fmaxf(ka, __shfl_xor_sync(0xffffffffu, ka, off));
                va = fmaxf(va, __shfl_xor_sync(0xffffffffu, va, off));
            }
            kscale = ka == 0.f ? 1.f : __fdiv_rn(ka, 448.f);
            vscale = va == 0.f ? 1.f : __fdiv_rn(va, 448.f);
            if (lane == 0) {
                a.k_scale[u] = kscale;
                a.v_scale[u] = vscale;
            }
        } else {
            kscale = kscale_st;
            vscale = vscale_st;
        }
        uint8_t *kd = static_cast<uint8_t *>(a.k_pages) + dst_row0 * D + lane * EPL;
        uint8_t *vd = static_cast<uint8_t *>(a.v_pages) + dst_row0 * D + lane * EPL;
        for (int j = 0; j < cnt; ++j) {
            uint32_t kw = 0, vw = 0;
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                const float kx = elem(ksrc, kpre, j, e);
                const float vx = elem(vsrc, vpre, j, e);
                kw |= (uint32_t)float_to_e4m3(__fdiv_rn(kx, kscale)) << (8 * e);
                vw |= (uint32_t)float_to_e4m3(__fdiv_rn(vx, vscale)) << (8 * e);
            }
            if constexpr (EPL == 4) {
                *reinterpret_cast<uint32_t *>(kd + (long long)j * D) = kw;
                *reinterpret_cast<uint32_t *>(vd + (long long)j * D) = vw;
            } else {
                *reinterpret_cast<uint16_t *>(kd + (long long)j * D) = (uint16_t)kw;
                *reinterpret_cast<uint16_t *>(vd + (long long)j * D) = (uint16_t)vw;
            }
        }
    }
}

template <int D, bool FP8>
__global__ void __launch_bounds__(kAppendWarps * 32) kv_append_kernel(AppendArgs a) {
    pdl_enter();
    append_unit<D, FP8>(a, blockIdx.x, blockIdx.y * kAppendWarps + (threadIdx.x >> 5), threadIdx.x & 31);
}

cudaError_t launch_kv_append(const AppendArgs &a, int B, cudaStream_t s) {
    const long long units = ((long long)a.T + 30) / kPage;  // ceil((T + 15) / 16)
    dim3 grid((unsigned)(B * a.Hkv), (unsigned)((units + kAppendWarps - 1) / kAppendWarps));
    dim3 block(kAppendWarps * 32);
    if (a.dtype == PFKV_KV_FP8_E4M3) {
        if (a.D == 128) return launch_pdl(kv_append_kernel<128, true>, grid, block, 0, s, a);
        return launch_pdl(kv_append_kernel<64, true>, grid, block, 0, s, a);
    }
    if (a.D == 128) return launch_pdl(kv_append_kernel<128, false>, grid, block, 0, s, a);
    return launch_pdl(kv_append_kernel<64, false>, grid, block, 0, s, a);
}

// --------------------------------------------------------------------------
// validate: one CTA per (request, kv head, tile of kValTile table entries).
// Bits for the live entries of the tile: LEN for a bad length, PAGE for an id
// outside the pool, TAG when the pool's tag differs from the expected one.
// Written (not OR-ed) to hflags[b][h][tile]; the attention kernels read them
// after this kernel completes.  A thread loads all of its page ids, then all
// of their tags and expected tags, so a tile costs two memory round trips.
// --------------------------------------------------------------------------
// One tile by a CTA of kValThreads threads (every thread must call it).
__device__ __forceinline__ void validate_tile(const DecodeArgs &a, int Hkv, int bh, int tile) {
    const int b = bh / Hkv, h = bh - b * Hkv;
    const int n = a.seq_lens[(long long)b * a.len_sb + (long long)h * a.len_sh];
    // the tile's table entries and expected tags load with the length (every
    // entry below max_pages is in the caller's table); the length then says
    // which of them are live
    const int p0 = tile * kValTile + threadIdx.x;
    const long long row = (long long)b * a.bt_sb + (long long)h * a.bt_sh;
    int id[kValPer];
    uint32_t want[kValPer];
#pragma unroll
    for (int j = 0; j < kValPer; ++j) {
        const int p = p0 + j * kValThreads;
        id[j] = p < a.max_pages ? a.block_tables[row + p] : 0;
        want[j] = p < a.max_pages ? a.expected_tags[row + p] : 0u;
    }
    uint32_t bits = 0;
    if (n < 0 || (long long)n > (long long)a.max_pages * kPage || n > a.max_seq_len) {
        bits = PFKV_FLAG_BAD_LENGTH;
    } else {
        const int np = (n + kPage - 1) / kPage;
        uint32_t tag[kValPer];
#pragma unroll
        for (int j = 0; j < kValPer; ++j) {
            const int p = p0 + j * kValThreads;
            const bool live = p < np;
            const bool in_pool = id[j] >= 0 && id[j] < a.num_pages;
            if (live && !in_pool) bits |= PFKV_FLAG_BAD_PAGE;
            const bool check = live && in_pool;
            tag[j] = check ? a.page_tags[(long long)id[j] * Hkv + h] : 0u;
            if (!check) want[j] = 0u;
        }
#pragma unroll
        for (int j = 0; j < kValPer; ++j)
            if (tag[j] != want[j]) bits |= PFKV_FLAG_TAG_MISMATCH;
    }
    const int any_len = __syncthreads_or(bits & PFKV_FLAG_BAD_LENGTH);
    const int any_page = __syncthreads_or(bits & PFKV_FLAG_BAD_PAGE);
    const int any_tag = __syncthreads_or(bits & PFKV_FLAG_TAG_MISMATCH);
    if (threadIdx.x == 0) {
        uint32_t f = 0;
        if (any_len) f |= PFKV_FLAG_BAD_LENGTH;
        if (any_page) f |= PFKV_FLAG_BAD_PAGE;
        if (any_tag) f |= PFKV_FLAG_TAG_MISMATCH;
        a.hflags[(long long)bh * a.htiles + tile] = f;
    }
}

__global__ void __launch_bounds__(kValThreads) validate_kernel(DecodeArgs a, int Hkv) {
    // wait first, then let the next kernel start: the split kernel relies on
    // it (DecodeArgs::early)
    pdl_enter();
    validate_tile(a, Hkv, blockIdx.x, blockIdx.y);
}

cudaError_t launch_validate(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s) {
    return launch_pdl(validate_kernel, dim3(p.Breq * p.Hkv, p.htiles), dim3(kValThreads), 0, s, a,
                      p.Hkv);
}

// --------------------------------------------------------------------------
// kv_append and validation of one decode step in one launch.  Validation
// reads only the block tables, tags and lengths, never the pool, so the two
// jobs are independent; the first nA CTAs append (kValThreads / 32 warps
// each, one unit per warp) and the others validate one tile each.  Like both
// kernels it waits for its predecessor first, then lets the next kernel
// start (DecodeArgs::early holds as after the validation kernel).
// --------------------------------------------------------------------------
constexpr int kStepAppendWarps = kValThreads / 32;

template <int D, bool FP8>
__global__ void __launch_bounds__(kValThreads) append_validate_kernel(AppendArgs ap, DecodeArgs a, int Hkv,
                                                                      int nA, int ay) {
    pdl_enter();
    if ((int)blockIdx.x < nA) {
        const int bh = blockIdx.x / ay, yy = blockIdx.x - bh * ay;
        append_unit<D, FP8>(ap, bh, yy * kStepAppendWarps + (threadIdx.x >> 5), threadIdx.x & 31);
        return;  // uniform per CTA: no barrier in this branch
    }
    const int i = blockIdx.x - nA;
    validate_tile(a, Hkv, i / a.htiles, i - i / a.htiles * a.htiles);
}

cudaError_t launch_append_validate(const AppendArgs &ap, int B, const DecodeArgs &a, const DecodePlan &p,
                                   cudaStream_t s) {
    const long long units = ((long long)ap.T + 30) / kPage;  // as launch_kv_append
    const int ay = (int)((units + kStepAppendWarps - 1) / kStepAppendWarps);
    const long long nA = (long long)B * ap.Hkv * ay;
    const long long nV = (long long)p.Breq * p.Hkv * p.htiles;
    if (nA + nV > 0x7fffffffLL) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)(nA + nV)), block(kValThreads);
    if (ap.dtype == PFKV_KV_FP8_E4M3) {
        if (ap.D == 128) return launch_pdl(append_validate_kernel<128, true>, grid, block, 0, s, ap, a, p.Hkv, (int)nA, ay);
        return launch_pdl(append_validate_kernel<64, true>, grid, block, 0, s, ap, a, p.Hkv, (int)nA, ay);
    }
    if (ap.D == 128) return launch_pdl(append_validate_kernel<128, false>, grid, block, 0, s, ap, a, p.Hkv, (int)nA, ay);
    return launch_pdl(append_validate_kernel<64, false>, grid, block, 0, s, ap, a, p.Hkv, (int)nA, ay);
}

// --------------------------------------------------------------------------
// e4m3 conversion utilities (the same device conversions the kernels use)
// --------------------------------------------------------------------------
__global__ void e4m3_encode_kernel(const float *x, int64_t n, uint8_t *out) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        out[i] = float_to_e4m3(x[i]);
}

__global__ void e4m3_decode_kernel(const uint8_t *c, int64_t n, float *out) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        out[i] = e4m3x2_to_float2((uint16_t)c[i]).x;
}

static unsigned grid_for(int64_t n) {
    int64_t g = (n + 255) / 256;
    if (g > 152LL * 32) g = 152LL * 32;
    return (unsigned)(g < 1 ? 1 : g);
}

cudaError_t launch_e4m3_encode(const float *x, int64_t n, uint8_t *out, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    e4m3_encode_kernel<<<grid_for(n), 256, 0, s>>>(x, n, out);
    return cudaGetLastError();
}

cudaError_t launch_e4m3_decode(const uint8_t *c, int64_t n, float *out, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    e4m3_decode_kernel<<<grid_for(n), 256, 0, s>>>(c, n, out);
    return cudaGetLastError();
}

cudaError_t preload_append() {
    cudaError_t e = cudaSuccess;
    auto one = [&](cudaError_t r) { if (e == cudaSuccess) e = r; };
    one(preload_kernel(kv_append_kernel<128, true>));
    one(preload_kernel(kv_append_kernel<64, true>));
    one(preload_kernel(kv_append_kernel<128, false>));
    one(preload_kernel(kv_append_kernel<64, false>));
    one(preload_kernel(validate_kernel));
    one(preload_kernel(append_validate_kernel<128, true>));
    one(preload_kernel(append_validate_kernel<64, true>));
    one(preload_kernel(append_validate_kernel<128, false>));
    one(preload_kernel(append_validate_kernel<64, false>));
    one(preload_kernel(e4m3_encode_kernel));
    one(preload_kernel(e4m3_decode_kernel));
    return e;
}

}  // namespace pfkv
