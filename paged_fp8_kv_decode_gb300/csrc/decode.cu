// decode.cu -- split-KV paged decode attention (decode_split) and the
// online-softmax combine of the chunks (decode_combine), sm_103a.
//
// What is computed: single-query attention for every (request, query head)
// over the tokens its kv head holds, read through a block table of integer
// page indices ("Workers AI targets the inference bottleneck", section "KV
// cache compression goes open source") from a pool stored as FP8 e4m3 or
// BF16 ("Cloudflare quantizes Kimi and GLM caches for 41% faster inference",
// 2nd paragraph).  Decode is a memory-bound matrix-vector product ("How we
// built the most efficient inference engine for Cloudflare's network",
// section "Batching to feed the Tensor Cores"), so the kernels are laid out
// for HBM bandwidth on CUDA cores, not for tensor cores.
//
// decode_split: one CTA per (request b, kv head h, chunk c).  Its warps take
// the chunk's 16-token units round robin.  Each warp owns a ring of STAGES
// shared-memory stages; lane 0 fills a stage with two 1-D bulk copies (the K
// and V slabs of a unit, contiguous in the pool layout) completing on the
// stage's mbarrier.  All G query heads of the kv head share every loaded slab
// (GQA).  Lane layout per pass: LPT lanes split one token's head_dim, TPP
// tokens per pass; e4m3 codes are converted to fp32 in registers and the
// unit's fp32 scale is applied once per score (K) and once per probability (V).
// Each warp keeps its own online-softmax state (running max in log2 units,
// per-lane partial sums); at the end the warps are merged through shared
// memory and the chunk's normalised output and log2-sum-exp are written to
// the workspace.
//
// decode_combine: one CTA per (b, query head): merges the chunks of the head
// with weights exp2(lse_c - max lse), writes bf16 output, and writes the
// request's flags (tag/bounds bits of the validation kernel, page-id and
// timeout bits of the split kernel, length bits), zeroing flagged requests.
#include <atomic>
#include <cfloat>

#include "pfkv_internal.cuh"

namespace pfkv {

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float fast_log2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int D, int G, bool FP8>
struct SplitCfg {
    static constexpr int KB = FP8 ? 1 : 2;         // bytes per element
    static constexpr int E = (G <= 4) ? 16 : 8;    // elements per lane per token
    static constexpr int LPT = D / E;              // lanes per token
    static constexpr int TPP = 32 / LPT;           // tokens per pass
    static constexpr int NPASS = kPage / TPP;      // passes per unit
    static constexpr int VB = E * KB;              // bytes per lane per token row
    static constexpr int ROWB = D * KB;            // bytes per token row
    static constexpr int UNITB = kPage * ROWB;     // bytes of one K (or V) slab
    static constexpr int STAGEB = 2 * UNITB;       // K + V slab
    static constexpr int NWARPS = 4;
    static constexpr int STAGES = (16384 / STAGEB) < 2 ? 2 : (16384 / STAGEB);
    static constexpr int MAXU = 8192 / kPage / NWARPS;  // units per warp at the max chunk
    static_assert(LPT >= 1 && LPT <= 32 && TPP * LPT == 32, "lane layout");
    static_assert(NPASS * TPP == kPage, "pass layout");
    static_assert(VB == 8 || VB == 16 || VB == 32, "vector width");

    // head-dim index of element e of the lane with in-token index c
    __device__ static constexpr int dim(int c, int e) {
        return VB <= 16 ? c * E + e : (e / 8) * (LPT * 8) + c * 8 + (e % 8);
    }

    struct Smem {
        alignas(128) uint8_t ring[NWARPS][STAGES][STAGEB];
        float merge_o[NWARPS][G][D];
        float merge_m[NWARPS][G];
        float merge_l[NWARPS][G];
        int phys[NWARPS][MAXU];
        float kscale[NWARPS][MAXU];
        float vscale[NWARPS][MAXU];
        alignas(8) uint64_t bar[NWARPS][STAGES];
        uint32_t status;
    };
};

// Load the lane's E elements of token row `row` of a slab in shared memory
// and convert them to fp32.
template <class C, bool FP8>
__device__ __forceinline__ void load_row(const uint8_t *slab, int row, int c, float (&v)[C::E]) {
    const uint8_t *p = slab + row * C::ROWB;
    if constexpr (FP8) {
        if constexpr (C::VB == 16) {
            const uint4 w = *reinterpret_cast<const uint4 *>(p + c * 16);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 lo = e4m3x2_to_float2((uint16_t)(ws[i] & 0xFFFF));
                const float2 hi = e4m3x2_to_float2((uint16_t)(ws[i] >> 16));
                v[4 * i + 0] = lo.x;
                v[4 * i + 1] = lo.y;
                v[4 * i + 2] = hi.x;
                v[4 * i + 3] = hi.y;
            }
        } else {
            const uint2 w = *reinterpret_cast<const uint2 *>(p + c * 8);
            const uint32_t ws[2] = {w.x, w.y};
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float2 lo = e4m3x2_to_float2((uint16_t)(ws[i] & 0xFFFF));
                const float2 hi = e4m3x2_to_float2((uint16_t)(ws[i] >> 16));
                v[4 * i + 0] = lo.x;
                v[4 * i + 1] = lo.y;
                v[4 * i + 2] = hi.x;
                v[4 * i + 3] = hi.y;
            }
        }
    } else {
        constexpr int PIECES = C::VB / 16;  // 16-byte pieces (8 bf16 each)
#pragma unroll
        for (int pc = 0; pc < PIECES; ++pc) {
            const uint4 w = *reinterpret_cast<const uint4 *>(p + pc * (C::LPT * 16) + c * 16);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = bf16x2_to_float2(ws[i]);
                v[pc * 8 + 2 * i] = f.x;
                v[pc * 8 + 2 * i + 1] = f.y;
            }
        }
    }
}

template <int D, int G, bool FP8>
__global__ void __launch_bounds__(SplitCfg<D, G, FP8>::NWARPS * 32)
    decode_split_kernel(DecodeArgs a, int Hkv, int chunk_tokens, int nchunks) {
    using C = SplitCfg<D, G, FP8>;
    constexpr int NW = C::NWARPS, ST = C::STAGES;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    typename C::Smem &sm = *reinterpret_cast<typename C::Smem *>(smem_raw);
    pdl_enter();

    const int BH = gridDim.x / nchunks;
    const int chunk = blockIdx.x / BH;
    const int bh = blockIdx.x - chunk * BH;
    const int b = bh / Hkv, h = bh - b * Hkv;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = lane / C::LPT, c = lane % C::LPT;

    // b is the virtual request (see DecodeArgs::kq)
    const int n = query_len(a, b, h);
    if (n < 0) return;
    const int tok0 = chunk * chunk_tokens;
    if (tok0 >= n) return;  // empty item
    if (request_rejected_cta(a, b / a.kq, Hkv)) return;  // rejected by the validation kernel
    const int tok1 = min(n, tok0 + chunk_tokens);
    const int p_begin = tok0 / kPage;
    const int npages = (tok1 - tok0 + kPage - 1) / kPage;
    const int nmine = warp < npages ? (npages - warp + NW - 1) / NW : 0;
    const long long bt_row = table_row(a, b, h);

    if (threadIdx.x == 0) sm.status = 0;
    // ---- per-warp unit metadata: page ids first (they gate the copies) ----
    uint32_t bad = 0;
    for (int i = lane; i < nmine; i += 32) {
        const long long bi = bt_row + p_begin + warp + i * NW;
        const int phys = a.block_tables[bi];
        const uint32_t eb = entry_bits(a, phys, h, Hkv, bi);
        bad |= eb;
        sm.phys[warp][i] = eb ? -1 : phys;
    }
    if (lane == 0) {
        for (int s = 0; s < ST; ++s) mbar_init(&sm.bar[warp][s], 1);
        fence_mbar_init();
    }
    __syncwarp();

    const uint64_t policy = l2_policy_evict_first();
    const uint8_t *kpool = static_cast<const uint8_t *>(a.k_pages);
    const uint8_t *vpool = static_cast<const uint8_t *>(a.v_pages);
    auto issue = [&](int i) {  // lane 0: bulk-copy unit i of this warp into its stage
        const int phys = sm.phys[warp][i];
        if (phys < 0) return;
        const int s = i % ST;
        const long long off = ((long long)phys * Hkv + h) * C::UNITB;
        uint8_t *dst = sm.ring[warp][s];
        mbar_arrive_expect_tx(&sm.bar[warp][s], C::STAGEB);
        bulk_g2s(dst, kpool + off, C::UNITB, &sm.bar[warp][s], policy);
        bulk_g2s(dst + C::UNITB, vpool + off, C::UNITB, &sm.bar[warp][s], policy);
    };
    if (lane == 0) {
        for (int i = 0; i < ST && i < nmine; ++i) issue(i);
    }
    // scales (only consumers need them; gathered while the copies fly)
    if constexpr (FP8) {
        for (int i = lane; i < nmine; i += 32) {
            const int phys = sm.phys[warp][i];
            const long long uidx = (long long)(phys < 0 ? 0 : phys) * Hkv + h;
            sm.kscale[warp][i] = a.k_scale[uidx];
            sm.vscale[warp][i] = a.v_scale[uidx];
        }
    }

    // ---- query: G heads x E elements, pre-scaled into log2 units ----
    float qr[G][C::E];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const __nv_bfloat16 *qp = a.q + ((long long)b * (Hkv * G) + h * G + g) * D;
#pragma unroll
        for (int e = 0; e < C::E; ++e) qr[g][e] = __bfloat162float(qp[C::dim(c, e)]) * a.q_scale;
    }
    __syncwarp();

    float m[G], l[G], o[G][C::E];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
#pragma unroll
        for (int e = 0; e < C::E; ++e) o[g][e] = 0.f;
    }

    uint32_t phase = 0;  // per-stage parity bits
    bool timed_out = false;
    int i = 0;
    for (; i < nmine; ++i) {
        const int s = i % ST;
        const int phys = sm.phys[warp][i];
        if (phys >= 0) {
            if (!mbar_wait_bounded(&sm.bar[warp][s], (phase >> s) & 1u)) {
                timed_out = true;
                break;
            }
            phase ^= 1u << s;
            const uint8_t *ks_slab = sm.ring[warp][s];
            const uint8_t *vs_slab = ks_slab + C::UNITB;
            const float ksc = FP8 ? sm.kscale[warp][i] : 1.f;
            const float vsc = FP8 ? sm.vscale[warp][i] : 1.f;
            const int unit_tok0 = (p_begin + warp + i * NW) * kPage;
            const int valid = min(kPage, tok1 - unit_tok0);

            // scores of this unit's tokens for all G heads (log2 units)
            float sc[C::NPASS][G];
#pragma unroll
            for (int r = 0; r < C::NPASS; ++r) {
                float kv[C::E];
                load_row<C, FP8>(ks_slab, r * C::TPP + t, c, kv);
                float acc[G];
#pragma unroll
                for (int g = 0; g < G; ++g) acc[g] = 0.f;
#pragma unroll
                for (int e = 0; e < C::E; ++e)
#pragma unroll
                    for (int g = 0; g < G; ++g) acc[g] = fmaf(qr[g][e], kv[e], acc[g]);
#pragma unroll
                for (int off = 1; off < C::LPT; off <<= 1)
#pragma unroll
                    for (int g = 0; g < G; ++g) acc[g] += __shfl_xor_sync(0xffffffffu, acc[g], off);
                const bool ok = r * C::TPP + t < valid;
#pragma unroll
                for (int g = 0; g < G; ++g) sc[r][g] = ok ? acc[g] * ksc : -INFINITY;
                if (a.mscore && ok && c == 0) store_scores<G>(a, bh, unit_tok0 + r * C::TPP + t, sc[r]);
            }
            // block maximum and (rare) rescale of the running state
            float mb[G];
            bool grow = false;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float x = sc[0][g];
#pragma unroll
                for (int r = 1; r < C::NPASS; ++r) x = fmaxf(x, sc[r][g]);
#pragma unroll
                for (int off = C::LPT; off < 32; off <<= 1)
                    x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
                mb[g] = x;
                grow |= x > m[g];
            }
            if (grow) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float mn = fmaxf(m[g], mb[g]);
                    const float alpha = fast_exp2(m[g] - mn);
                    m[g] = mn;
                    l[g] *= alpha;
#pragma unroll
                    for (int e = 0; e < C::E; ++e) o[g][e] *= alpha;
                }
            }
            // probabilities and the value accumulation
            float pv[C::NPASS][G];
#pragma unroll
            for (int r = 0; r < C::NPASS; ++r)
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float p = fast_exp2(sc[r][g] - m[g]);
                    l[g] += p;
                    pv[r][g] = p * vsc;
                }
#pragma unroll
            for (int r = 0; r < C::NPASS; ++r) {
                if (r * C::TPP + t < valid) {
                    float vv[C::E];
                    load_row<C, FP8>(vs_slab, r * C::TPP + t, c, vv);
#pragma unroll
                    for (int e = 0; e < C::E; ++e)
#pragma unroll
                        for (int g = 0; g < G; ++g) o[g][e] = fmaf(pv[r][g], vv[e], o[g][e]);
                }
            }
        }
        __syncwarp();
        if (lane == 0 && i + ST < nmine) {
            fence_proxy_async_smem();
            issue(i + ST);
        }
    }
    if (timed_out) {
        // drain the copies this warp still has in flight (bounded), then stop
        for (int k = i; k < nmine && k < i + ST; ++k) {
            const int s = k % ST;
            if (sm.phys[warp][k] >= 0) {
                if (mbar_wait_bounded(&sm.bar[warp][s], (phase >> s) & 1u)) phase ^= 1u << s;
            }
        }
        bad |= kStatusTimeout;
    }

    // ---- warp totals: sum the per-token-lane partials ----
#pragma unroll
    for (int off = C::LPT; off < 32; off <<= 1) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            l[g] += __shfl_xor_sync(0xffffffffu, l[g], off);
#pragma unroll
            for (int e = 0; e < C::E; ++e) o[g][e] += __shfl_xor_sync(0xffffffffu, o[g][e], off);
        }
    }
    if (t == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < C::E; ++e) sm.merge_o[warp][g][C::dim(c, e)] = o[g][e];
    }
    if (lane == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            sm.merge_m[warp][g] = m[g];
            sm.merge_l[warp][g] = l[g];
        }
    }
    bad = __reduce_or_sync(0xffffffffu, bad);
    if (lane == 0 && bad) atomicOr(&sm.status, bad);
    __syncthreads();

    // ---- merge the warps; write the chunk's normalised output and lse ----
    const long long row0 = ((long long)b * (Hkv * G) + h * G) * nchunks + chunk;
    for (int x = threadIdx.x; x < G * D; x += NW * 32) {
        const int g = x / D, d = x - g * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, sm.merge_m[w][g]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float wt = sm.merge_m[w][g] == -INFINITY ? 0.f : fast_exp2(sm.merge_m[w][g] - M);
            L += sm.merge_l[w][g] * wt;
            O += sm.merge_o[w][g][d] * wt;
        }
        const long long row = row0 + (long long)g * nchunks;
        a.o[row * D + d] = L > 0.f ? O / L : 0.f;
        if (d == 0) a.lse[row] = L > 0.f ? M + fast_log2(L) : -INFINITY;
    }
    if (threadIdx.x == 0) a.status[(long long)bh * nchunks + chunk] = sm.status;
}

// --------------------------------------------------------------------------
// combine
// --------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(DecodeArgs a, int Hkv, int G,
                                                            int chunk_tokens, int nchunks) {
    __shared__ uint32_t s_flags;
    __shared__ float s_red[D / 32];
    pdl_enter();
    const int Hq = Hkv * G;
    const int b = blockIdx.x / Hq, hq = blockIdx.x - b * Hq, h = hq / G;
    const int tid = threadIdx.x;
    if (tid == 0) s_flags = 0;
    __syncthreads();

    // b is the virtual request (see DecodeArgs::kq); the flags belong to the
    // request rb and cover all of its query tokens
    const int rb = b / a.kq, v0 = rb * a.kq;
    // request flags: lengths and validation bits of every kv head ...
    uint32_t f = 0;
    for (int i = tid; i < Hkv; i += D)
        if (query_len(a, v0, i) < 0) f |= PFKV_FLAG_BAD_LENGTH;
    if (a.hflags)
        for (int i = tid; i < Hkv * a.htiles; i += D) f |= a.hflags[(long long)rb * Hkv * a.htiles + i];
    if (f) atomicOr(&s_flags, f);
    __syncthreads();
    // ... then the split kernel's per-chunk status (only written for live
    // chunks of requests the validation kernel passed)
    if (s_flags == 0) {
        f = 0;
        for (int v = v0; v < v0 + a.kq; ++v)
            for (int i = 0; i < Hkv; ++i) {
                const int ni = query_len(a, v, i);
                const int nch = (ni + chunk_tokens - 1) / chunk_tokens;
                for (int cc = tid; cc < nch; cc += D) f |= a.status[(long long)(v * Hkv + i) * nchunks + cc];
            }
        if (f) atomicOr(&s_flags, f);
        __syncthreads();
    }
    const uint32_t flags = s_flags;
    if (b == v0 && hq == 0 && tid == 0 && a.flags) a.flags[rb] = (uint8_t)flags;
    if (b == v0 && hq == 0 && tid == 0 && a.rflags) a.rflags[rb] = (uint8_t)flags;

    const int n = max(0, query_len(a, b, h));
    __nv_bfloat16 *out = a.out + ((long long)b * Hq + hq) * D;
    if (flags != 0 || n == 0) {
        out[tid] = __float2bfloat16_rn(0.f);
        return;
    }
    const int nch = (n + chunk_tokens - 1) / chunk_tokens;
    const long long row0 = ((long long)b * Hq + hq) * nchunks;
    const float *lse = a.lse + row0;
    const float *o = a.o + row0 * D;
    if (nch == 1) {
        if (a.lse_fin && tid == 0) a.lse_fin[(long long)b * Hq + hq] = lse[0];
        out[tid] = __float2bfloat16_rn(o[tid]);
        return;
    }
    float M = -INFINITY;
    for (int cc = tid; cc < nch; cc += D) M = fmaxf(M, lse[cc]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    if ((tid & 31) == 0) s_red[tid >> 5] = M;
    __syncthreads();
    M = s_red[0];
#pragma unroll
    for (int w = 1; w < D / 32; ++w) M = fmaxf(M, s_red[w]);
    float acc = 0.f, wsum = 0.f;
    for (int cc = 0; cc < nch; ++cc) {
        const float lc = lse[cc];
        const float w = lc == -INFINITY ? 0.f : fast_exp2(lc - M);
        wsum += w;
        acc = fmaf(w, o[(long long)cc * D + tid], acc);
    }
    if (a.lse_fin && tid == 0)
        a.lse_fin[(long long)b * Hq + hq] = wsum > 0.f ? M + __log2f(wsum) : -INFINITY;
    out[tid] = __float2bfloat16_rn(wsum > 0.f ? acc / wsum : 0.f);
}

// --------------------------------------------------------------------------
// launch
// --------------------------------------------------------------------------
// the dynamic shared-memory opt-in is per device; set it once on each
template <int D, int G, bool FP8>
static cudaError_t configure_split() {
    static std::atomic<unsigned long long> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(decode_split_kernel<D, G, FP8>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)sizeof(typename SplitCfg<D, G, FP8>::Smem));
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    return cudaSuccess;
}

template <int D, int G, bool FP8>
static cudaError_t launch_split_t(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s) {
    using C = SplitCfg<D, G, FP8>;
    const size_t smem = sizeof(typename C::Smem);
    cudaError_t e = configure_split<D, G, FP8>();
    if (e != cudaSuccess) return e;
    const long long items = (long long)p.B * p.Hkv * p.nchunks;
    return launch_pdl(decode_split_kernel<D, G, FP8>, dim3((unsigned)items), dim3(C::NWARPS * 32),
                      smem, s, a, p.Hkv, p.chunk_tokens, p.nchunks);
}

template <int D, int G>
static cudaError_t launch_split_dt(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s) {
    return p.dtype == PFKV_KV_FP8_E4M3 ? launch_split_t<D, G, true>(a, p, s)
                                       : launch_split_t<D, G, false>(a, p, s);
}

template <int D>
static cudaError_t launch_split_g(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s) {
    switch (p.G) {
        case 1: return launch_split_dt<D, 1>(a, p, s);
        case 2: return launch_split_dt<D, 2>(a, p, s);
        case 4: return launch_split_dt<D, 4>(a, p, s);
        case 8: return launch_split_dt<D, 8>(a, p, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_split(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s) {
    if (p.kind == 1) return launch_split_pers(a, p, s);
    return p.D == 128 ? launch_split_g<128>(a, p, s) : launch_split_g<64>(a, p, s);
}

template <int D>
static cudaError_t preload_split_d() {
    cudaError_t e = cudaSuccess;
    auto one = [&](cudaError_t r) { if (e == cudaSuccess) e = r; };
    one(configure_split<D, 1, true>());
    one(configure_split<D, 2, true>());
    one(configure_split<D, 4, true>());
    one(configure_split<D, 8, true>());
    one(configure_split<D, 1, false>());
    one(configure_split<D, 2, false>());
    one(configure_split<D, 4, false>());
    one(configure_split<D, 8, false>());
    one(preload_kernel(decode_combine_kernel<D>));
    return e;
}

cudaError_t preload_split_generic() {
    cudaError_t e = preload_split_d<128>();
    if (e == cudaSuccess) e = preload_split_d<64>();
    return e;
}

cudaError_t launch_combine(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s) {
    if (p.kind == 1) return launch_combine_pers(a, p, s);
    const unsigned grid = (unsigned)(p.B * p.Hq);
    if (p.D == 128)
        return launch_pdl(decode_combine_kernel<128>, dim3(grid), dim3(128), 0, s, a, p.Hkv, p.G,
                          p.chunk_tokens, p.nchunks);
    return launch_pdl(decode_combine_kernel<64>, dim3(grid), dim3(64), 0, s, a, p.Hkv, p.G,
                      p.chunk_tokens, p.nchunks);
}

}  // namespace pfkv
