// decode_swz.cu -- split-KV paged decode attention for e4m3 pools with
// head_dim 128 and query groups of up to 4 heads (the Llama-3.1-8B shape),
// fed by 2-D TMA tile loads with the 128-byte shared-memory swizzle.
//
// Same computation and workspace contract as decode_split_kernel in
// decode.cu (single-query attention over the tokens a kv head holds, read
// through the block table from the FP8 pool; partial results per chunk), with
// a layout chosen to cut instructions and shared-memory traffic per byte:
//  * work granule = 2 units = 32 tokens.  Lane (t, c) owns head_dim slice c
//    (16 dims) of the G query heads in registers and, in pass r, token 4r + t.
//    K rows arrive through TMA with the 128-byte swizzle (16-byte chunk c of
//    row j stored at chunk c ^ j%8); a quarter-warp reads one row, so the
//    swizzle keeps the reads conflict-free.
//  * e4m3 pairs -> fp32 pairs in registers, packed fp32x2 FMAs.
//  * the 8 lanes of a token group finish each score with a reduce-scatter
//    (xor 4, 2, 1): afterwards lane (t, c) holds all G scores of token 4c + t,
//    so each lane computes G exponentials per granule and no score is
//    computed twice.
//  * online softmax once per granule: per-head warp max (redux.sync.max.f32),
//    lazy rescale (only when the running max grows by more than 2^8).
//  * values: lane (t, c) accumulates dims of slice c over tokens 4r + t,
//    reading each token's probabilities (times the unit's V scale) as
//    ready-made pairs from shared memory.
// Each warp owns a 3-stage ring (8 KB per stage: K and V of 2 units) that its
// lane 0 fills with TMA tile loads completing on the stage's mbarrier.
#include <atomic>
#include <cuda.h>

#include "pfkv_internal.cuh"

namespace pfkv {

namespace {

__device__ __forceinline__ float fexp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float flog2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float warp_max(float x) {
    float m;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(m) : "f"(x));
    return m;
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Four e4m3 codes of a 32-bit word -> four exact fp32 values (two pairs),
// through the hardware e4m3x2 -> f16x2 conversion on each 16-bit half of the
// word and f16 -> f32; register halves are addressed directly.
__device__ __forceinline__ void dequant4(uint32_t w, float2 &lo, float2 &hi) {
    asm("{\n\t.reg .b16 l, h, a0, a1, b0, b1;\n\t.reg .b32 x, y;\n\t"
        "mov.b32 {l, h}, %4;\n\t"
        "cvt.rn.f16x2.e4m3x2 x, l;\n\t"
        "cvt.rn.f16x2.e4m3x2 y, h;\n\t"
        "mov.b32 {a0, a1}, x;\n\t"
        "mov.b32 {b0, b1}, y;\n\t"
        "cvt.f32.f16 %0, a0;\n\t"
        "cvt.f32.f16 %1, a1;\n\t"
        "cvt.f32.f16 %2, b0;\n\t"
        "cvt.f32.f16 %3, b1;\n\t}"
        : "=f"(lo.x), "=f"(lo.y), "=f"(hi.x), "=f"(hi.y)
        : "r"(w));
}

// 16 e4m3 codes (one swizzle chunk) -> 8 fp32 pairs (exact values)
__device__ __forceinline__ void dequant16(const uint4 w, float2 (&f)[8]) {
    dequant4(w.x, f[0], f[1]);
    dequant4(w.y, f[2], f[3]);
    dequant4(w.z, f[4], f[5]);
    dequant4(w.w, f[6], f[7]);
}

constexpr float kLazyRescale = 8.0f;  // log2 units

}  // namespace

template <int G>
struct SwzCfg {
    static constexpr int D = 128;
    static constexpr int ROWB = 128;               // e4m3 row of head_dim 128
    static constexpr int UNITB = kPage * ROWB;     // 2 KB slab
    static constexpr int GU = 2;                   // units per granule
    static constexpr int GT = GU * kPage;          // 32 tokens: one per lane
    static constexpr int STAGEB = 2 * GU * UNITB;  // K u0 | K u1 | V u0 | V u1
    static constexpr int NWARPS = 4;
    static constexpr int STAGES = 3;
    static constexpr int MAXGR = 8192 / GT / NWARPS;
    static constexpr int MAXU = MAXGR * GU;
    struct Smem {
        alignas(1024) uint8_t ring[NWARPS][STAGES][STAGEB];
        alignas(16) float p[NWARPS][GT][2 * G];
        int phys[NWARPS][MAXU];
        float kscale[NWARPS][MAXU];
        float vscale[NWARPS][MAXU];
        alignas(8) uint64_t bar[NWARPS][STAGES];
        uint32_t status;
    };
    // per-warp merge record, written into the warp's own (drained) ring
    struct Merge {
        float o[G][D];
        float m[G];
        float l[G];
    };
    static_assert(sizeof(Merge) <= STAGES * STAGEB, "merge record fits the ring");
};

template <int G>
__global__ void __launch_bounds__(SwzCfg<G>::NWARPS * 32)
    decode_split_swz_kernel(const __grid_constant__ CUtensorMap tmk,
                            const __grid_constant__ CUtensorMap tmv, DecodeArgs a, int Hkv,
                            int chunk_tokens, int nchunks) {
    using C = SwzCfg<G>;
    constexpr int NW = C::NWARPS, ST = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    typename C::Smem &sm = *reinterpret_cast<typename C::Smem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    pdl_enter();

    const int BH = gridDim.x / nchunks;
    const int chunk = blockIdx.x / BH;
    const int bh = blockIdx.x - chunk * BH;
    const int b = bh / Hkv, h = bh - b * Hkv;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // b is the virtual request (see DecodeArgs::kq)
    const int n = query_len(a, b, h);
    if (n < 0) return;
    const int tok0 = chunk * chunk_tokens;
    if (tok0 >= n) return;
    if (request_rejected_cta(a, b / a.kq, Hkv)) return;  // rejected by the validation kernel
    const int tok1 = min(n, tok0 + chunk_tokens);
    const int p_begin = tok0 / kPage;
    const int nunits = (tok1 - tok0 + kPage - 1) / kPage;
    const int ngr = (nunits + C::GU - 1) / C::GU;
    const int nmine = warp < ngr ? (ngr - warp + NW - 1) / NW : 0;
    const long long bt_row = table_row(a, b, h);

    // ---- unit metadata of this warp's granules (page ids gate the copies) ----
    uint32_t bad = 0;
    for (int k = lane; k < C::GU * nmine; k += 32) {
        const int u = C::GU * (warp + (k / C::GU) * NW) + (k % C::GU);  // unit within chunk
        int phys = -2;                                                    // absent
        if (u < nunits) {
            const long long bi = bt_row + p_begin + u;
            phys = a.block_tables[bi];
            const uint32_t eb = entry_bits(a, phys, h, Hkv, bi);
            if (eb) {
                bad |= eb;
                phys = -1;
            }
        }
        sm.phys[warp][k] = phys;
    }
    if (lane == 0) {
        for (int s = 0; s < ST; ++s) mbar_init(&sm.bar[warp][s], 1);
        fence_mbar_init();
    }
    if (threadIdx.x == 0) sm.status = 0;
    __syncthreads();
    const int vt = lane >> 3, vc = lane & 7;  // token in pass, 16-dim slice
    // ---- query slice of the G heads, pre-scaled to log2 units ----
    float2 q2[G][8];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const __nv_bfloat16 *qp = a.q + ((long long)b * (Hkv * G) + h * G + g) * C::D + vc * 16;
        const uint4 w0 = *reinterpret_cast<const uint4 *>(qp);
        const uint4 w1 = *reinterpret_cast<const uint4 *>(qp + 8);
        const uint32_t ws[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float2 f = bf16x2_to_float2(ws[e]);
            q2[g][e] = make_float2(f.x * a.q_scale, f.y * a.q_scale);
        }
    }

    const uint64_t policy = l2_policy_evict_first();
    auto issue = [&](int i) {  // lane 0: TMA the K and V slabs of granule i
        const int s = i % ST;
        const int p0 = sm.phys[warp][C::GU * i], p1 = sm.phys[warp][C::GU * i + 1];
        const uint32_t bytes = (p0 >= 0 ? 2 * C::UNITB : 0) + (p1 >= 0 ? 2 * C::UNITB : 0);
        if (bytes == 0) return;
        uint8_t *dst = sm.ring[warp][s];
        mbar_arrive_expect_tx(&sm.bar[warp][s], bytes);
        if (p0 >= 0) {
            const int row = (p0 * Hkv + h) * kPage;
            tma_load_2d(dst, &tmk, 0, row, &sm.bar[warp][s], policy);
            tma_load_2d(dst + 2 * C::UNITB, &tmv, 0, row, &sm.bar[warp][s], policy);
        }
        if (p1 >= 0) {
            const int row = (p1 * Hkv + h) * kPage;
            tma_load_2d(dst + C::UNITB, &tmk, 0, row, &sm.bar[warp][s], policy);
            tma_load_2d(dst + 3 * C::UNITB, &tmv, 0, row, &sm.bar[warp][s], policy);
        }
    };
    if (lane == 0) {
        for (int i = 0; i < ST && i < nmine; ++i) issue(i);
    }
    for (int k = lane; k < C::GU * nmine; k += 32) {
        const int phys = sm.phys[warp][k];
        const long long uidx = (long long)(phys < 0 ? 0 : phys) * Hkv + h;
        sm.kscale[warp][k] = a.k_scale[uidx];
        sm.vscale[warp][k] = a.v_scale[uidx];
    }
    __syncwarp();

    // per-warp online-softmax state
    float m[G], l[G];
    float2 o[G][8];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) o[g][e] = make_float2(0.f, 0.f);
    }
    uint32_t phase = 0;
    bool timed_out = false;
    int i = 0;
    for (; i < nmine; ++i) {
        const int s = i % ST;
        const int p0 = sm.phys[warp][C::GU * i], p1 = sm.phys[warp][C::GU * i + 1];
        if (p0 >= 0 || p1 >= 0) {
            if (!mbar_wait_bounded(&sm.bar[warp][s], (phase >> s) & 1u)) {
                timed_out = true;
                break;
            }
            phase ^= 1u << s;
            const uint8_t *stage = sm.ring[warp][s];
            const int gtok0 = (p_begin + C::GU * (warp + i * NW)) * kPage;
            const bool u0 = p0 >= 0, u1 = p1 >= 0;
            const bool full = u0 && u1 && gtok0 + C::GT <= tok1;

            // ---- scores: partial dot products of slice vc, token 4r + vt ----
            float part[8][G];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int row = 4 * (r & 3) + vt;
                const uint8_t *krow = stage + (r >> 2) * C::UNITB + row * C::ROWB;
                const uint4 w = *reinterpret_cast<const uint4 *>(krow + ((vc ^ (row & 7)) << 4));
                float2 kf[8];
                dequant16(w, kf);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float2 acc = __fmul2_rn(q2[g][0], kf[0]);
#pragma unroll
                    for (int e = 1; e < 8; ++e) acc = __ffma2_rn(q2[g][e], kf[e], acc);
                    part[r][g] = acc.x + acc.y;
                }
            }
            // reduce-scatter over the 8 lanes of the token group: lane vc ends
            // with the full scores of pass r = vc (token 4 vc + vt)
            const bool bA = vc & 4, bB = vc & 2, bC = vc & 1;
            float r1[4][G], r2[2][G], sc[G];
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float snd = bA ? part[r][g] : part[r + 4][g];
                    const float kp = bA ? part[r + 4][g] : part[r][g];
                    r1[r][g] = kp + __shfl_xor_sync(0xffffffffu, snd, 4);
                }
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float snd = bB ? r1[r][g] : r1[r + 2][g];
                    const float kp = bB ? r1[r + 2][g] : r1[r][g];
                    r2[r][g] = kp + __shfl_xor_sync(0xffffffffu, snd, 2);
                }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float snd = bC ? r2[0][g] : r2[1][g];
                const float kp = bC ? r2[1][g] : r2[0][g];
                sc[g] = kp + __shfl_xor_sync(0xffffffffu, snd, 1);
            }
            const int my_tok = 4 * vc + vt;       // token (in granule) whose scores I hold
            const int my_u = vc >> 2;
            {
                const bool ok = (my_u ? u1 : u0) && gtok0 + my_tok < tok1;
                const float ksc = sm.kscale[warp][C::GU * i + my_u];
#pragma unroll
                for (int g = 0; g < G; ++g) sc[g] = ok ? sc[g] * ksc : -INFINITY;
                if (a.mscore && ok) store_scores<G>(a, bh, gtok0 + my_tok, sc);
            }
            // ---- online softmax over the granule ----
            float mb[G];
            bool grow = false;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                mb[g] = warp_max(sc[g]);
                grow |= mb[g] > m[g] + kLazyRescale;
            }
            if (grow) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float mn = fmaxf(m[g], mb[g]);
                    const float alpha = fexp2(m[g] - mn);
                    const float2 a2 = make_float2(alpha, alpha);
                    m[g] = mn;
                    l[g] *= alpha;
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[g][e] = __fmul2_rn(o[g][e], a2);
                }
            }
            {
                const float vsc = sm.vscale[warp][C::GU * i + my_u];
                float pp[2 * G];
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float p = fexp2(sc[g] - m[g]);
                    l[g] += p;
                    pp[2 * g] = pp[2 * g + 1] = p * vsc;
                }
                if constexpr (G >= 2) {
                    float4 *dstp = reinterpret_cast<float4 *>(sm.p[warp][my_tok]);
#pragma unroll
                    for (int x = 0; x < G / 2; ++x)
                        dstp[x] = make_float4(pp[4 * x], pp[4 * x + 1], pp[4 * x + 2], pp[4 * x + 3]);
                } else {
                    *reinterpret_cast<float2 *>(sm.p[warp][my_tok]) = make_float2(pp[0], pp[1]);
                }
            }
            __syncwarp();
            // ---- values: lane (vt, vc) accumulates slice vc over tokens 4r + vt ----
            auto value_pass = [&](int r) {
                const int tl = 4 * r + vt;
                const int row = 4 * (r & 3) + vt;
                const uint8_t *vrow = stage + 2 * C::UNITB + (r >> 2) * C::UNITB + row * C::ROWB;
                const uint4 w = *reinterpret_cast<const uint4 *>(vrow + ((vc ^ (row & 7)) << 4));
                float2 vf[8];
                dequant16(w, vf);
                float2 pg[G];
                const float2 *ps = reinterpret_cast<const float2 *>(sm.p[warp][tl]);
#pragma unroll
                for (int g = 0; g < G; ++g) pg[g] = ps[g];
#pragma unroll
                for (int g = 0; g < G; ++g)
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[g][e] = __ffma2_rn(pg[g], vf[e], o[g][e]);
            };
            if (full) {
#pragma unroll
                for (int r = 0; r < 8; ++r) value_pass(r);
            } else {
                // tokens past the sequence end or in a missing unit are skipped:
                // their rows may hold stale bytes (even NaN codes)
                const int nv0 = u0 ? min(16, tok1 - gtok0) : 0;
                const int nv1 = u1 ? min(16, tok1 - gtok0 - 16) : 0;
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const int row = 4 * (r & 3) + vt;
                    if (row < ((r >> 2) ? nv1 : nv0)) value_pass(r);
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
        for (int k = i; k < nmine && k < i + ST; ++k) {
            const int s = k % ST;
            if (sm.phys[warp][C::GU * k] >= 0 || sm.phys[warp][C::GU * k + 1] >= 0) {
                if (mbar_wait_bounded(&sm.bar[warp][s], (phase >> s) & 1u)) phase ^= 1u << s;
            }
        }
        bad |= kStatusTimeout;
    }

    // ---- warp totals ----
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) l[g] += __shfl_xor_sync(0xffffffffu, l[g], off);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
#pragma unroll
            for (int off = 8; off < 32; off <<= 1) {
                o[g][e].x += __shfl_xor_sync(0xffffffffu, o[g][e].x, off);
                o[g][e].y += __shfl_xor_sync(0xffffffffu, o[g][e].y, off);
            }
        }
    }
    __syncwarp();
    typename C::Merge &mine = *reinterpret_cast<typename C::Merge *>(sm.ring[warp][0]);
    if (vt == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                mine.o[g][vc * 16 + 2 * e] = o[g][e].x;
                mine.o[g][vc * 16 + 2 * e + 1] = o[g][e].y;
            }
    }
    if (lane == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            mine.m[g] = m[g];
            mine.l[g] = l[g];
        }
    }
    bad = __reduce_or_sync(0xffffffffu, bad);
    if (lane == 0 && bad) atomicOr(&sm.status, bad);
    __syncthreads();

    // ---- merge the warps; write the chunk's normalised output and lse ----
    const long long row0 = ((long long)b * (Hkv * G) + h * G) * nchunks + chunk;
    for (int x = threadIdx.x; x < G * C::D; x += NW * 32) {
        const int g = x / C::D, d = x - g * C::D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w)
            M = fmaxf(M, reinterpret_cast<const typename C::Merge *>(sm.ring[w][0])->m[g]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const typename C::Merge &mw = *reinterpret_cast<const typename C::Merge *>(sm.ring[w][0]);
            const float wt = mw.m[g] == -INFINITY ? 0.f : fexp2(mw.m[g] - M);
            L += mw.l[g] * wt;
            O += mw.o[g][d] * wt;
        }
        const long long row = row0 + (long long)g * nchunks;
        a.o[row * C::D + d] = L > 0.f ? O / L : 0.f;
        if (d == 0) a.lse[row] = L > 0.f ? M + flog2(L) : -INFINITY;
    }
    if (threadIdx.x == 0) a.status[(long long)bh * nchunks + chunk] = sm.status;
}

// --------------------------------------------------------------------------
// host side: tensor maps over the pools and the launch
// --------------------------------------------------------------------------
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::atomic<EncodeTiledFn> fn{nullptr};
    EncodeTiledFn f = fn.load(std::memory_order_acquire);
    if (!f) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !p) {
            cudaGetLastError();
            return nullptr;
        }
        f = reinterpret_cast<EncodeTiledFn>(p);
        fn.store(f, std::memory_order_release);
    }
    return f;
}

// 2-D map over an e4m3 pool: rows of 128 bytes (one token of one kv head),
// boxes of 16 rows (one unit), 128-byte swizzle.
bool encode_pool_map(CUtensorMap *map, const void *pool, long long rows) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    cuuint64_t dims[2] = {128, (cuuint64_t)rows};
    cuuint64_t strides[1] = {128};
    cuuint32_t box[2] = {128, (cuuint32_t)kPage};
    cuuint32_t estr[2] = {1, 1};
    return f(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(pool), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int G>
cudaError_t configure_swz() {
    static std::atomic<unsigned long long> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(decode_split_swz_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)(sizeof(typename SwzCfg<G>::Smem) + 1024));
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    return cudaSuccess;
}

template <int G>
cudaError_t launch_swz_g(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s) {
    using C = SwzCfg<G>;
    const size_t smem = sizeof(typename C::Smem) + 1024;
    cudaError_t e = configure_swz<G>();
    if (e != cudaSuccess) return e;
    CUtensorMap tk, tv;
    const long long rows = (long long)a.num_pages * p.Hkv * kPage;
    if (!encode_pool_map(&tk, a.k_pages, rows) || !encode_pool_map(&tv, a.v_pages, rows))
        return cudaErrorInvalidValue;
    const long long items = (long long)p.B * p.Hkv * p.nchunks;
    return launch_pdl(decode_split_swz_kernel<G>, dim3((unsigned)items), dim3(C::NWARPS * 32), smem,
                      s, tk, tv, a, p.Hkv, p.chunk_tokens, p.nchunks);
}

}  // namespace

bool swz_supported(const DecodePlan &p, int num_pages) {
    // TMA row coordinates are 32-bit
    const long long rows = (long long)num_pages * p.Hkv * kPage;
    return p.dtype == PFKV_KV_FP8_E4M3 && p.D == 128 && p.G <= 4 && rows < (1LL << 31);
}

cudaError_t preload_split_swz() {
    cudaError_t e = configure_swz<1>();
    if (e == cudaSuccess) e = configure_swz<2>();
    if (e == cudaSuccess) e = configure_swz<4>();
    return e;
}

cudaError_t launch_split_swz(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s) {
    switch (p.G) {
        case 1: return launch_swz_g<1>(a, p, s);
        case 2: return launch_swz_g<2>(a, p, s);
        case 4: return launch_swz_g<4>(a, p, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace pfkv
