// decode_pers.cu -- persistent, load-balanced split-KV decode attention for
// e4m3 pools with head_dim 128 and query groups of up to 4 heads, plus the
// combine kernel that merges its partial rows.
//
// What is computed is the attention of decode.cu (single query per head over
// the tokens its kv head holds, read through the block table from the FP8
// pool); this file changes how the work is cut and fed:
//
// Segments and balanced ranges.  A segment is one (request b, kv head h,
// chunk c) — c is always 0 unless the caller fixes a split size.  Every CTA
// computes the same exclusive prefix sum of the segments' 16-token units
// (units of a request the validation kernel rejected count as zero).  With U
// units in all and W workers, worker w takes the units
// [ceil(wU/W), ceil((w+1)U/W)): equal shares, crossing segment boundaries, so
// no worker idles while another finishes a long sequence.  A worker writes one
// partial row (normalised output and log2-sum-exp per query head) for every
// segment it touches, at row index segment + worker, which is unique.
//
// Workers.  A worker is a pair of warps sharing a 3-stage shared-memory ring
// (8 KB per stage: K and V slabs of a 2-unit granule, each slab one 2 KB 1-D
// bulk copy; a quarter-warp reads one 128-byte row, so the linear layout is
// free of bank conflicts):
//  * the score warp holds a 16-dim slice of the G query heads in registers
//    (lane (t, c): slice c, row 4r + t of a unit in pass r), converts K bytes
//    to fp32 pairs, takes packed fp32x2 dot products, finishes each score with
//    a select-free reduce-scatter over the 8 lanes of a token group (so lane
//    (t, c) ends with the G scores of token 4c + t) and hands the value warp
//    the raw scores;
//  * the value warp keeps a window of unit metadata (page id, K and V scales,
//    bad-id bit) for the next 64 units in registers, turns the raw scores into
//    probabilities (online softmax per granule, lazy rescale), accumulates
//    its 16-dim slice of the output in registers, writes the partial row at
//    the end of each segment, and refills the stage it has just finished
//    with the bulk copies of the granule ST ahead.
// Splitting scores and values over two warps halves the registers each needs,
// so 12 warps fit an SM, and the two phases of neighbouring granules overlap.
#include <atomic>

#include "pfkv_internal.cuh"

namespace pfkv {

namespace {

__device__ __forceinline__ float pexp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float plog2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float pwarp_max(float x) {
    float m;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(m) : "f"(x));
    return m;
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void named_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void pdequant4(uint32_t w, float2 &lo, float2 &hi) {
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

__device__ __forceinline__ void pdequant16(const uint4 w, float2 (&f)[8]) {
    pdequant4(w.x, f[0], f[1]);
    pdequant4(w.y, f[2], f[3]);
    pdequant4(w.z, f[4], f[5]);
    pdequant4(w.w, f[6], f[7]);
}

constexpr float kLazy = 8.0f;  // rescale only when the max grows by > 2^8

// worker of global unit x when U units are shared by W workers (see header)
__device__ __forceinline__ int worker_of(long long x, long long U, int W) {
    return (int)((x * W) / U);
}

}  // namespace

template <int G>
struct PersCfg {
    static constexpr int D = 128;
    static constexpr int ROWB = 128;
    static constexpr int UNITB = kPage * ROWB;   // 2 KB
    static constexpr int GT = 32;                // tokens per granule (2 units)
    static constexpr int STAGEB = 4 * UNITB;     // K u0 | K u1 | V u0 | V u1
    static constexpr int PAIRS = 6;
    static constexpr int STAGES = 3;
    static constexpr int NT = PAIRS * 64;
    static constexpr int MAXK = 4096;            // segments (prefix array in smem)
    static constexpr int MAXB = 4096;            // requests
    // raw scores of one granule, row = the writing lane (lane (t, c) holds
    // token 4c + t), handed from the score warp to the value warp
    struct alignas(16) SBuf {
        float s[GT][G];
    };
    struct Pair {
        alignas(1024) uint8_t ring[STAGES][STAGEB];
        alignas(16) SBuf sb[STAGES];
        alignas(16) float p[GT][2 * G];   // value warp: probability x V scale, as pairs
        alignas(16) __nv_bfloat16 q[2][G][D];
        alignas(8) uint64_t full[STAGES];
        alignas(8) uint64_t sready[STAGES];
        alignas(8) uint64_t qbar[2];
        int ngran;
        uint32_t score_status;            // timeouts seen by the score warp
    };
    static_assert(sizeof(SBuf) % 16 == 0, "vector stores into every stage buffer");
    struct Smem {
        Pair pair[PAIRS];
        int prefix[MAXK + 1];
        int part[NT];
        uint8_t rflag[MAXB];
        uint8_t last_nv[MAXK];   // tokens in the last unit of each segment
    };
};

// The segment containing global unit x (prefix: exclusive sums, K segments;
// segments with no units never contain a unit).
__device__ __forceinline__ int seg_of(const int *prefix, int K, int x) {
    int lo = 0, hi = K;  // prefix[lo] <= x < prefix[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= x) lo = mid;
        else hi = mid;
    }
    return lo;
}

// MASS: also store every live token's final scores for the attention-mass
// pass (a separate instantiation, so that the plain kernel carries no trace of
// it in its inner loop).
template <int G, bool MASS>
__global__ void __launch_bounds__(PersCfg<G>::NT, 1)
    decode_split_pers_kernel(DecodeArgs a, int Hkv, int B, int nchunks, int chunk_tokens,
                             int *ws_prefix) {
    using C = PersCfg<G>;
    constexpr int ST = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    typename C::Smem &sm = *reinterpret_cast<typename C::Smem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x;
    const int K = B * Hkv * nchunks;
    pdl_enter();

    // ---------------- prologue: request flags, unit prefix sums ----------------
    // B counts virtual requests (see DecodeArgs::kq); rflag is per request
    const int Breq = B / a.kq;
    for (int b = tid; b < Breq; b += C::NT) sm.rflag[b] = 0;
    __syncthreads();
    if (a.hflags) {  // [Breq][Hkv][htiles], read in parallel
        const int per_req = Hkv * a.htiles;
        for (int i = tid; i < Breq * per_req; i += C::NT)
            if (a.hflags[i]) sm.rflag[i / per_req] = 1;
    }
    __syncthreads();
    const int per = (K + C::NT - 1) / C::NT;
    const int k0 = min(K, tid * per), k1 = min(K, k0 + per);
    int local = 0;
    for (int k = k0; k < k1; ++k) {
        const int bh = k / nchunks, c = k - bh * nchunks;
        const int b = bh / Hkv, h = bh - b * Hkv;  // b: virtual request
        const int n = query_len(a, b, h);
        int units = 0, lastnv = 0;
        if (!sm.rflag[b / a.kq] && n >= 0) {
            const int pages = (n + kPage - 1) / kPage;
            const int cp = chunk_tokens / kPage;
            units = max(0, min(pages, (c + 1) * cp) - c * cp);
            const int tok_end = min(n, (c + 1) * chunk_tokens);
            lastnv = tok_end - (tok_end - 1) / kPage * kPage;
        }
        sm.prefix[k] = units;  // the count, turned into the prefix below
        sm.last_nv[k] = (uint8_t)lastnv;
        local += units;
    }
    sm.part[tid] = local;
    __syncthreads();
    if (tid < 32) {  // exclusive scan of the per-thread partials by one warp
        int carry = 0;
        for (int base = 0; base < C::NT; base += 32) {
            const int v = sm.part[base + tid];
            int x = v;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, off);
                if (tid >= off) x += y;
            }
            sm.part[base + tid] = carry + x - v;
            carry += __shfl_sync(0xffffffffu, x, 31);
        }
        if (tid == 0) sm.prefix[K] = carry;
    }
    __syncthreads();
    {
        int run = sm.part[tid];
        for (int k = k0; k < k1; ++k) {  // each thread converts its own range
            const int units = sm.prefix[k];
            sm.prefix[k] = run;
            run += units;
        }
    }
    __syncthreads();
    const int U = sm.prefix[K];  // unit counts stay far below 2^31 (rows < 2^31 / 16)
    // never more workers than units: every worker then owns at least one unit,
    // so all workers between a segment's first and last unit write its rows
    const int W = min((int)gridDim.x * C::PAIRS, U);
    if (blockIdx.x == 0) {
        for (int k = tid; k <= K; k += C::NT) ws_prefix[k] = sm.prefix[k];
    }
    if (U == 0) return;

    // ---------------- the worker ----------------
    // Warps map to the SM's four sub-partitions by warp index mod 4; score
    // warps are 0..PAIRS-1 and value warps PAIRS..2*PAIRS-1 so that the
    // FMA-heavy score warps spread over all four sub-partitions.
    const int warp = tid >> 5, lane = tid & 31;
    const int pi = warp % C::PAIRS;     // pair index in the CTA
    const bool is_score = warp < C::PAIRS;
    typename C::Pair &P = sm.pair[pi];
    const int w = blockIdx.x * C::PAIRS + pi;
    const int x0 = w < W ? (int)(((long long)w * U + W - 1) / W) : U;
    const int x1 = w < W ? (int)(((long long)(w + 1) * U + W - 1) / W) : U;
    const int vt = lane >> 3, vc = lane & 7;

    // granule cursor (2 units, never across a segment), shared logic of both warps
    struct Cursor {
        int x, seg_end, k;
    };
    auto cursor_init = [&](Cursor &c) {
        c.x = x0;
        c.k = seg_of(sm.prefix, K, x0);
        c.seg_end = min(sm.prefix[c.k + 1], x1);
    };
    auto cursor_next = [&](Cursor &c, int n) {
        c.x += n;
        if (c.x >= c.seg_end && c.x < x1) {
            c.k = seg_of(sm.prefix, K, c.x);
            c.seg_end = min(sm.prefix[c.k + 1], x1);
        }
    };

    if (is_score) {
        int ngran = 0;
        if (x0 < x1) {
            int x = x0;
            int k = seg_of(sm.prefix, K, x);
            while (x < x1) {
                const int e = min(sm.prefix[k + 1], x1);
                ngran += (e - x + 1) / 2;
                x = e;
                ++k;
                while (k < K && sm.prefix[k + 1] == sm.prefix[k]) ++k;
            }
        }
        if (lane == 0) {
            P.ngran = ngran;
            P.score_status = 0;
            for (int s = 0; s < ST; ++s) {
                mbar_init(&P.full[s], 1);
                mbar_init(&P.sready[s], 1);
            }
            mbar_init(&P.qbar[0], 1);
            mbar_init(&P.qbar[1], 1);
            fence_mbar_init();
        }
    }
    named_sync(1 + pi, 64);
    const int ngran = P.ngran;
    if (ngran == 0) return;
    const uint64_t policy = l2_policy_evict_first();

    if (is_score) {
        // ===================== score warp =====================
        // q slice of the current segment in registers; K dot products; the
        // reduce-scatter; raw scores to the value warp.
        Cursor con;
        cursor_init(con);
        auto q_copy = [&](int slot, int k) {  // lane 0
            const int bh = k / nchunks;
            const __nv_bfloat16 *src = a.q + (long long)bh * G * C::D;  // (b*Hkv + h)*G rows
            mbar_arrive_expect_tx(&P.qbar[slot], G * C::D * 2);
            bulk_g2s(&P.q[slot][0][0], src, G * C::D * 2, &P.qbar[slot], policy);
        };
        int seg_ord = 0;
        int next_seg_k = -1;
        if (lane == 0) q_copy(0, con.k);
        if (con.seg_end < x1) {
            next_seg_k = seg_of(sm.prefix, K, con.seg_end);
            if (lane == 0) q_copy(1, next_seg_k);
        }
        float2 q2[G][8];
        uint32_t q_phase = 0, status = 0;
        uint32_t parity = 0;  // every stage completes one phase per round of ST granules
        int s = 0;
        bool seg_start = true;
        for (int i = 0; i < ngran; ++i) {
            if (seg_start) {
                const int slot = seg_ord & 1;
                if (!mbar_wait_bounded(&P.qbar[slot], (q_phase >> slot) & 1u)) status |= kStatusTimeout;
                q_phase ^= 1u << slot;
                const __nv_bfloat16 *qs = &P.q[slot][0][0];
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const uint4 w0 = *reinterpret_cast<const uint4 *>(qs + g * C::D + vc * 16);
                    const uint4 w1 = *reinterpret_cast<const uint4 *>(qs + g * C::D + vc * 16 + 8);
                    const uint32_t ws[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float2 f = bf16x2_to_float2(ws[e]);
                        q2[g][e] = make_float2(f.x * a.q_scale, f.y * a.q_scale);
                    }
                }
                __syncwarp();
                // the slot just read is free: prefetch the segment after next
                if (next_seg_k >= 0) {
                    const int e = min(sm.prefix[next_seg_k + 1], x1);
                    const int k2 = e < x1 ? seg_of(sm.prefix, K, e) : -1;
                    if (k2 >= 0 && lane == 0) {
                        fence_proxy_async_smem();
                        q_copy(slot, k2);
                    }
                    next_seg_k = k2;
                }
                seg_start = false;
            }
            const int n_units = min(2, con.seg_end - con.x);
            if (!mbar_wait_bounded(&P.full[s], parity)) status |= kStatusTimeout;
            const uint8_t *stage = P.ring[s];

            // ---- partial dot products and the reduce-scatter ----
            // Lane (vt, vc) ends with the scores of token 4 vc + vt, i.e. pass
            // vc: row 4 (vc & 3) + vt of unit vc >> 2.  The reduce-scatter folds
            // the 8 passes in three levels (xor 4, 2, 1 between lanes); at each
            // level a lane keeps the half named by its own bit of vc (bA, bB, bC:
            // bits 2, 1, 0) and sends the other half.  Computing the passes in a
            // lane-dependent order puts the kept half and the sent half in fixed
            // registers, so no level needs a select: level-1 slot j holds row
            // 4 (j ^ 2 bB ^ bC) + vt, of unit bA (kept) and of unit 1 - bA (sent).
            // Each pair of passes is folded as soon as it is computed, so at most
            // 24 partials are live.
            const int bA = (vc >> 2) & 1, bB = (vc >> 1) & 1, bC = vc & 1;
            const uint8_t *kkeep = stage + bA * C::UNITB + vt * C::ROWB + (vc << 4);
            const uint8_t *ksend = stage + (bA ^ 1) * C::UNITB + vt * C::ROWB + (vc << 4);
            float r1[4][G], r2[2][G], sc[G];
            auto dot_row = [&](const uint8_t *krow, float (&pr)[G]) {
                const uint4 wv = *reinterpret_cast<const uint4 *>(krow);
                float2 kf[8];
                pdequant16(wv, kf);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float2 acc = __fmul2_rn(q2[g][0], kf[0]);
#pragma unroll
                    for (int e = 1; e < 8; ++e) acc = __ffma2_rn(q2[g][e], kf[e], acc);
                    pr[g] = acc.x + acc.y;
                }
            };
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int roff = 4 * (j ^ (2 * bB) ^ bC) * C::ROWB;
                float keep[G], send[G];
                dot_row(kkeep + roff, keep);
                dot_row(ksend + roff, send);
#pragma unroll
                for (int g = 0; g < G; ++g) r1[j][g] = keep[g] + __shfl_xor_sync(0xffffffffu, send[g], 4);
            }
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int g = 0; g < G; ++g)
                    r2[j][g] = r1[j][g] + __shfl_xor_sync(0xffffffffu, r1[j + 2][g], 2);
#pragma unroll
            for (int g = 0; g < G; ++g) sc[g] = r2[0][g] + __shfl_xor_sync(0xffffffffu, r2[1][g], 1);
            // lane (vt, vc) now holds the G raw scores of token 4 vc + vt
            if constexpr (G == 4) {
                *reinterpret_cast<float4 *>(P.sb[s].s[lane]) = make_float4(sc[0], sc[1], sc[2], sc[3]);
            } else if constexpr (G == 2) {
                *reinterpret_cast<float2 *>(P.sb[s].s[lane]) = make_float2(sc[0], sc[1]);
            } else {
                P.sb[s].s[lane][0] = sc[0];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&P.sready[s]);
            const bool seg_end = con.x + n_units >= con.seg_end;
            cursor_next(con, n_units);
            if (seg_end) {
                seg_start = true;
                ++seg_ord;
            }
            if (++s == ST) {
                s = 0;
                parity ^= 1u;
            }
        }
        if (status && lane == 0) atomicOr(&P.score_status, status);
    } else {
        // ===================== value warp =====================
        // unit metadata window: lane l holds unit base + l (cur) and
        // base + 32 + l (nxt): page id (-1 bad, -2 absent) and the two scales
        int base = x0;
        int cphys, nphys;
        float cks, cvs, nks, nvs;
        uint32_t cbad, nbad;
        auto load_ids = [&](int bx, int &phys, uint32_t &bad) {
            const int x = bx + lane;
            phys = -2;
            bad = 0;
            if (x < x1) {
                const int k = seg_of(sm.prefix, K, x);
                const int bh = k / nchunks, c = k - bh * nchunks;
                const int b = bh / Hkv, h = bh - b * Hkv;
                const int page = c * (chunk_tokens / kPage) + (int)(x - sm.prefix[k]);
                const long long bi = table_row(a, b, h) + page;
                const int id = a.block_tables[bi];
                bad = entry_bits(a, id, h, Hkv, bi);
                phys = bad ? -1 : id * Hkv + h;  // unit index
            }
        };
        auto load_scales = [&](int phys, float &ks, float &vs) {
            const long long u = phys >= 0 ? phys : 0;
            ks = a.k_scale[u];
            vs = a.v_scale[u];
        };
        load_ids(base, cphys, cbad);
        load_ids(base + 32, nphys, nbad);
        load_scales(cphys, cks, cvs);
        load_scales(nphys, nks, nvs);
        // metadata of unit x (in [base, base + 64)).  One uniform branch picks
        // the window half (a select would wait for the next half's loads even
        // when only the current one is read).
        struct UnitMeta {
            int phys;
            float ks, vs;
            uint32_t bad;
        };
        auto unit_meta = [&](int x) {
            UnitMeta m;
            const int d = x - base;
            if (d < 32) {
                m.phys = __shfl_sync(0xffffffffu, cphys, d);
                m.ks = __shfl_sync(0xffffffffu, cks, d);
                m.vs = __shfl_sync(0xffffffffu, cvs, d);
                m.bad = __shfl_sync(0xffffffffu, cbad, d);
            } else {
                m.phys = __shfl_sync(0xffffffffu, nphys, d - 32);
                m.ks = __shfl_sync(0xffffffffu, nks, d - 32);
                m.vs = __shfl_sync(0xffffffffu, nvs, d - 32);
                m.bad = __shfl_sync(0xffffffffu, nbad, d - 32);
            }
            return m;
        };
        auto unit_phys = [&](int x) {
            const int d = x - base;
            if (d < 32) return __shfl_sync(0xffffffffu, cphys, d);
            return __shfl_sync(0xffffffffu, nphys, d - 32);
        };
        Cursor iss, con;
        cursor_init(iss);
        cursor_init(con);
        // load (or mark empty) the granule at cursor c into stage s; lane 0 issues
        auto issue_at = [&](const Cursor &c, int s) {
            const int n = min(2, c.seg_end - c.x);
            const int p0 = unit_phys(c.x);
            const int p1 = n == 2 ? unit_phys(c.x + 1) : -2;
            if (lane == 0) {
                if (p0 < 0 && p1 < 0) {
                    mbar_arrive(&P.full[s]);
                } else {
                    uint8_t *dst = P.ring[s];
                    const uint8_t *kp = static_cast<const uint8_t *>(a.k_pages);
                    const uint8_t *vp = static_cast<const uint8_t *>(a.v_pages);
                    mbar_arrive_expect_tx(&P.full[s], (p0 >= 0 ? 2 * C::UNITB : 0) + (p1 >= 0 ? 2 * C::UNITB : 0));
                    if (p0 >= 0) {
                        bulk_g2s(dst, kp + (long long)p0 * C::UNITB, C::UNITB, &P.full[s], policy);
                        bulk_g2s(dst + 2 * C::UNITB, vp + (long long)p0 * C::UNITB, C::UNITB, &P.full[s], policy);
                    }
                    if (p1 >= 0) {
                        bulk_g2s(dst + C::UNITB, kp + (long long)p1 * C::UNITB, C::UNITB, &P.full[s], policy);
                        bulk_g2s(dst + 3 * C::UNITB, vp + (long long)p1 * C::UNITB, C::UNITB, &P.full[s], policy);
                    }
                }
            }
            return n;
        };
        for (int j = 0; j < ST && j < ngran; ++j) cursor_next(iss, issue_at(iss, j));

        float m[G], l[G];
        float2 o[G][8];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            m[g] = -INFINITY;
            l[g] = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) o[g][e] = make_float2(0.f, 0.f);
        }
        uint32_t parity = 0, seg_status = 0;
        int s = 0;
        bool pending_scales = false;
        for (int i = 0; i < ngran; ++i) {
            // metadata window upkeep
            if (pending_scales) {
                load_scales(nphys, nks, nvs);
                pending_scales = false;
            }
            if (con.x >= base + 32) {
                base += 32;
                cphys = nphys; cks = nks; cvs = nvs; cbad = nbad;
                load_ids(base + 32, nphys, nbad);
                pending_scales = true;
            }
            const int n_units = min(2, con.seg_end - con.x);
            const UnitMeta u0m = unit_meta(con.x);
            UnitMeta u1m = {-2, 0.f, 0.f, 0u};
            if (n_units == 2) u1m = unit_meta(con.x + 1);
            seg_status |= u0m.bad | u1m.bad;
            const int seg_last = sm.prefix[con.k + 1] - 1;
            const int lnv = sm.last_nv[con.k];
            const int nv0 = u0m.phys >= 0 ? (con.x == seg_last ? lnv : kPage) : 0;
            const int nv1 = u1m.phys >= 0 ? (con.x + 1 == seg_last ? lnv : kPage) : 0;
            const float ks0 = u0m.ks, ks1 = u1m.ks, vs0 = u0m.vs, vs1 = u1m.vs;

            if (!mbar_wait_bounded(&P.sready[s], parity)) seg_status |= kStatusTimeout;

            // ---- online softmax over the granule (lane: token 4 vc + vt) ----
            const int my_u = vc >> 2, my_row = (4 * vc + vt) & 15;
            const bool ok = my_row < (my_u ? nv1 : nv0);
            const float ksc = my_u ? ks1 : ks0;
            float sc[G];
            if constexpr (G == 4) {
                const float4 v4 = *reinterpret_cast<const float4 *>(P.sb[s].s[lane]);
                sc[0] = v4.x; sc[1] = v4.y; sc[2] = v4.z; sc[3] = v4.w;
            } else if constexpr (G == 2) {
                const float2 v2 = *reinterpret_cast<const float2 *>(P.sb[s].s[lane]);
                sc[0] = v2.x; sc[1] = v2.y;
            } else {
                sc[0] = P.sb[s].s[lane][0];
            }
#pragma unroll
            for (int g = 0; g < G; ++g) sc[g] = ok ? sc[g] * ksc : -INFINITY;
            if (MASS && ok) {  // scores for the attention-mass pass
                const int bh = con.k / nchunks, c = con.k - bh * nchunks;
                const int page = c * (chunk_tokens / kPage) + (con.x + my_u - sm.prefix[con.k]);
                store_scores<G>(a, bh, page * kPage + my_row, sc);
            }
            float mb[G];
            bool grow = false;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                mb[g] = pwarp_max(sc[g]);
                grow |= mb[g] > m[g] + kLazy;
            }
            if (grow) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float mn = fmaxf(m[g], mb[g]);
                    const float alpha = m[g] == -INFINITY ? 0.f : pexp2(m[g] - mn);
                    const float2 a2 = make_float2(alpha, alpha);
                    m[g] = mn;
                    l[g] *= alpha;
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[g][e] = __fmul2_rn(o[g][e], a2);
                }
            }
            {
                const float vsc = my_u ? vs1 : vs0;
                float pp[2 * G];
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float pr = ok ? pexp2(sc[g] - m[g]) : 0.f;
                    l[g] += pr;
                    pp[2 * g] = pp[2 * g + 1] = pr * vsc;
                }
                // rows transposed (t, c) -> 8 t + c: a quarter-warp's stores land
                // in consecutive rows
                float *dstp = P.p[8 * vt + vc];
                if constexpr (G >= 2) {
#pragma unroll
                    for (int x = 0; x < G / 2; ++x)
                        reinterpret_cast<float4 *>(dstp)[x] =
                            make_float4(pp[4 * x], pp[4 * x + 1], pp[4 * x + 2], pp[4 * x + 3]);
                } else {
                    *reinterpret_cast<float2 *>(dstp) = make_float2(pp[0], pp[1]);
                }
            }
            __syncwarp();

            // ---- values: lane (vt, vc) accumulates slice vc over tokens 4r + vt ----
            const uint8_t *stage = P.ring[s];
            auto value_pass = [&](int r) {
                const int row = 4 * (r & 3) + vt;
                const uint8_t *vrow = stage + 2 * C::UNITB + (r >> 2) * C::UNITB + row * C::ROWB;
                const uint4 wv = *reinterpret_cast<const uint4 *>(vrow + (vc << 4));
                float2 vf[8];
                pdequant16(wv, vf);
                // token 4r + vt was scored by lane (t = vt, c = r): row 8 vt + r
                const float2 *ps = reinterpret_cast<const float2 *>(P.p[8 * vt + r]);
                float2 pg[G];
#pragma unroll
                for (int g = 0; g < G; ++g) pg[g] = ps[g];
#pragma unroll
                for (int g = 0; g < G; ++g)
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[g][e] = __ffma2_rn(pg[g], vf[e], o[g][e]);
            };
            if (nv0 == kPage && nv1 == kPage) {
#pragma unroll
                for (int r = 0; r < 8; ++r) value_pass(r);
            } else {
                // tokens past the sequence end or in a missing unit are skipped:
                // their rows may hold stale bytes (even NaN codes)
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const int row = 4 * (r & 3) + vt;
                    if (row < ((r >> 2) ? nv1 : nv0)) value_pass(r);
                }
            }
            const bool seg_end = con.x + n_units >= con.seg_end;
            if (seg_end) {
                // finish the segment: sum the lanes, normalise, write the row
                const int row = con.k + w;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float lt = l[g];
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) lt += __shfl_xor_sync(0xffffffffu, lt, off);
                    const float inv = lt > 0.f ? 1.f / lt : 0.f;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
#pragma unroll
                        for (int off = 8; off < 32; off <<= 1) {
                            o[g][e].x += __shfl_xor_sync(0xffffffffu, o[g][e].x, off);
                            o[g][e].y += __shfl_xor_sync(0xffffffffu, o[g][e].y, off);
                        }
                    }
                    if (vt == 0) {
                        float4 *dst = reinterpret_cast<float4 *>(a.o + ((long long)row * G + g) * C::D + vc * 16);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            dst[e] = make_float4(o[g][2 * e].x * inv, o[g][2 * e].y * inv,
                                                 o[g][2 * e + 1].x * inv, o[g][2 * e + 1].y * inv);
                    }
                    if (lane == 0) a.lse[(long long)row * G + g] = lt > 0.f ? m[g] + plog2(lt) : -INFINITY;
                    m[g] = -INFINITY;
                    l[g] = 0.f;
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[g][e] = make_float2(0.f, 0.f);
                }
                if (lane == 0) a.status[row] = seg_status | P.score_status;
                seg_status = 0;
            }
            // refill this stage with the granule ST ahead
            __syncwarp();
            if (i + ST < ngran) {
                if (lane == 0) fence_proxy_async_smem();
                cursor_next(iss, issue_at(iss, s));
            }
            cursor_next(con, n_units);
            if (++s == ST) {
                s = 0;
                parity ^= 1u;
            }
        }
    }
}

// --------------------------------------------------------------------------
// combine for the persistent layout: the rows of segment k are k + p for the
// workers p that touched it.  One CTA of 16 warps per (request b, kv head h):
//  1. the request's flags: lengths and validation bits of every kv head and
//     the status rows of every segment of the request, in parallel;
//  2. the rows of (b, h), flattened: chunk c owns rows [cstart[c], cstart[c+1])
//     of the flat order, the first at workspace row cbase[c];
//  3. M = max lse per query head, over all rows, in parallel;
//  4. each warp accumulates exp2(lse - M)-weighted rows j = warp, warp + 16, ...
//     (lane l owns dims [4l, 4l + 4) of every query head of the group);
//  5. the warps' sums meet in shared memory; out = sum / weight, bf16.
// --------------------------------------------------------------------------
constexpr int kCombThreads = 512;
constexpr int kCombWarps = kCombThreads / 32;
constexpr int kCombMaxChunks = PersCfg<1>::MAXK;  // segments per (b, h) <= all segments

template <int G>
struct CombSmem {
    union {
        struct {
            int cstart[kCombMaxChunks + 1];
            int cbase[kCombMaxChunks];
        } rows;
        struct {
            float acc[kCombWarps][G][128];
            float wsum[kCombWarps][G];
        } red;
    } u;
    int part[kCombThreads];
    float mred[kCombWarps][G];
    uint32_t flags;
    int ndef;  // segments with long row lists, gathered a warp each
};

template <int G>
__global__ void __launch_bounds__(kCombThreads) decode_combine_pers_kernel(DecodeArgs a, int Hkv,
                                                                          int nchunks, int W,
                                                                          const int *ws_prefix) {
    constexpr int D = 128, NT = kCombThreads, NW = kCombWarps;
    __shared__ CombSmem<G> sm;
    pdl_enter();
    const int b = blockIdx.x / Hkv, h = blockIdx.x - b * Hkv;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = gridDim.x / Hkv;
    const int K = B * Hkv * nchunks;
    const int U = ws_prefix[K];
    W = min(W, U);  // as in the split kernel
    if (tid == 0) {
        sm.flags = 0;
        sm.ndef = 0;
    }
    __syncthreads();

    // ---- 1. request flags (b is a virtual request; the flags belong to the
    //      request rb and cover all of its query tokens) ----
    const int rb = b / a.kq, v0 = rb * a.kq;
    uint32_t f = 0;
    for (int i = tid; i < Hkv; i += NT)
        if (query_len(a, v0, i) < 0) f |= PFKV_FLAG_BAD_LENGTH;
    if (a.hflags)
        for (int i = tid; i < Hkv * a.htiles; i += NT) f |= a.hflags[(long long)rb * Hkv * a.htiles + i];
    // rows of the request's segments (rejected requests have none): a thread
    // per segment; a segment with many rows (few long segments, many workers
    // each) is deferred to a warp whose lanes take its rows.  The deferred
    // list borrows the row tables' space, which phase 2 fills later.
    if (U > 0) {
        for (int it = tid; it < a.kq * Hkv * nchunks; it += NT) {
            const int k = v0 * Hkv * nchunks + it;
            const int u0 = ws_prefix[k], u1 = ws_prefix[k + 1];
            if (u1 == u0) continue;
            const int p0 = worker_of(u0, U, W), p1 = worker_of(u1 - 1, U, W);
            if (p1 - p0 < 8) {
                for (int p = p0; p <= p1; ++p) f |= a.status[k + p];
            } else {
                sm.u.rows.cbase[atomicAdd(&sm.ndef, 1)] = k;
            }
        }
    }
    if (f) atomicOr(&sm.flags, f);
    __syncthreads();
    f = 0;
    for (int d = warp; d < sm.ndef; d += NW) {
        const int k = sm.u.rows.cbase[d];
        const int p0 = worker_of(ws_prefix[k], U, W), p1 = worker_of(ws_prefix[k + 1] - 1, U, W);
        for (int p = p0 + lane; p <= p1; p += 32) f |= a.status[k + p];
    }
    if (f) atomicOr(&sm.flags, f);
    __syncthreads();
    const uint32_t flags = sm.flags;
    if (b == v0 && h == 0 && tid == 0 && a.flags) a.flags[rb] = (uint8_t)flags;
    if (b == v0 && h == 0 && tid == 0 && a.rflags) a.rflags[rb] = (uint8_t)flags;
    const int n = max(0, query_len(a, b, h));
    uint2 *out = reinterpret_cast<uint2 *>(a.out + (long long)(b * Hkv + h) * G * D);
    if (flags != 0 || n == 0 || U == 0) {
        for (int i = tid; i < G * D / 4; i += NT) out[i] = make_uint2(0u, 0u);
        return;
    }

    // ---- 2. flat row order: per-thread chunk ranges, scanned by one warp ----
    const int kbase = (b * Hkv + h) * nchunks;
    const int per = (nchunks + NT - 1) / NT;
    const int c0 = min(nchunks, tid * per), c1 = min(nchunks, c0 + per);
    int local = 0;
    for (int c = c0; c < c1; ++c) {
        const int k = kbase + c;
        const int u0 = ws_prefix[k], u1 = ws_prefix[k + 1];
        int cnt = 0, base = 0;
        if (u1 > u0) {
            const int p0 = worker_of(u0, U, W), p1 = worker_of(u1 - 1, U, W);
            cnt = p1 - p0 + 1;
            base = k + p0;
        }
        sm.u.rows.cstart[c] = cnt;  // the count, turned into the start below
        sm.u.rows.cbase[c] = base;
        local += cnt;
    }
    sm.part[tid] = local;
    __syncthreads();
    if (tid < 32) {
        int carry = 0;
        for (int base = 0; base < NT; base += 32) {
            const int v = sm.part[base + tid];
            int x = v;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, off);
                if (tid >= off) x += y;
            }
            sm.part[base + tid] = carry + x - v;
            carry += __shfl_sync(0xffffffffu, x, 31);
        }
        if (tid == 0) sm.u.rows.cstart[nchunks] = carry;
    }
    __syncthreads();
    {
        int run = sm.part[tid];
        for (int c = c0; c < c1; ++c) {
            const int cnt = sm.u.rows.cstart[c];
            sm.u.rows.cstart[c] = run;
            run += cnt;
        }
    }
    __syncthreads();
    const int R = sm.u.rows.cstart[nchunks];
    // workspace row of flat row j (chunks with no rows never contain j)
    auto row_of = [&](int j) {
        int lo = 0, hi = nchunks;  // cstart[lo] <= j < cstart[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (sm.u.rows.cstart[mid] <= j) lo = mid;
            else hi = mid;
        }
        return sm.u.rows.cbase[lo] + (j - sm.u.rows.cstart[lo]);
    };

    // ---- 3. M per query head (thread tid always sees head tid % G) ----
    const int gm = tid % G;
    float mx = -INFINITY;
    for (int idx = tid; idx < R * G; idx += NT) mx = fmaxf(mx, a.lse[(long long)row_of(idx / G) * G + gm]);
#pragma unroll
    for (int off = 16; off >= G; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane < G) sm.mred[warp][lane] = mx;
    __syncthreads();
    float M[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        M[g] = sm.mred[0][g];
#pragma unroll
        for (int w2 = 1; w2 < NW; ++w2) M[g] = fmaxf(M[g], sm.mred[w2][g]);
    }

    // ---- 4. weighted sums, rows spread over the warps ----
    float4 acc[G];
    float wsum[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        acc[g] = make_float4(0.f, 0.f, 0.f, 0.f);
        wsum[g] = 0.f;
    }
#pragma unroll 4
    for (int j = warp; j < R; j += NW) {
        const long long row = row_of(j);
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float lc = a.lse[row * G + g];
            const float wt = lc == -INFINITY ? 0.f : pexp2(lc - M[g]);
            const float4 ov = *reinterpret_cast<const float4 *>(a.o + (row * G + g) * D + lane * 4);
            wsum[g] += wt;
            acc[g].x = fmaf(wt, ov.x, acc[g].x);
            acc[g].y = fmaf(wt, ov.y, acc[g].y);
            acc[g].z = fmaf(wt, ov.z, acc[g].z);
            acc[g].w = fmaf(wt, ov.w, acc[g].w);
        }
    }
    __syncthreads();  // the row tables are dead: their space takes the sums
#pragma unroll
    for (int g = 0; g < G; ++g) {
        *reinterpret_cast<float4 *>(&sm.u.red.acc[warp][g][lane * 4]) = acc[g];
        if (lane == 0) sm.u.red.wsum[warp][g] = wsum[g];
    }
    __syncthreads();

    // ---- 5. out = sum over warps / weight over warps ----
    for (int i = tid; i < G * D / 4; i += NT) {
        const int g = i / (D / 4), d4 = i - g * (D / 4);
        float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
        float ws = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < NW; ++w2) {
            const float4 v = *reinterpret_cast<const float4 *>(&sm.u.red.acc[w2][g][d4 * 4]);
            s4.x += v.x;
            s4.y += v.y;
            s4.z += v.z;
            s4.w += v.w;
            ws += sm.u.red.wsum[w2][g];
        }
        const float inv = ws > 0.f ? 1.f / ws : 0.f;
        if (a.lse_fin && d4 == 0) {
            float Mg = M[0];  // M[g] without a dynamically indexed register array
#pragma unroll
            for (int x = 1; x < G; ++x) Mg = g == x ? M[x] : Mg;
            a.lse_fin[(long long)(b * Hkv + h) * G + g] = ws > 0.f ? Mg + plog2(ws) : -INFINITY;
        }
        const __nv_bfloat162 lo = __floats2bfloat162_rn(s4.x * inv, s4.y * inv);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(s4.z * inv, s4.w * inv);
        out[i] = make_uint2(*reinterpret_cast<const uint32_t *>(&lo),
                            *reinterpret_cast<const uint32_t *>(&hi));
    }
}

// --------------------------------------------------------------------------
// host side
// --------------------------------------------------------------------------
namespace {

template <int G, bool MASS>
cudaError_t launch_pers_gm(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s) {
    using C = PersCfg<G>;
    const size_t smem = sizeof(typename C::Smem) + 1024;
    static std::atomic<unsigned long long> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(decode_split_pers_kernel<G, MASS>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    return launch_pdl(decode_split_pers_kernel<G, MASS>, dim3(p.pers_ctas), dim3(C::NT), smem, s,
                      a, p.Hkv, p.B, p.nchunks, p.chunk_tokens, a.ws_prefix);
}

template <int G>
cudaError_t launch_pers_g(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s) {
    return a.mscore ? launch_pers_gm<G, true>(a, p, s) : launch_pers_gm<G, false>(a, p, s);
}

}  // namespace

int pers_workers_per_cta() { return PersCfg<4>::PAIRS; }

bool pers_supported(const DecodePlan &p, int num_pages) {
    const long long rows = (long long)num_pages * p.Hkv * kPage;
    const long long K = (long long)p.B * p.Hkv * p.nchunks;
    return p.dtype == PFKV_KV_FP8_E4M3 && p.D == 128 && p.G <= 4 && rows < (1LL << 31) &&
           K <= PersCfg<4>::MAXK && p.Breq <= PersCfg<4>::MAXB;
}

cudaError_t launch_split_pers(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s) {
    switch (p.G) {
        case 1: return launch_pers_g<1>(a, p, s);
        case 2: return launch_pers_g<2>(a, p, s);
        case 4: return launch_pers_g<4>(a, p, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_combine_pers(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s) {
    const int W = p.pers_ctas * PersCfg<4>::PAIRS;
    const dim3 grid((unsigned)(p.B * p.Hkv));
    switch (p.G) {
        case 1: return launch_pdl(decode_combine_pers_kernel<1>, grid, dim3(kCombThreads), 0, s, a, p.Hkv, p.nchunks, W, (const int *)a.ws_prefix);
        case 2: return launch_pdl(decode_combine_pers_kernel<2>, grid, dim3(kCombThreads), 0, s, a, p.Hkv, p.nchunks, W, (const int *)a.ws_prefix);
        case 4: return launch_pdl(decode_combine_pers_kernel<4>, grid, dim3(kCombThreads), 0, s, a, p.Hkv, p.nchunks, W, (const int *)a.ws_prefix);
    }
    return cudaErrorInvalidValue;
}

}  // namespace pfkv
