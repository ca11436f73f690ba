// combine_pers.cu -- merge the partial rows of the persistent split kernel
// (decode_pers.cu) into the output, with the request flags.
//
// The split kernel writes, for every segment k (request b, kv head h, chunk c)
// and every worker p that took units of it, the normalised partial output and
// the log2-sum-exp of each query head at row k + p, and the status bits of
// that worker's part at status[k + p].  The workers of segment k are
// pers_worker_of(first unit) .. pers_worker_of(last unit).  The combine takes
//   out = sum_rows 2^(lse - M) o / sum_rows 2^(lse - M),   M = max_rows lse,
// per query head, rounded to bf16, and zeroes every head of a request whose
// validation bits, lengths or status rows carry a flag.
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

// VL consecutive floats (4 or 2: one vector load)
template <int VL>
__device__ __forceinline__ void load_vec(float (&v)[VL], const float *p) {
    if constexpr (VL == 4) {
        const float4 t = *reinterpret_cast<const float4 *>(p);
        v[0] = t.x, v[1] = t.y, v[2] = t.z, v[3] = t.w;
    } else {
        const float2 t = *reinterpret_cast<const float2 *>(p);
        v[0] = t.x, v[1] = t.y;
    }
}

template <int VL>
__device__ __forceinline__ void store_vec(float *p, const float (&v)[VL]) {
    if constexpr (VL == 4) *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
    else *reinterpret_cast<float2 *>(p) = make_float2(v[0], v[1]);
}

}  // namespace

// --------------------------------------------------------------------------
// One CTA of NW warps per (request b, kv head h) and group of GS of its G
// query heads.  A head with one chunk and few rows takes one CTA of 8 warps
// for all G query heads (GS = G); a head with many chunks or many rows takes
// CTAs of 16 warps, one per group of GS query heads, with GS as small as keeps
// all CTAs in one wave, so that the rows' bytes spread over as many SMs as
// there are:
//  1. before the wait for the split kernel: the request's lengths and
//     validation words, and the unit prefix of every segment of the request
//     (the split kernel's prologue arithmetic on the same lengths, so the
//     same integers); the chunks of (b, h) are scanned into a flat row order
//     (chunk c owns flat rows [cstart[c], cstart[c+1])).  A CTA starts as soon
//     as the split kernel's CTA on its SM has ended, so this part overlaps the
//     split kernel's last workers.  Where the grid's share of length loads
//     would be large (kCombEarlyLoads), the prefix is read from the split
//     kernel's copy after the wait instead;
//  2. after the wait: the status rows of the request's segments (a thread per
//     segment; lists of 8 or more rows go to a warp each) and the rows of
//     (b, h): warp w merges flat rows w, w + NW, ..., several at a time with
//     their loads issued together, with a running max per query head (lane l
//     owns dims [l D / 32, (l + 1) D / 32) of every head);
//  the warps' (max, weight, sum) meet in shared memory; out = sum / weight,
//  bf16, or zeros if the request carries a flag.
//
// Before its wait the kernel reads only the call's inputs and the validation
// words: the validation kernel had completed when the split kernel passed its
// own wait, and the split kernel lets this kernel launch only after that.
// --------------------------------------------------------------------------
constexpr int kCombMaxChunks = kPersMaxSegments;  // segments per (b, h) <= all segments
constexpr int kCombShortList = 8;                  // status rows a thread gathers itself
constexpr int kCombMaxDeferred = 256;              // longer lists handed to warps
constexpr long long kCombEarlyLoads = 1LL << 20;   // segments x CTAs for the early prefix

template <int GS, int NW, int D>
struct CombSmem {
    union {
        struct {
            int pfx[kCombMaxChunks + 1];     // unit prefix at the request's segments
            int cstart[kCombMaxChunks + 1];  // flat row order of the chunks of (b, h)
        } rows;
        struct {
            float acc[NW][GS][D];
            float wsum[NW][GS];
            float wmax[NW][GS];
        } red;
    } u;
    int part[NW * 32];
    int defk[kCombMaxDeferred];
    uint32_t flags;
    int ndef, U;
};

// Exclusive scan of one int per thread over the block (NT threads, one warp
// scans the per-thread values); returns this thread's prefix, and the total
// in *total.  Ends with the block synchronised.
template <int NT>
__device__ __forceinline__ int block_exclusive_scan(int v, int *part, int *total) {
    const int tid = threadIdx.x;
    part[tid] = v;
    __syncthreads();
    if (tid < 32) {
        int carry = 0;
        for (int base = 0; base < NT; base += 32) {
            const int x0 = part[base + tid];
            int x = x0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, off);
                if (tid >= off) x += y;
            }
            part[base + tid] = carry + x - x0;
            carry += __shfl_sync(0xffffffffu, x, 31);
        }
        if (tid == 0) *total = carry;
    }
    __syncthreads();
    return part[tid];
}

template <int G, int GS, int NW, int D>
__global__ void __launch_bounds__(NW * 32, 16 / NW) decode_combine_pers_kernel(DecodeArgs a, int Hkv,
                                                                          int nchunks, int chunk_tokens,
                                                                          int W, const int *ws_prefix) {
    static_assert(G % GS == 0, "query-head groups split G evenly");
    static_assert(D == 128 || D == 64, "head_dim 128 or 64");
    constexpr int NT = NW * 32, HG = G / GS, VL = D / 32;
    __shared__ CombSmem<GS, NW, D> sm;
    // CTA (b, h, gi) merges query heads gi GS .. gi GS + GS - 1 of (b, h)
    const int bhx = blockIdx.x / HG, gi = blockIdx.x - bhx * HG, g0 = gi * GS;
    const int b = bhx / Hkv, h = bhx - b * Hkv;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = gridDim.x / (Hkv * HG);
    const int K = B * Hkv * nchunks;
    const bool early = (long long)K * gridDim.x <= kCombEarlyLoads;  // uniform
    if (!early) pdl_enter();
    if (tid == 0) {
        sm.flags = 0;
        sm.ndef = 0;
    }

    // ---- 1. request flags (b is a virtual request; the flags belong to the
    //      request rb and cover all of its query tokens), the unit prefix at
    //      the request's segments, the chunks of (b, h) ----
    const int rb = b / a.kq, v0 = rb * a.kq;
    uint32_t f = 0;
    for (int i = tid; i < Hkv; i += NT)
        if (query_len(a, v0, i) < 0) f |= PFKV_FLAG_BAD_LENGTH;
    if (a.hflags)
        for (int i = tid; i < Hkv * a.htiles; i += NT) f |= a.hflags[(long long)rb * Hkv * a.htiles + i];
    const int nseg = a.kq * Hkv * nchunks, kseg0 = v0 * Hkv * nchunks;
    int *pfx = sm.u.rows.pfx;  // pfx[i]: first unit of segment kseg0 + i (i <= nseg)
    if (early) {
        const int per = (K + NT - 1) / NT;
        const int k0 = min(K, tid * per), k1 = min(K, k0 + per);
        int local = 0, nbh = -1, n = 0;
        for (int k = k0; k < k1; ++k) {
            const int bh = k / nchunks;
            if (bh != nbh) {
                n = query_len(a, bh / Hkv, bh - bh / Hkv * Hkv);
                nbh = bh;
            }
            local += segment_units(n, k - bh * nchunks, chunk_tokens);
        }
        int run = block_exclusive_scan<NT>(local, sm.part, &sm.U);
        nbh = -1;
        for (int k = k0; k < k1; ++k) {
            const int bh = k / nchunks;
            if (bh != nbh) {
                n = query_len(a, bh / Hkv, bh - bh / Hkv * Hkv);
                nbh = bh;
            }
            if (k >= kseg0 && k <= kseg0 + nseg) pfx[k - kseg0] = run;
            run += segment_units(n, k - bh * nchunks, chunk_tokens);
        }
        if (kseg0 + nseg == K && tid == 0) pfx[nseg] = sm.U;  // the request's end is the end
    } else {
        for (int i = tid; i <= nseg; i += NT) pfx[i] = ws_prefix[kseg0 + i];
        if (tid == 0) sm.U = ws_prefix[K];
    }
    __syncthreads();
    const int U = sm.U;
    W = min(W, U);  // as in the split kernel
    // status rows of this thread's segment (one segment per thread covers
    // every request of up to NT segments; more go round the loop below)
    int sk = -1, sp0 = 0, scnt = 0;
    if (U > 0 && tid < nseg) {
        const int u0 = pfx[tid], u1 = pfx[tid + 1];
        if (u1 > u0) {
            sk = kseg0 + tid;
            sp0 = pers_worker_of(u0, U, W);
            scnt = pers_worker_of(u1 - 1, U, W) - sp0 + 1;
        }
    }
    const int kbase = (b * Hkv + h) * nchunks, cb = kbase - kseg0;  // chunk c: pfx[cb + c]
    const int per = (nchunks + NT - 1) / NT;
    const int c0 = min(nchunks, tid * per), c1 = min(nchunks, c0 + per);
    int local = 0;
    for (int c = c0; c < c1; ++c) {
        const int u0 = pfx[cb + c], u1 = pfx[cb + c + 1];
        if (U > 0 && u1 > u0) local += pers_worker_of(u1 - 1, U, W) - pers_worker_of(u0, U, W) + 1;
    }
    {
        int run = block_exclusive_scan<NT>(local, sm.part, &sm.u.rows.cstart[nchunks]);
        for (int c = c0; c < c1; ++c) {
            const int u0 = pfx[cb + c], u1 = pfx[cb + c + 1];
            sm.u.rows.cstart[c] = run;
            if (U > 0 && u1 > u0) run += pers_worker_of(u1 - 1, U, W) - pers_worker_of(u0, U, W) + 1;
        }
    }
    __syncthreads();
    // Each chunk's first workspace row (its first worker writes row
    // kbase + c + the worker's index), written over the chunk's unit prefix,
    // which nothing reads any more: one division per chunk, not per row.
    int *crow = pfx + cb;
    for (int c = c0; c < c1; ++c) crow[c] = kbase + c + (U > 0 ? pers_worker_of(crow[c], U, W) : 0);
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
        return (long long)crow[lo] + (j - sm.u.rows.cstart[lo]);
    };
    if (early) pdl_enter();  // what follows reads the split kernel's results

    // ---- 2. status rows (loaded now, used after the merge) and the rows ----
    uint32_t st[kCombShortList];
#pragma unroll
    for (int i = 0; i < kCombShortList; ++i) st[i] = 0u;
    if (scnt > 0 && scnt <= kCombShortList) {
#pragma unroll
        for (int i = 0; i < kCombShortList; ++i)
            if (i < scnt) st[i] = a.status[sk + sp0 + i];
    }
    float M[GS], S[GS];
    float acc[GS][VL];
#pragma unroll
    for (int g = 0; g < GS; ++g) {
        M[g] = -INFINITY;
        S[g] = 0.f;
#pragma unroll
        for (int v = 0; v < VL; ++v) acc[g][v] = 0.f;
    }
    constexpr int RB = GS == 8 ? 1 : GS == 1 ? 8 : 4;  // rows in flight per warp (registers)
    for (int j0 = warp; j0 < R; j0 += RB * NW) {
        float lc[RB][GS];
        float ov[RB][GS][VL];
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            const int j = j0 + r * NW;
            const long long row = j < R ? row_of(j) : 0;
#pragma unroll
            for (int g = 0; g < GS; ++g) {
                lc[r][g] = j < R ? a.lse[row * G + g0 + g] : -INFINITY;
                if (j < R) {
                    load_vec<VL>(ov[r][g], a.o + (row * G + g0 + g) * D + lane * VL);
                } else {
#pragma unroll
                    for (int v = 0; v < VL; ++v) ov[r][g][v] = 0.f;
                }
            }
        }
#pragma unroll
        for (int r = 0; r < RB; ++r) {
#pragma unroll
            for (int g = 0; g < GS; ++g) {
                if (lc[r][g] == -INFINITY) continue;  // uniform: no token of this head in the row
                if (lc[r][g] > M[g]) {
                    const float sc = M[g] == -INFINITY ? 0.f : pexp2(M[g] - lc[r][g]);
                    S[g] *= sc;
#pragma unroll
                    for (int v = 0; v < VL; ++v) acc[g][v] *= sc;
                    M[g] = lc[r][g];
                }
                const float wt = pexp2(lc[r][g] - M[g]);
                S[g] += wt;
#pragma unroll
                for (int v = 0; v < VL; ++v) acc[g][v] = fmaf(wt, ov[r][g][v], acc[g][v]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < kCombShortList; ++i) f |= st[i];
    if (scnt > kCombShortList) {  // a long list: a warp takes it below
        const int d = atomicAdd(&sm.ndef, 1);
        if (d < kCombMaxDeferred) sm.defk[d] = tid;
        else
            for (int p = 0; p < scnt; ++p) f |= a.status[sk + sp0 + p];
    }
    // segments beyond the first NT of the request (long requests with many
    // chunks): the same gathering, a thread per segment
    for (int it = tid + NT; U > 0 && it < nseg; it += NT) {
        const int k = kseg0 + it;
        const int u0 = ws_prefix[k], u1 = ws_prefix[k + 1];  // pfx now holds chunk rows
        if (u1 == u0) continue;
        const int p0 = pers_worker_of(u0, U, W), p1 = pers_worker_of(u1 - 1, U, W);
        for (int p = p0; p <= p1; ++p) f |= a.status[k + p];
    }
    __syncthreads();  // deferred list complete; the row tables are dead
    {
        const int ndef = min(sm.ndef, kCombMaxDeferred);
        for (int d = warp; d < ndef; d += NW) {
            const int t = sm.defk[d];  // the thread that found the list
            const int k = kseg0 + t;
            const int u0 = ws_prefix[k], u1 = ws_prefix[k + 1];
            const int p0 = pers_worker_of(u0, U, W), p1 = pers_worker_of(u1 - 1, U, W);
            for (int p = p0 + lane; p <= p1; p += 32) f |= a.status[k + p];
        }
    }
    if (f) atomicOr(&sm.flags, f);
#pragma unroll
    for (int g = 0; g < GS; ++g) {
        store_vec<VL>(&sm.u.red.acc[warp][g][lane * VL], acc[g]);
        if (lane == 0) {
            sm.u.red.wsum[warp][g] = S[g];
            sm.u.red.wmax[warp][g] = M[g];
        }
    }
    __syncthreads();
    const uint32_t flags = sm.flags;
    if (b == v0 && h == 0 && gi == 0 && tid == 0 && a.flags) a.flags[rb] = (uint8_t)flags;
    if (b == v0 && h == 0 && gi == 0 && tid == 0 && a.rflags) a.rflags[rb] = (uint8_t)flags;
    const int n = max(0, query_len(a, b, h));
    uint2 *out = reinterpret_cast<uint2 *>(a.out + ((long long)(b * Hkv + h) * G + g0) * D);
    if (flags != 0 || n == 0 || U == 0) {
        for (int i = tid; i < GS * D / 4; i += NT) out[i] = make_uint2(0u, 0u);
        return;
    }

    // ---- out = merged sum / merged weight ----
    for (int i = tid; i < GS * D / 4; i += NT) {
        const int g = i / (D / 4), d4 = i - g * (D / 4);
        float Mg = -INFINITY;
#pragma unroll
        for (int w2 = 0; w2 < NW; ++w2) Mg = fmaxf(Mg, sm.u.red.wmax[w2][g]);
        float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
        float ws = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < NW; ++w2) {
            const float mw = sm.u.red.wmax[w2][g];
            const float sc = mw == -INFINITY ? 0.f : pexp2(mw - Mg);
            const float4 v = *reinterpret_cast<const float4 *>(&sm.u.red.acc[w2][g][d4 * 4]);
            s4.x = fmaf(sc, v.x, s4.x);
            s4.y = fmaf(sc, v.y, s4.y);
            s4.z = fmaf(sc, v.z, s4.z);
            s4.w = fmaf(sc, v.w, s4.w);
            ws = fmaf(sc, sm.u.red.wsum[w2][g], ws);
        }
        const float inv = ws > 0.f ? 1.f / ws : 0.f;
        if (a.lse_fin && d4 == 0)
            a.lse_fin[(long long)(b * Hkv + h) * G + g0 + g] = ws > 0.f ? Mg + plog2(ws) : -INFINITY;
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

template <int G, int GS, int NW, int D>
cudaError_t launch_comb_d(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s) {
    const unsigned grid = (unsigned)(p.B * p.Hkv * (G / GS));
    return launch_pdl(decode_combine_pers_kernel<G, GS, NW, D>, dim3(grid), dim3(NW * 32), 0, s, a, p.Hkv,
                      p.nchunks, p.chunk_tokens, p.workers, (const int *)a.ws_prefix);
}

template <int G, int GS, int NW>
cudaError_t launch_comb(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s) {
    if (p.D == 64) return launch_comb_d<G, GS, NW, 64>(a, p, s);
    return p.D == 128 ? launch_comb_d<G, GS, NW, 128>(a, p, s) : cudaErrorInvalidValue;
}

template <int G>
cudaError_t launch_combine_g(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s) {
    const long long heads = (long long)p.B * p.Hkv;
    // One chunk per head and at most 16 workers' rows per head on average: 8
    // warps for all G query heads.
    if (p.nchunks == 1 && (long long)p.workers <= 16 * heads) return launch_comb<G, G, 8>(a, p, s);
    // Many rows per head: 16 warps (one CTA per SM), and the G query heads
    // split into as many groups as keep every CTA in one wave over the SMs.
    int hg = 1;
    while (hg < G && heads * hg * 2 <= p.pers_ctas) hg *= 2;
    if constexpr (G == 8) {
        if (hg == 8) return launch_comb<8, 1, 16>(a, p, s);
        if (hg == 4) return launch_comb<8, 2, 16>(a, p, s);
        if (hg == 2) return launch_comb<8, 4, 16>(a, p, s);
        return launch_comb<8, 8, 8>(a, p, s);  // 16 warps x 8 heads would not fit static shared memory
    } else if constexpr (G == 4) {
        if (hg == 4) return launch_comb<4, 1, 16>(a, p, s);
        if (hg == 2) return launch_comb<4, 2, 16>(a, p, s);
        return launch_comb<4, 4, 16>(a, p, s);
    } else if constexpr (G == 2) {
        if (hg == 2) return launch_comb<2, 1, 16>(a, p, s);
        return launch_comb<2, 2, 16>(a, p, s);
    } else {
        return launch_comb<1, 1, 16>(a, p, s);
    }
}

}  // namespace

namespace {
template <int D>
cudaError_t preload_combine_d() {
    cudaError_t e = cudaSuccess;
    auto one = [&](cudaError_t r) { if (e == cudaSuccess) e = r; };
    one(preload_kernel(decode_combine_pers_kernel<8, 8, 8, D>));
    one(preload_kernel(decode_combine_pers_kernel<8, 4, 16, D>));
    one(preload_kernel(decode_combine_pers_kernel<8, 2, 16, D>));
    one(preload_kernel(decode_combine_pers_kernel<8, 1, 16, D>));
    one(preload_kernel(decode_combine_pers_kernel<4, 4, 8, D>));
    one(preload_kernel(decode_combine_pers_kernel<4, 4, 16, D>));
    one(preload_kernel(decode_combine_pers_kernel<4, 2, 16, D>));
    one(preload_kernel(decode_combine_pers_kernel<4, 1, 16, D>));
    one(preload_kernel(decode_combine_pers_kernel<2, 2, 8, D>));
    one(preload_kernel(decode_combine_pers_kernel<2, 2, 16, D>));
    one(preload_kernel(decode_combine_pers_kernel<2, 1, 16, D>));
    one(preload_kernel(decode_combine_pers_kernel<1, 1, 8, D>));
    one(preload_kernel(decode_combine_pers_kernel<1, 1, 16, D>));
    return e;
}
}  // namespace

cudaError_t preload_combine_pers() {
    cudaError_t e = preload_combine_d<128>();
    if (e == cudaSuccess) e = preload_combine_d<64>();
    return e;
}

cudaError_t launch_combine_pers(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s) {
    switch (p.G) {
        case 1: return launch_combine_g<1>(a, p, s);
        case 2: return launch_combine_g<2>(a, p, s);
        case 4: return launch_combine_g<4>(a, p, s);
        case 8: return launch_combine_g<8>(a, p, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace pfkv
