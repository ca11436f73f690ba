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

}  // namespace

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
constexpr int kCombMaxChunks = kPersMaxSegments;  // segments per (b, h) <= all segments

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
    // rows of the request's segments: a thread
    // per segment; a segment with many rows (few long segments, many workers
    // each) is deferred to a warp whose lanes take its rows.  The deferred
    // list borrows the row tables' space, which phase 2 fills later.
    if (U > 0) {
        for (int it = tid; it < a.kq * Hkv * nchunks; it += NT) {
            const int k = v0 * Hkv * nchunks + it;
            const int u0 = ws_prefix[k], u1 = ws_prefix[k + 1];
            if (u1 == u0) continue;
            const int p0 = pers_worker_of(u0, U, W), p1 = pers_worker_of(u1 - 1, U, W);
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
        const int p0 = pers_worker_of(ws_prefix[k], U, W), p1 = pers_worker_of(ws_prefix[k + 1] - 1, U, W);
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
            const int p0 = pers_worker_of(u0, U, W), p1 = pers_worker_of(u1 - 1, U, W);
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

template <int G>
cudaError_t launch_combine_g(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s) {
    const int W = p.pers_ctas * kPersWorkers;
    return launch_pdl(decode_combine_pers_kernel<G>, dim3((unsigned)(p.B * p.Hkv)), dim3(kCombThreads), 0, s, a,
                      p.Hkv, p.nchunks, W, (const int *)a.ws_prefix);
}

}  // namespace

cudaError_t launch_combine_pers(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s) {
    switch (p.G) {
        case 1: return launch_combine_g<1>(a, p, s);
        case 2: return launch_combine_g<2>(a, p, s);
        case 4: return launch_combine_g<4>(a, p, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace pfkv
