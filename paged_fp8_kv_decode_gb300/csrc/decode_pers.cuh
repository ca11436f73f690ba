// decode_pers.cuh -- persistent, load-balanced split-KV decode attention for
// FP8 e4m3 or BF16 pools with head_dim 128 or 64 and query groups of up to 8
// heads (its partial rows are merged by combine_pers.cu).  Included by the
// translation units that instantiate it (decode_pers.cu, decode_pers_d64.cu).
//
// What is computed is the attention of decode.cu (single query per head over
// the tokens its kv head holds, read through the block table from the FP8
// pool); this kernel changes how the work is cut and fed, and moves both
// contractions onto the tensor cores:
//
// Segments and balanced ranges.  A segment is one (request b, kv head h,
// chunk c) — c is always 0 unless the caller fixes a split size.  Every CTA
// computes the same exclusive prefix sum of the segments' 16-token units
// (units of a request the validation kernel rejected are counted, then
// skipped).  With U units in all and W workers, worker w takes the units
// [ceil(wU/W), ceil((w+1)U/W)): equal shares, crossing segment boundaries, so
// no worker idles while another finishes a long sequence.  A worker writes one
// partial row (normalised output and log2-sum-exp per query head) for every
// segment it touches, at row index segment + worker, which is unique.
//
// Workers.  A worker is one warp with a shared-memory ring of granules (K and
// V slabs of two FP8 units or one BF16 unit; 24 KB per worker with 8 workers,
// 16 KB with 12).  Each slab arrives by one TMA tensor copy with the 128-byte
// swizzle (16-byte chunk c of 128-byte line L lands at chunk c ^ (L & 7)),
// which keeps the fragment loads below free of bank conflicts.  Per unit of
// 16 tokens the warp
//  * takes the scores S = K Q^T as D / 16 m16n8k16 MMAs (f16 operands, fp32
//    accumulation): the 16 tokens are the M rows, the G query heads the N
//    columns (zero-padded to 8), the D dims the reduction.  e4m3 bytes
//    become f16 A fragments with one conversion per register (every e4m3
//    value is exact in f16); Q sits in registers as f16 B fragments, scaled
//    by a power of two so that its largest element lies in [1, 2);
//  * runs the online softmax on the accumulator fragment (lane (g, t) holds
//    tokens g and g + 8 of heads 2t and 2t + 1), with a lazy rescale;
//  * accumulates O^T = V^T P^T as D / 8 MMAs: the D dims are the M rows (in
//    D / 16 tiles), tokens the reduction, heads the columns.  A byte permute
//    pairs two tokens of one dim, the conversion makes the A fragment, and
//    the probabilities, times the unit's V scale over a power-of-two
//    reference, become f16 B fragments through shuffles: each as a hi + lo
//    pair (two MMAs per tile), so that a weight carries 22 bits of its fp32
//    value rather than f16's 11.
// The dims of the score reduction are taken in a permuted order (lane t owns
// dims [t D / 4, (t + 1) D / 4) of both K and Q), which changes nothing in
// the sum.
#pragma once

#include <atomic>
#include <type_traits>

#include <cuda.h>
#include <cudaTypedefs.h>

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

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// four e4m3 codes -> two f16 pairs (bytes 0, 1 -> lo; bytes 2, 3 -> hi; the
// lower byte of each pair lands in the lower half)
__device__ __forceinline__ void e4m3x4_to_f16x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

// D += A B for one 16x8x16 tile: f16 A (row-major fragment), f16 B
// (column-major fragment), fp32 accumulators
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// the same with bf16 operands
__device__ __forceinline__ void mma_16816_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf162(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ uint4 lds128(const uint8_t *p) {
    return *reinterpret_cast<const uint4 *>(p);
}

__device__ __forceinline__ uint2 lds64(const uint8_t *p) {
    return *reinterpret_cast<const uint2 *>(p);
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Two fp32 values as a sum of two f16 pairs: hi = f16(x), lo = f16(x - hi).
// hi + lo is within 2^-22 |x| (plus 2^-25 absolute, the f16 subnormal step)
// of x, where hi alone is within 2^-11 |x|.
__device__ __forceinline__ void split_half2(float x, float y, uint32_t &hi, uint32_t &lo) {
    const __half2 h = __floats2half2_rn(x, y);
    const float2 f = __half22float2(h);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = pack_half2(x - f.x, y - f.y);
}

// The same with bf16 pairs: hi + lo within 2^-18 |x| (hi alone: 2^-9 |x|).
__device__ __forceinline__ void split_bf162(float x, float y, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
    const float2 f = __bfloat1622float2(h);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = pack_bf162(x - f.x, y - f.y);
}

// 2^e as fp32 for e in [-126, 127]
__device__ __forceinline__ float pow2i(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }

// smallest e with x < 2^e for finite x > 0 (-126 for zero and subnormals),
// clamped to 126
__device__ __forceinline__ int exp_above(float x) {
    const int eb = (int)((__float_as_uint(x) >> 23) & 0xffu);
    return min(126, max(eb, 0) - 126);
}

// TMA: one unit of a pool seen as [units][lines][128 B] (see pool_tensor_map)
// into shared memory, 128-byte swizzled, completing its bytes on `bar`
__device__ __forceinline__ void tma_unit(void *dst, const CUtensorMap *map, int unit, uint64_t *bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(0), "r"(unit), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

constexpr float kLazy = 8.0f;   // rescale only when the max grows by > 2^8
constexpr int kNoScale = -1000; // V-scale reference of a worker that has seen no unit yet

}  // namespace

// Kernel shape: worker warps per CTA, ring stages per worker, and units per
// granule.  A ring stage (granule) is 8 KB: two FP8 units or one BF16 unit at
// head_dim 128, four FP8 or two BF16 units at 64 (where per-token work weighs
// twice as much per byte, and a granule's fixed work is spread over more
// tokens).  Two worker counts are built, both with 192 KB of rings: 8 workers
// x 3 stages, and 12 workers x 2 stages, which hides more latency when every
// worker streams long runs (see pers_workers_for).
template <int WK, bool BF, int HD>
struct PersCfg {
    static_assert(WK == 8 || WK == 12, "8 or 12 workers per CTA");
    static_assert(HD == 128 || HD == 64, "head_dim 128 or 64");
    static constexpr int D = HD;
    static constexpr int ROWB = D * (BF ? 2 : 1);  // one token row of a slab
    static constexpr int UNITB = kPage * ROWB;     // FP8 2 KB / 1 KB, BF16 4 KB / 2 KB
    static constexpr int GU = (BF ? 1 : 2) * (128 / HD);
    static constexpr int STAGEB = 2 * GU * UNITB;  // K u0 .. K u(GU-1) | V u0 .. V u(GU-1)
    static constexpr int WORKERS = WK;
    static constexpr int STAGES = WK == 8 ? 3 : 2;
    static_assert(STAGEB == 8192, "8 KB granules");
    static constexpr int KS = D / 16;  // k-steps of the score MMAs (the dims)
    static constexpr int MT = D / 16;  // m-tiles of the value MMAs (the dims)
    static constexpr int QW = D / 32;  // 16-byte words of a lane's query dims
    static constexpr int NT = WORKERS * 32;
    static constexpr int MAXK = kPersMaxSegments;  // segments (prefix array in smem)
    static constexpr int MAXB = kPersMaxRequests;  // requests
    struct Smem {
        alignas(1024) uint8_t ring[WORKERS][STAGES][STAGEB];
        alignas(8) uint64_t full[WORKERS][STAGES];
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
template <int G, bool MASS, int WK, bool BF, int HD>
__global__ void __launch_bounds__(PersCfg<WK, BF, HD>::NT, 1)
    decode_split_pers_kernel(const __grid_constant__ CUtensorMap tmk,
                             const __grid_constant__ CUtensorMap tmv, DecodeArgs a, int Hkv, int B,
                             int nchunks, int chunk_tokens, int *ws_prefix) {
    using C = PersCfg<WK, BF, HD>;
    constexpr int ST = C::STAGES;
    static_assert(G == 1 || G == 2 || G == 4 || G == 8, "query groups of 1, 2, 4 or 8 heads");
    extern __shared__ uint8_t smem_raw[];
    typename C::Smem &sm = *reinterpret_cast<typename C::Smem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x;
    const int K = B * Hkv * nchunks;
    const int Breq = B / a.kq;  // B counts virtual requests (see DecodeArgs::kq)
    // Without a.early, wait for the previous kernels right away.  With it, the
    // part up to the second pdl_enter() below runs while the validation kernel
    // finishes: it reads only inputs of the call (lengths, block tables, tags,
    // queries), never the pool, the scales or the validation bits, and it
    // writes only shared memory.
    if (!a.early) pdl_enter();
    if (tid == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
    }
    {
        // pull the block-table rows into L2 while the prefix sums are built
        const int nrows = Breq * (a.bt_sh != 0 ? Hkv : 1);
        const int lines = (a.max_pages * 4 + 127) / 128 + 1;
        for (int i = blockIdx.x * C::NT + tid; i < nrows * lines; i += gridDim.x * C::NT) {
            const int r = i / lines, l = i - r * lines;
            const int b = a.bt_sh != 0 ? r / Hkv : r, h = a.bt_sh != 0 ? r - b * Hkv : 0;
            const long long e = min((long long)l * 32, (long long)a.max_pages - 1);
            const int32_t *ptr = a.block_tables + (long long)b * a.bt_sb + (long long)h * a.bt_sh + e;
            asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
        }
    }

    // ---------------- prologue: unit prefix sums ----------------
    // They do not depend on the validation bits: units of rejected requests
    // stay in the sums (see skip_rejected below).
    const int per = (K + C::NT - 1) / C::NT;
    const int k0 = min(K, tid * per), k1 = min(K, k0 + per);
    int local = 0, nbh = -1, n = 0;
    for (int k = k0; k < k1; ++k) {
        const int bh = k / nchunks, c = k - bh * nchunks;
        if (bh != nbh) {  // one length load per (request, head) of the range
            const int b = bh / Hkv, h = bh - b * Hkv;  // b: virtual request
            n = query_len(a, b, h);
            nbh = bh;
        }
        const int units = segment_units(n, c, chunk_tokens);
        int lastnv = 0;
        if (n >= 0) {
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
    const int W = min((int)gridDim.x * C::WORKERS, U);

    // ---------------- the worker: one warp ----------------
    const int warp = tid >> 5, lane = tid & 31;
    const int w = blockIdx.x * C::WORKERS + warp;
    const int x0 = w < W ? (int)(((long long)w * U + W - 1) / W) : U;
    const int x1 = w < W ? (int)(((long long)(w + 1) * U + W - 1) / W) : U;
    const bool idle = x0 >= x1;
    // fragment coordinates: lane (g, t) = (lane / 4, lane % 4)
    const int fg = lane >> 2, ft = lane & 3;
    uint8_t(*ring)[C::STAGEB] = sm.ring[warp];
    uint64_t *full = sm.full[warp];

    // granule cursor (GU units, never across a segment)
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
    int ngran = 0;        // granules of the worker's range, counted below
    uint64_t policy = 0;  // L2 policy of the copies, made below

    // unit metadata window: lane l holds unit base + l (cur) and base + 32 + l
    // (nxt): unit index (-1 bad, -2 absent), the two scales and the bad bits
    int base = x0;
    int cphys, nphys;
    float cks, cvs, nks, nvs;
    uint32_t cbad, nbad;
    // req: the unit's request (-1 for no unit), for skip_rejected()
    // A window entry: its table entry and page id (with the expected tag for
    // the fused check), loaded before any is used, then its status bits (one
    // more round for the pool's tag of the id when the check is fused).
    struct Entry {
        long long bi;
        int h, req, id;
        uint32_t want;
        bool live;
    };
    auto entry_load = [&](int x, Entry &e) {
        e.live = x < x1;
        e.bi = 0;
        e.h = 0;
        e.req = -1;
        e.id = 0;
        e.want = 0u;
        if (e.live) {
            const int k = seg_of(sm.prefix, K, x);
            const int bh = k / nchunks, c = k - bh * nchunks;
            const int b = bh / Hkv, h = bh - b * Hkv;
            const int page = c * (chunk_tokens / kPage) + (int)(x - sm.prefix[k]);
            e.bi = table_row(a, b, h) + page;
            e.h = h;
            e.req = b / a.kq;
            e.id = a.block_tables[e.bi];
            if (a.fuse_tags) e.want = a.expected_tags[e.bi];
        }
    };
    auto entry_tag = [&](const Entry &e) -> uint32_t {
        const bool in_pool = e.id >= 0 && e.id < a.num_pages;
        return e.live && a.fuse_tags && in_pool ? a.page_tags[(long long)e.id * Hkv + e.h] : 0u;
    };
    // the same bits as entry_bits, from the loaded values
    auto entry_finish = [&](const Entry &e, uint32_t tag, int &phys, uint32_t &bad, int &req) {
        phys = -2;
        bad = 0;
        req = -1;
        if (!e.live) return;
        if (e.id < 0 || e.id >= a.num_pages) bad = PFKV_FLAG_BAD_PAGE;
        else if (a.fuse_tags && tag != e.want) bad = PFKV_FLAG_TAG_MISMATCH;
        phys = bad ? -1 : e.id * Hkv + e.h;  // unit index
        req = e.req;
    };
    auto load_ids = [&](int bx, int &phys, uint32_t &bad, int &req) {
        Entry e;
        entry_load(bx + lane, e);
        entry_finish(e, entry_tag(e), phys, bad, req);
    };
    // units of a request the validation kernel rejected are absent
    auto skip_rejected = [&](int req, int &phys, uint32_t &bad) {
        if (req >= 0 && sm.rflag[req]) {
            phys = -2;
            bad = 0;
        }
    };
    auto load_scales = [&](int phys, float &ks, float &vs) {
        if constexpr (BF) {  // a BF16 pool has no scales
            ks = vs = 1.f;
        } else {
            const long long u = phys >= 0 ? phys : 0;
            ks = a.k_scale[u];
            vs = a.v_scale[u];
        }
    };
    int creq = -1, nreq = -1;
    // the first window's table entries (both halves): loaded here, used after
    // the wait below, so that their loads overlap those of the validation bits
    Entry first0, first1;
    if (!idle) {
        entry_load(base + lane, first0);
        entry_load(base + 32 + lane, first1);
    }
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
        const int n = min(C::GU, c.seg_end - c.x);
        int pu[C::GU];
        uint32_t bytes = 0;
#pragma unroll
        for (int u = 0; u < C::GU; ++u) {
            pu[u] = u < n ? unit_phys(c.x + u) : -2;
            bytes += pu[u] >= 0 ? 2 * C::UNITB : 0;
        }
        if (lane == 0) {
            if (bytes == 0) {
                mbar_arrive(&full[s]);
            } else {
                uint8_t *dst = ring[s];
                mbar_arrive_expect_tx(&full[s], bytes);
#pragma unroll
                for (int u = 0; u < C::GU; ++u) {
                    if (pu[u] >= 0) {
                        tma_unit(dst + u * C::UNITB, &tmk, pu[u], &full[s], policy);
                        tma_unit(dst + (C::GU + u) * C::UNITB, &tmv, pu[u], &full[s], policy);
                    }
                }
            }
        }
        return n;
    };

    // query: raw bf16 of head fg, dims [E ft, E ft + E) with E = D / 4,
    // fetched one segment ahead; f16 B fragments of the current segment
    // (qb0/qb1[ks]: dims E ft + 4 ks + {0, 1} / {2, 3}) and the factor that
    // undoes the power-of-two scaling and applies sm_scale * log2(e)
    uint4 qraw[C::QW];
    auto q_fetch = [&](int k) {
        if (fg < G) {
            const int bh = k / nchunks;
            const uint4 *src =
                reinterpret_cast<const uint4 *>(a.q + ((long long)bh * G + fg) * C::D + (C::D / 4) * ft);
#pragma unroll
            for (int j = 0; j < C::QW; ++j) qraw[j] = __ldg(src + j);
        } else {
#pragma unroll
            for (int j = 0; j < C::QW; ++j) qraw[j] = make_uint4(0u, 0u, 0u, 0u);
        }
    };
    uint32_t qb0[C::KS], qb1[C::KS];
    float qmul = 0.f;
    if (!idle) q_fetch(con.k);
    // what the first copies need but no load waits for: done while the
    // table-entry and query loads above are in flight
    if (!idle) {
        int x = x0;
        int k = seg_of(sm.prefix, K, x);
        while (x < x1) {
            const int e = min(sm.prefix[k + 1], x1);
            ngran += (e - x + C::GU - 1) / C::GU;
            x = e;
            ++k;
            while (k < K && sm.prefix[k + 1] == sm.prefix[k]) ++k;
        }
    }
    if (!idle && lane == 0) {
        for (int s = 0; s < ST; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    policy = l2_policy_evict_first();

    // ---------------- after the previous kernels: validation bits ----------------
    if (a.early) pdl_enter();
    if (blockIdx.x == 0) {
        for (int k = tid; k <= K; k += C::NT) ws_prefix[k] = sm.prefix[k];
    }
    for (int b = tid; b < Breq; b += C::NT) sm.rflag[b] = 0;
    __syncthreads();
    if (a.hflags) {  // [Breq][Hkv][htiles], read in parallel
        const int per_req = Hkv * a.htiles;
        for (int i = tid; i < Breq * per_req; i += C::NT)
            if (a.hflags[i]) sm.rflag[i / per_req] = 1;
    }
    __syncthreads();
    if (idle) return;  // no block-wide barrier follows
    {
        const uint32_t t0 = entry_tag(first0), t1 = entry_tag(first1);
        entry_finish(first0, t0, cphys, cbad, creq);
        entry_finish(first1, t1, nphys, nbad, nreq);
    }
    // no page is read before its request has passed validation
    skip_rejected(creq, cphys, cbad);
    skip_rejected(nreq, nphys, nbad);
    load_scales(cphys, cks, cvs);
    load_scales(nphys, nks, nvs);
    for (int j = 0; j < ST && j < ngran; ++j) cursor_next(iss, issue_at(iss, j));


    // Fragment offsets inside a swizzled slab.  Its 128-byte lines are
    // numbered L (a row of R bytes is line R / 128 of it, or R / 128 rows
    // share a line), and 16-byte chunk c of line L sits at chunk c ^ (L & 7).
    auto swz = [](int line, int chunk) { return line * 128 + ((chunk ^ (line & 7)) << 4); };
    constexpr int KC = C::ROWB / 64;  // 16-byte K chunks a lane reads per row (dims E ft ..)
    int offK[KC], offKh[KC];          // rows fg and fg + 8
    int offV[4] = {0, 0, 0, 0};       // V: the lane's four token rows
    int vtok[4] = {0, 0, 0, 0};       // ... which tokens they are
    uint32_t vsel0 = 0, vsel1 = 0;    // byte permutes that pair tokens (a, b) of one dim
    int obase = 0;                    // first dim of the lane's output tiles
    if constexpr (!BF && C::D == 128) {
        // K (A of S = K Q^T): row fg (+8: +1 KB), chunks 2 ft, 2 ft + 1 (dims 32 ft ..)
        offK[0] = swz(fg, 2 * ft);
        offK[1] = swz(fg, 2 * ft + 1);
        // V (A of O^T = V^T P^T): rows 2 ft, 2 ft + 1 (+8: +1 KB), chunk fg
        offV[0] = swz(2 * ft, fg);
        offV[1] = swz(2 * ft + 1, fg);
        vtok[0] = 2 * ft;
        vtok[1] = 2 * ft + 1;
        obase = 16 * fg;
    } else if constexpr (!BF) {
        // head_dim 64: a 64-byte row r is half r & 1 of line r / 2.  K: row
        // fg is chunk 4 (fg & 1) + ft of line fg / 2, row fg + 8 the same
        // chunk of line fg / 2 + 4 (another swizzle phase)
        offK[0] = swz(fg >> 1, 4 * (fg & 1) + ft);
        offKh[0] = swz((fg >> 1) + 4, 4 * (fg & 1) + ft);
        // V: 8 bytes (dims 16 c + 8 hh ..) of tokens 2 ft, 2 ft + 1 and the
        // same + 8; lanes with s = 1 read the pair in the other order, which
        // puts every 16-lane phase of an 8-byte load on distinct banks
        const int sv = fg & 1, c = (fg & 1) + 2 * (fg >> 2), hh = (fg >> 1) & 1;
        vtok[0] = 2 * ft + sv;
        vtok[1] = 2 * ft + 1 - sv;
        vtok[2] = vtok[0] + 8;
        vtok[3] = vtok[1] + 8;
#pragma unroll
        for (int r = 0; r < 4; ++r) offV[r] = swz(vtok[r] >> 1, 4 * (vtok[r] & 1) + c) + 8 * hh;
        vsel0 = sv ? 0x1504u : 0x5140u;
        vsel1 = sv ? 0x3726u : 0x7362u;
        obase = 16 * c + 8 * hh;
    } else if constexpr (C::D == 128) {
        // K: row fg (+8: +2 KB), dims 32 ft .. 32 ft + 31: half ft / 2, chunks
        // 4 (ft & 1) + j
        const int hk = ft >> 1;
#pragma unroll
        for (int j = 0; j < KC; ++j) offK[j] = swz(2 * fg + hk, 4 * (ft & 1) + j);
        // V: rows ft and ft + 4 (+8: +2 KB), in half fg / 4 the chunks
        // fg & 3 and (fg & 3) + 4, i.e. dims 64 h + 8 (fg & 3) + 0..7 and the
        // same + 32
        const int hv = fg >> 2, gg = fg & 3;
        offV[0] = swz(2 * ft + hv, gg);
        offV[1] = swz(2 * ft + hv, gg + 4);
        offV[2] = swz(2 * (ft + 4) + hv, gg);
        offV[3] = swz(2 * (ft + 4) + hv, gg + 4);
        obase = 64 * hv + 8 * gg;
    } else {
        // head_dim 64: a row is one line.  K: row fg (+8: +1 KB), chunks
        // 2 ft, 2 ft + 1 (dims 16 ft ..)
        offK[0] = swz(fg, 2 * ft);
        offK[1] = swz(fg, 2 * ft + 1);
        // V: chunk fg (dims 8 fg ..) of tokens ft, ft + 4 and the same + 8;
        // lanes with s = 1 read the pair in the other order, which puts the
        // eight lanes of every 16-byte load phase on distinct banks
        const int sv = fg & 1;
        vtok[0] = ft + 4 * sv;
        vtok[1] = ft + 4 - 4 * sv;
        vtok[2] = vtok[0] + 8;
        vtok[3] = vtok[1] + 8;
#pragma unroll
        for (int r = 0; r < 4; ++r) offV[r] = swz(vtok[r], fg);
        vsel0 = sv ? 0x1054u : 0x5410u;
        vsel1 = sv ? 0x3276u : 0x7632u;
        obase = 8 * fg;
    }
    if constexpr (BF || C::D == 128) {
#pragma unroll
        for (int j = 0; j < KC; ++j) offKh[j] = offK[j] + 8 * C::ROWB;
    }
    // shuffle sources of the probability fragment of head fg: FP8 pairs the
    // tokens (2 ft, 2 ft + 1) and (2 ft + 8, 2 ft + 9), BF16 pairs (ft, ft + 4)
    // and (ft + 8, ft + 12); and which of the source's two heads is fg
    const int src0 = (BF ? 4 : 8) * ft + (fg >> 1), src1 = src0 + (BF ? 16 : 4);
    const bool odd_head = (fg & 1) != 0;

    // online softmax state of heads 2 ft (A) and 2 ft + 1 (B); O^T fragments:
    // o[mt][0] = (dim 16 fg + 2 mt, head A), [1] = (same dim, head B),
    // [2] = (dim + 1, head A), [3] = (dim + 1, head B); O is kept in units of
    // 2^eO (the V-scale reference)
    float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
    float o[C::MT][4];
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    int eO = kNoScale;
    float vref = 0.f;  // 2^-eO

    uint32_t parity = 0, seg_status = 0;
    int s = 0;
    bool pending_scales = false, seg_start = true;
    for (int i = 0; i < ngran; ++i) {
        // metadata window upkeep
        if (pending_scales) {
            load_scales(nphys, nks, nvs);
            pending_scales = false;
        }
        if (con.x >= base + 32) {
            base += 32;
            cphys = nphys; cks = nks; cvs = nvs; cbad = nbad;
            int req;
            load_ids(base + 32, nphys, nbad, req);
            skip_rejected(req, nphys, nbad);
            pending_scales = true;
        }
        if (seg_start && BF) {
            // BF16: the query's bf16 pairs are the B fragments as they are
#pragma unroll
            for (int ks = 0; ks < C::KS; ++ks) {
                qb0[ks] = word_of(qraw[ks >> 1], 2 * (ks & 1));
                qb1[ks] = word_of(qraw[ks >> 1], 2 * (ks & 1) + 1);
            }
            qmul = a.q_scale;
            if (con.seg_end < x1) q_fetch(seg_of(sm.prefix, K, con.seg_end));
            seg_start = false;
        }
        if (seg_start) {
            // this segment's query fragments, then fetch the next segment's
            uint32_t amax = 0;
#pragma unroll
            for (int j = 0; j < C::QW; ++j) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint32_t wq = word_of(qraw[j], c);
                    amax = max(amax, max((wq << 16) & 0x7fff0000u, wq & 0x7fff0000u));
                }
            }
            asm volatile("redux.sync.max.u32 %0, %0, 0xffffffff;" : "+r"(amax));
            const int eq = min(126, max(-126, (int)(amax >> 23) - 127));
            const float down = pow2i(-eq);
            qmul = a.q_scale * pow2i(eq);
#pragma unroll
            for (int ks = 0; ks < C::KS; ++ks) {
                const float2 f0 = bf16x2_to_float2(word_of(qraw[ks >> 1], 2 * (ks & 1)));
                const float2 f1 = bf16x2_to_float2(word_of(qraw[ks >> 1], 2 * (ks & 1) + 1));
                qb0[ks] = pack_half2(f0.x * down, f0.y * down);
                qb1[ks] = pack_half2(f1.x * down, f1.y * down);
            }
            if (con.seg_end < x1) q_fetch(seg_of(sm.prefix, K, con.seg_end));
            seg_start = false;
        }
        const int n_units = min(C::GU, con.seg_end - con.x);
        UnitMeta um[C::GU];
        int nv[C::GU];
        const int seg_last = sm.prefix[con.k + 1] - 1;
        const int lnv = sm.last_nv[con.k];
        bool full_gran = n_units == C::GU;
#pragma unroll
        for (int u = 0; u < C::GU; ++u) {
            um[u] = UnitMeta{-2, 0.f, 0.f, 0u};
            if (u < n_units) um[u] = unit_meta(con.x + u);
            seg_status |= um[u].bad;
            nv[u] = um[u].phys >= 0 ? (con.x + u == seg_last ? lnv : kPage) : 0;
            full_gran = full_gran && nv[u] == kPage;
        }

        if (!mbar_wait_bounded(&full[s], parity)) seg_status |= kStatusTimeout;
        const uint8_t *stage = ring[s];

        // One granule.  FULL: every unit holds 16 live tokens, so no unit needs
        // a check and the units' MMA chains interleave.
        auto granule = [&](auto full_tag) {
            constexpr bool FULL = decltype(full_tag)::value;
            // ---- scores: S = K Q^T per unit; sc[u][j]: token fg (+8 for j >= 2),
            //      head 2 ft (+1 for odd j); -inf outside the unit's live rows ----
            float sc[C::GU][4];
            float c0[C::GU][4], c1[C::GU][4];
#pragma unroll
            for (int u = 0; u < C::GU; ++u) {
#pragma unroll
                for (int j = 0; j < 4; ++j) c0[u][j] = c1[u][j] = 0.f;
            }
#pragma unroll
            for (int u = 0; u < C::GU; ++u) {
                if ((FULL || nv[u] > 0) && !BF) {
                    const uint8_t *kb = stage + u * C::UNITB;
                    uint4 ra[KC], rb[KC];
#pragma unroll
                    for (int j = 0; j < KC; ++j) {
                        ra[j] = lds128(kb + offK[j]);
                        rb[j] = lds128(kb + offKh[j]);
                    }
#pragma unroll
                    for (int ks = 0; ks < C::KS; ++ks) {
                        const uint32_t wa = word_of(ra[ks >> 2], ks & 3);
                        const uint32_t wb = word_of(rb[ks >> 2], ks & 3);
                        uint32_t a0, a2, a1, a3;
                        e4m3x4_to_f16x2(wa, a0, a2);
                        e4m3x4_to_f16x2(wb, a1, a3);
                        if (ks & 1) mma_16816(c1[u], a0, a1, a2, a3, qb0[ks], qb1[ks]);
                        else mma_16816(c0[u], a0, a1, a2, a3, qb0[ks], qb1[ks]);
                    }
                }
                if ((FULL || nv[u] > 0) && BF) {
                    // BF16: the bf16 pairs of K are the A fragments as they are
                    const uint8_t *kb = stage + u * C::UNITB;
                    uint4 ra[KC], rb[KC];
#pragma unroll
                    for (int j = 0; j < KC; ++j) {
                        ra[j] = lds128(kb + offK[j]);
                        rb[j] = lds128(kb + offKh[j]);
                    }
#pragma unroll
                    for (int ks = 0; ks < C::KS; ++ks) {
                        const uint32_t a0 = word_of(ra[ks >> 1], 2 * (ks & 1));
                        const uint32_t a2 = word_of(ra[ks >> 1], 2 * (ks & 1) + 1);
                        const uint32_t a1 = word_of(rb[ks >> 1], 2 * (ks & 1));
                        const uint32_t a3 = word_of(rb[ks >> 1], 2 * (ks & 1) + 1);
                        if (ks & 1) mma_16816_bf16(c1[u], a0, a1, a2, a3, qb0[ks], qb1[ks]);
                        else mma_16816_bf16(c0[u], a0, a1, a2, a3, qb0[ks], qb1[ks]);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < C::GU; ++u) {
                const float f = qmul * um[u].ks;
                const bool lo_ok = FULL || fg < nv[u], hi_ok = FULL || fg + 8 < nv[u];
                sc[u][0] = lo_ok ? (c0[u][0] + c1[u][0]) * f : -INFINITY;
                sc[u][1] = lo_ok ? (c0[u][1] + c1[u][1]) * f : -INFINITY;
                sc[u][2] = hi_ok ? (c0[u][2] + c1[u][2]) * f : -INFINITY;
                sc[u][3] = hi_ok ? (c0[u][3] + c1[u][3]) * f : -INFINITY;
                if (MASS) {  // scores for the attention-mass pass
                    const int bh = con.k / nchunks, c = con.k - bh * nchunks;
                    const int tok0 = (c * (chunk_tokens / kPage) + (con.x + u - sm.prefix[con.k])) * kPage + fg;
                    float *dst = a.mscore + ((long long)bh * a.mlen + tok0) * G;
                    if (2 * ft < G) {
                        if (lo_ok) dst[2 * ft] = sc[u][0];
                        if (hi_ok) dst[8 * G + 2 * ft] = sc[u][2];
                    }
                    if (2 * ft + 1 < G) {
                        if (lo_ok) dst[2 * ft + 1] = sc[u][1];
                        if (hi_ok) dst[8 * G + 2 * ft + 1] = sc[u][3];
                    }
                }
            }

            // ---- online softmax: granule max per head over the token rows ----
            float mbA = fmaxf(sc[0][0], sc[0][2]), mbB = fmaxf(sc[0][1], sc[0][3]);
#pragma unroll
            for (int u = 1; u < C::GU; ++u) {
                mbA = fmaxf(mbA, fmaxf(sc[u][0], sc[u][2]));
                mbB = fmaxf(mbB, fmaxf(sc[u][1], sc[u][3]));
            }
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mbA = fmaxf(mbA, __shfl_xor_sync(0xffffffffu, mbA, off));
                mbB = fmaxf(mbB, __shfl_xor_sync(0xffffffffu, mbB, off));
            }
            const bool grow = mbA > mA + kLazy || mbB > mB + kLazy;
            // V-scale reference: 2^eO bounds every live unit's V scale seen so far
            int eneed = kNoScale;  // (a BF16 pool has no V scale: eO stays 0)
#pragma unroll
            for (int u = 0; u < C::GU; ++u)
                if (!BF && (FULL || nv[u] > 0)) eneed = max(eneed, exp_above(um[u].vs));
            const bool scale_up = eneed > eO;
            float fA = 1.f, fB = 1.f;
            if (scale_up) {
                const int d = eO - eneed;  // < 0
                const float r = (eO == kNoScale || d < -126) ? 0.f : pow2i(d);
                fA = fB = r;
                eO = eneed;
                vref = pow2i(-eO);
            }
            if (grow) {
                const float nA = fmaxf(mA, mbA), nB = fmaxf(mB, mbB);
                const float aA = mA == -INFINITY ? 0.f : pexp2(mA - nA);
                const float aB = mB == -INFINITY ? 0.f : pexp2(mB - nB);
                mA = nA;
                mB = nB;
                lA *= aA;
                lB *= aB;
                fA *= aA;
                fB *= aB;
            }
            if (grow || scale_up) {
#pragma unroll
                for (int mt = 0; mt < C::MT; ++mt) {
                    o[mt][0] *= fA;
                    o[mt][2] *= fA;
                    o[mt][1] *= fB;
                    o[mt][3] *= fB;
                }
            }

            // ---- probabilities -> B fragments of the V product; V product ----
#pragma unroll
            for (int u = 0; u < C::GU; ++u) {
                const bool lo_ok = FULL || fg < nv[u], hi_ok = FULL || fg + 8 < nv[u];
                const float pA0 = lo_ok ? pexp2(sc[u][0] - mA) : 0.f;
                const float pB0 = lo_ok ? pexp2(sc[u][1] - mB) : 0.f;
                const float pA1 = hi_ok ? pexp2(sc[u][2] - mA) : 0.f;
                const float pB1 = hi_ok ? pexp2(sc[u][3] - mB) : 0.f;
                lA += pA0 + pA1;
                lB += pB0 + pB1;
                if (!FULL && nv[u] == 0) continue;  // uniform: nothing of this unit is live
                const float vs = um[u].vs * vref;
                // X0: head A at tokens (fg, fg + 8); X1: head B.  Each weight
                // (times the unit's V scale over the reference; BF16: no V
                // scale) enters the MMA as a hi + lo pair of 16-bit values
                // (L0, L1: the lo parts): a single 16-bit weight would err by
                // 2^-11 (bf16: 2^-9) of w |v|, which near-cancelling large
                // values turn into errors above the output's tolerance.
                uint32_t X0, X1, L0, L1;
                if constexpr (BF) {
                    split_bf162(pA0, pA1, X0, L0);
                    split_bf162(pB0, pB1, X1, L1);
                } else {
                    split_half2(pA0 * vs, pA1 * vs, X0, L0);
                    split_half2(pB0 * vs, pB1 * vs, X1, L1);
                }
                // head fg: Y0 = tokens (a, a + 8), Y1 = (b, b + 8) with (a, b) =
                // (2 ft, 2 ft + 1) for FP8 and (ft, ft + 4) for BF16 (both
                // heads of the source lane travel; this lane keeps its own)
                const uint32_t s00 = __shfl_sync(0xffffffffu, X0, src0), s01 = __shfl_sync(0xffffffffu, X1, src0);
                const uint32_t s10 = __shfl_sync(0xffffffffu, X0, src1), s11 = __shfl_sync(0xffffffffu, X1, src1);
                const uint32_t l00 = __shfl_sync(0xffffffffu, L0, src0), l01 = __shfl_sync(0xffffffffu, L1, src0);
                const uint32_t l10 = __shfl_sync(0xffffffffu, L0, src1), l11 = __shfl_sync(0xffffffffu, L1, src1);
                const uint32_t Y0 = odd_head ? s01 : s00, Y1 = odd_head ? s11 : s10;
                const uint32_t Z0 = odd_head ? l01 : l00, Z1 = odd_head ? l11 : l10;
                const uint32_t pb0 = __byte_perm(Y0, Y1, 0x5410);  // tokens a, b
                const uint32_t pb1 = __byte_perm(Y0, Y1, 0x7632);  // tokens a + 8, b + 8
                const uint32_t pl0 = __byte_perm(Z0, Z1, 0x5410);
                const uint32_t pl1 = __byte_perm(Z0, Z1, 0x7632);

                const uint8_t *vb = stage + (C::GU + u) * C::UNITB;
                if constexpr (C::D == 64) {
                    // the lane's four token rows (a, b, a + 8, b + 8 in the
                    // order vtok gives); rows past the live tokens may hold
                    // stale bytes (even NaN codes): zero them so that 0 x row
                    // stays 0
                    constexpr int NWD = BF ? 4 : 2;  // 32-bit words a lane reads per row
                    uint32_t rw[4][NWD];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        if constexpr (BF) {
                            const uint4 v = lds128(vb + offV[r]);
                            rw[r][0] = v.x, rw[r][1] = v.y, rw[r][2] = v.z, rw[r][3] = v.w;
                        } else {
                            const uint2 v = lds64(vb + offV[r]);
                            rw[r][0] = v.x, rw[r][1] = v.y;
                        }
                        if (!FULL && vtok[r] >= nv[u]) {
#pragma unroll
                            for (int q = 0; q < NWD; ++q) rw[r][q] = 0u;
                        }
                    }
#pragma unroll
                    for (int q = 0; q < NWD; ++q) {
                        uint32_t a0, a1, a2, a3;
                        if constexpr (BF) {
                            // dims (2q, 2q + 1) of the chunk -> tile q
                            a0 = __byte_perm(rw[0][q], rw[1][q], vsel0);
                            a1 = __byte_perm(rw[0][q], rw[1][q], vsel1);
                            a2 = __byte_perm(rw[2][q], rw[3][q], vsel0);
                            a3 = __byte_perm(rw[2][q], rw[3][q], vsel1);
                            mma_16816_bf16(o[q], a0, a1, a2, a3, pb0, pb1);
                            mma_16816_bf16(o[q], a0, a1, a2, a3, pl0, pl1);
                        } else {
                            // dims 4q, 4q + 1 -> tile 2q; 4q + 2, 4q + 3 -> tile 2q + 1
                            e4m3x4_to_f16x2(__byte_perm(rw[0][q], rw[1][q], vsel0), a0, a1);
                            e4m3x4_to_f16x2(__byte_perm(rw[2][q], rw[3][q], vsel0), a2, a3);
                            mma_16816(o[2 * q], a0, a1, a2, a3, pb0, pb1);
                            mma_16816(o[2 * q], a0, a1, a2, a3, pl0, pl1);
                            e4m3x4_to_f16x2(__byte_perm(rw[0][q], rw[1][q], vsel1), a0, a1);
                            e4m3x4_to_f16x2(__byte_perm(rw[2][q], rw[3][q], vsel1), a2, a3);
                            mma_16816(o[2 * q + 1], a0, a1, a2, a3, pb0, pb1);
                            mma_16816(o[2 * q + 1], a0, a1, a2, a3, pl0, pl1);
                        }
                    }
                    continue;
                }
                if constexpr (BF) {
                    // rows ft, ft + 4, ft + 8, ft + 12; chunks A and B of each
                    uint4 ra[4], rb[4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        ra[r] = lds128(vb + (r & 2 ? 8 * C::ROWB : 0) + offV[(r & 1) * 2]);
                        rb[r] = lds128(vb + (r & 2 ? 8 * C::ROWB : 0) + offV[(r & 1) * 2 + 1]);
                    }
                    if (!FULL && nv[u] < kPage) {
                        // rows past the live tokens may hold stale bytes (even
                        // NaN codes): zero them so that 0 x row stays 0
                        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                        for (int r = 0; r < 4; ++r)
                            if (ft + 4 * r >= nv[u]) ra[r] = rb[r] = z;
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        // dims (2q, 2q + 1) of chunk A -> tile q; of chunk B -> tile 4 + q
                        uint32_t w0 = word_of(ra[0], q), w1 = word_of(ra[1], q);
                        uint32_t w2 = word_of(ra[2], q), w3 = word_of(ra[3], q);
                        uint32_t a0 = __byte_perm(w0, w1, 0x5410), a1 = __byte_perm(w0, w1, 0x7632);
                        uint32_t a2 = __byte_perm(w2, w3, 0x5410), a3 = __byte_perm(w2, w3, 0x7632);
                        mma_16816_bf16(o[q], a0, a1, a2, a3, pb0, pb1);
                        mma_16816_bf16(o[q], a0, a1, a2, a3, pl0, pl1);
                        w0 = word_of(rb[0], q), w1 = word_of(rb[1], q);
                        w2 = word_of(rb[2], q), w3 = word_of(rb[3], q);
                        a0 = __byte_perm(w0, w1, 0x5410), a1 = __byte_perm(w0, w1, 0x7632);
                        a2 = __byte_perm(w2, w3, 0x5410), a3 = __byte_perm(w2, w3, 0x7632);
                        mma_16816_bf16(o[4 + q], a0, a1, a2, a3, pb0, pb1);
                        mma_16816_bf16(o[4 + q], a0, a1, a2, a3, pl0, pl1);
                    }
                    continue;
                }
                uint4 r0 = lds128(vb + offV[0]), r1 = lds128(vb + offV[1]);
                uint4 r2 = lds128(vb + 8 * C::ROWB + offV[0]), r3 = lds128(vb + 8 * C::ROWB + offV[1]);
                if (!FULL && nv[u] < kPage) {
                    // rows past the live tokens may hold stale bytes (even NaN
                    // codes): zero them so that 0 x row stays 0
                    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                    if (2 * ft >= nv[u]) r0 = z;
                    if (2 * ft + 1 >= nv[u]) r1 = z;
                    if (2 * ft + 8 >= nv[u]) r2 = z;
                    if (2 * ft + 9 >= nv[u]) r3 = z;
                }
#pragma unroll
                for (int wd = 0; wd < 4; ++wd) {
                    const uint32_t w0 = word_of(r0, wd), w1 = word_of(r1, wd);
                    const uint32_t w2 = word_of(r2, wd), w3 = word_of(r3, wd);
                    uint32_t a0, a1, a2, a3;
                    e4m3x4_to_f16x2(__byte_perm(w0, w1, 0x5140), a0, a1);  // dims 4wd, 4wd+1
                    e4m3x4_to_f16x2(__byte_perm(w2, w3, 0x5140), a2, a3);
                    mma_16816(o[2 * wd], a0, a1, a2, a3, pb0, pb1);
                    mma_16816(o[2 * wd], a0, a1, a2, a3, pl0, pl1);
                    e4m3x4_to_f16x2(__byte_perm(w0, w1, 0x7362), a0, a1);  // dims 4wd+2, 4wd+3
                    e4m3x4_to_f16x2(__byte_perm(w2, w3, 0x7362), a2, a3);
                    mma_16816(o[2 * wd + 1], a0, a1, a2, a3, pb0, pb1);
                    mma_16816(o[2 * wd + 1], a0, a1, a2, a3, pl0, pl1);
                }
            }
        };
        if (full_gran) granule(std::true_type{});
        else granule(std::false_type{});

        const bool seg_end = con.x + n_units >= con.seg_end;
        if (seg_end) {
            // finish the segment: sum l over the token rows, normalise, write
            float tA = lA, tB = lB;
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                tA += __shfl_xor_sync(0xffffffffu, tA, off);
                tB += __shfl_xor_sync(0xffffffffu, tB, off);
            }
            const float up = BF ? 1.f : (eO == kNoScale ? 0.f : pow2i(eO));
            const float iA = tA > 0.f ? up / tA : 0.f, iB = tB > 0.f ? up / tB : 0.f;
            const long long row = con.k + w;
            // tile mt holds dims (d, d + 1) in components (0, 2) for head A and
            // (1, 3) for head B, with d = obase + 2 mt (BF16 head_dim 128: plus
            // 24 for mt >= 4)
            auto store_head = [&](int head, int c0, int c1, float inv) {
                float *orow = a.o + (row * G + head) * C::D;
                float4 *dst = reinterpret_cast<float4 *>(orow + obase);
#pragma unroll
                for (int e = 0; e < C::MT / 2; ++e) {
                    const float4 v = make_float4(o[2 * e][c0] * inv, o[2 * e][c1] * inv,
                                                 o[2 * e + 1][c0] * inv, o[2 * e + 1][c1] * inv);
                    if (BF && C::D == 128 && e >= 2) dst[e + 6] = v;  // dims + 32
                    else dst[e] = v;
                }
            };
            if (2 * ft < G) {
                store_head(2 * ft, 0, 2, iA);
                if (fg == 0) a.lse[row * G + 2 * ft] = tA > 0.f ? mA + plog2(tA) : -INFINITY;
            }
            if (2 * ft + 1 < G) {
                store_head(2 * ft + 1, 1, 3, iB);
                if (fg == 0) a.lse[row * G + 2 * ft + 1] = tB > 0.f ? mB + plog2(tB) : -INFINITY;
            }
            if (lane == 0) a.status[row] = seg_status;
            seg_status = 0;
            mA = mB = -INFINITY;
            lA = lB = 0.f;
#pragma unroll
            for (int mt = 0; mt < C::MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
            eO = kNoScale;
            vref = 0.f;
            seg_start = true;
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

// --------------------------------------------------------------------------
// host side
// --------------------------------------------------------------------------
namespace {

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library)
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// A pool as a tensor of 128-byte lines read in one box per unit, with the
// 128-byte swizzle: [units][unit_bytes / 128][128 B], the unit index
// outermost (32-bit, like the unit indices).  An FP8 row of head_dim 128 is
// one line and of 64 half a line; a BF16 row of head_dim 128 is two lines
// (the swizzle spans at most 128 bytes) and of 64 one.
cudaError_t pool_tensor_map(CUtensorMap *map, const void *pages, long long units, int unit_bytes) {
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {128, (cuuint64_t)(unit_bytes / 128), (cuuint64_t)units};
    const cuuint64_t strides[2] = {128, (cuuint64_t)unit_bytes};
    const cuuint32_t box[3] = {128, (cuuint32_t)(unit_bytes / 128), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(pages), dims, strides,
                           box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int WK, bool BF, int HD>
constexpr size_t pers_smem_bytes() {
    return sizeof(typename PersCfg<WK, BF, HD>::Smem) + 1024;
}

// The dynamic shared-memory opt-in of one instantiation, set once per device.
template <int G, bool MASS, int WK, bool BF, int HD>
cudaError_t configure_pers() {
    static std::atomic<unsigned long long> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(decode_split_pers_kernel<G, MASS, WK, BF, HD>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)pers_smem_bytes<WK, BF, HD>());
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    return cudaSuccess;
}

template <int G, bool MASS, int WK, bool BF, int HD>
cudaError_t launch_pers_gm(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s) {
    using C = PersCfg<WK, BF, HD>;
    const size_t smem = pers_smem_bytes<WK, BF, HD>();
    cudaError_t e = configure_pers<G, MASS, WK, BF, HD>();
    if (e != cudaSuccess) return e;
    const long long units = (long long)a.num_pages * p.Hkv;
    alignas(64) CUtensorMap tmk, tmv;
    if ((e = pool_tensor_map(&tmk, a.k_pages, units, C::UNITB)) != cudaSuccess) return e;
    if ((e = pool_tensor_map(&tmv, a.v_pages, units, C::UNITB)) != cudaSuccess) return e;
    return launch_pdl(decode_split_pers_kernel<G, MASS, WK, BF, HD>, dim3(p.pers_ctas), dim3(C::NT), smem,
                      s, tmk, tmv, a, p.Hkv, p.B, p.nchunks, p.chunk_tokens, a.ws_prefix);
}

template <int G, int WK, bool BF, int HD>
cudaError_t launch_pers_gw(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s) {
    return a.mscore ? launch_pers_gm<G, true, WK, BF, HD>(a, p, s)
                    : launch_pers_gm<G, false, WK, BF, HD>(a, p, s);
}

template <int G, bool BF, int HD>
cudaError_t launch_pers_gb(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s) {
    switch (p.pers_ctas > 0 ? p.workers / p.pers_ctas : 0) {
        case 8: return launch_pers_gw<G, 8, BF, HD>(a, p, s);
        case 12: return launch_pers_gw<G, 12, BF, HD>(a, p, s);
    }
    return cudaErrorInvalidValue;
}

template <int G, int HD>
cudaError_t launch_pers_g(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s) {
    return p.dtype == PFKV_KV_BF16 ? launch_pers_gb<G, true, HD>(a, p, s) : launch_pers_gb<G, false, HD>(a, p, s);
}

template <int G, int HD>
cudaError_t preload_pers_g() {
    cudaError_t e = cudaSuccess;
    auto one = [&](cudaError_t r) { if (e == cudaSuccess) e = r; };
    one(configure_pers<G, false, 8, false, HD>());
    one(configure_pers<G, true, 8, false, HD>());
    one(configure_pers<G, false, 12, false, HD>());
    one(configure_pers<G, true, 12, false, HD>());
    one(configure_pers<G, false, 8, true, HD>());
    one(configure_pers<G, true, 8, true, HD>());
    one(configure_pers<G, false, 12, true, HD>());
    one(configure_pers<G, true, 12, true, HD>());
    return e;
}

// Every instantiation of one head_dim: shared-memory opt-ins set, modules
// loaded.
template <int HD>
cudaError_t preload_pers_hd() {
    cudaError_t e = preload_pers_g<1, HD>();
    if (e == cudaSuccess) e = preload_pers_g<2, HD>();
    if (e == cudaSuccess) e = preload_pers_g<4, HD>();
    if (e == cudaSuccess) e = preload_pers_g<8, HD>();
    return e;
}

template <int HD>
cudaError_t launch_pers_hd(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s) {
    switch (p.G) {
        case 1: return launch_pers_g<1, HD>(a, p, s);
        case 2: return launch_pers_g<2, HD>(a, p, s);
        case 4: return launch_pers_g<4, HD>(a, p, s);
        case 8: return launch_pers_g<8, HD>(a, p, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

}  // namespace pfkv
