// mass.cu -- the attention-mass pass: per token of every unflagged (request,
// kv head), the summed softmax weight of the group's query heads, added to
// the caller's running totals.  An eviction policy keeps such totals and
// evicts the entries with the lowest ("Workers AI targets the inference
// bottleneck", section "KV cache compression goes open source", 3rd
// paragraph).  It runs after the combine: the split kernels left each live
// token's final scores (log2 units) in the workspace and the combine each
// head's log2-sum-exp over all its tokens, so weight = 2^(score - lse).
#include "pfkv_internal.cuh"

namespace pfkv {

namespace {

constexpr int kMassThreads = 256;

template <int G>
__global__ void __launch_bounds__(kMassThreads) attn_mass_kernel(DecodeArgs a, int Hkv) {
    pdl_enter();
    const int bh = blockIdx.x;
    const int b = bh / Hkv, h = bh - b * Hkv;
    const int j = blockIdx.y * kMassThreads + threadIdx.x;
    if (a.rflags[b]) return;  // aborted request: no mass
    // lengths of unflagged requests are within [0, max_seq_len]
    const int n = a.seq_lens[(long long)b * a.len_sb + (long long)h * a.len_sh];
    if (j >= n) return;
    const float *sc = a.mscore + ((long long)bh * a.mlen + j) * G;
    const float *lf = a.lse_fin + (long long)bh * G;  // heads h*G .. h*G + G - 1
    float sum = 0.f;
#pragma unroll
    for (int g = 0; g < G; ++g) sum += exp2f(sc[g] - lf[g]);
    float *dst = a.mass + (long long)b * a.mass_sb + (long long)h * a.mass_sh + j;
    *dst += sum;
}

}  // namespace

cudaError_t launch_mass(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s) {
    if (a.mlen <= 0) return cudaSuccess;
    const dim3 grid((unsigned)(p.B * p.Hkv), (unsigned)((a.mlen + kMassThreads - 1) / kMassThreads));
    switch (p.G) {
        case 1: return launch_pdl(attn_mass_kernel<1>, grid, dim3(kMassThreads), 0, s, a, p.Hkv);
        case 2: return launch_pdl(attn_mass_kernel<2>, grid, dim3(kMassThreads), 0, s, a, p.Hkv);
        case 4: return launch_pdl(attn_mass_kernel<4>, grid, dim3(kMassThreads), 0, s, a, p.Hkv);
        case 8: return launch_pdl(attn_mass_kernel<8>, grid, dim3(kMassThreads), 0, s, a, p.Hkv);
    }
    return cudaErrorInvalidValue;
}

cudaError_t preload_mass() {
    cudaError_t e = preload_kernel(attn_mass_kernel<1>);
    if (e == cudaSuccess) e = preload_kernel(attn_mass_kernel<2>);
    if (e == cudaSuccess) e = preload_kernel(attn_mass_kernel<4>);
    if (e == cudaSuccess) e = preload_kernel(attn_mass_kernel<8>);
    return e;
}

}  // namespace pfkv
