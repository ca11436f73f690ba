// decode_pers.cu -- host entry points of the persistent split-KV kernel
// (decode_pers.cuh): head_dim 128 is built here, head_dim 64 in
// decode_pers_d64.cu, so that the two sets of instantiations compile in
// parallel.
#include "decode_pers.cuh"

namespace pfkv {

// 12 workers when each SM has more than 8 x 64 units to stream (by the
// host-known bound: every head at max_seq_len); 8 otherwise.  Measured on the
// GB300: 12 workers (2 stages each) beat 8 (3 stages) on long contexts and
// large sweeps, by 1 us per step on the Llama-shaped layer (B=32, bound 131K
// units) in back-to-back steps, and by 4 us on the B=8 BF16 sweep; with fewer
// units per worker (the B=1 sweep: 16K units) the per-worker startup and the
// partial rows weigh more and 8 workers were 1.5-2 us faster.
int pers_workers_for(long long units_bound, int num_sms) {
    return units_bound > (long long)num_sms * 8 * 64 ? 12 : 8;
}

bool pers_supported(const DecodePlan &p) {
    return (p.dtype == PFKV_KV_FP8_E4M3 || p.dtype == PFKV_KV_BF16) && (p.D == 128 || p.D == 64) &&
           p.G <= 8;
}

cudaError_t preload_split_pers() {
    cudaError_t e = preload_pers_hd<128>();
    if (e == cudaSuccess) e = preload_split_pers_d64();
    return e;
}

cudaError_t launch_split_pers(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s) {
    if (p.D == 64) return launch_split_pers_d64(a, p, s);
    return p.D == 128 ? launch_pers_hd<128>(a, p, s) : cudaErrorInvalidValue;
}

}  // namespace pfkv
