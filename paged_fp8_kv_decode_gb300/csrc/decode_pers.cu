// decode_pers.cu -- host entry points of the persistent split-KV kernel
// (decode_pers.cuh): head_dim 128 is built here, head_dim 64 in
// decode_pers_d64.cu, so that the two sets of instantiations compile in
// parallel.
#include "decode_pers.cuh"

namespace pfkv {

// 12 workers when each SM has more than 8 x 192 units to stream (by the
// host-known bound: every head at max_seq_len); 8 otherwise.  Measured on the
// GB300: 12 x 2 stages was 6% faster on 128K-512K contexts and 4% faster on a
// 64 x 32K batch, but 4% slower on a batch of 32 lengths up to 8K, where the
// per-worker startup and the partial rows weigh more.
int pers_workers_for(long long units_bound, int num_sms) {
    return units_bound > (long long)num_sms * 8 * 192 ? 12 : 8;
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
