// decode_pers_d64.cu -- the persistent split-KV kernel (decode_pers.cuh) for
// head_dim 64, in a translation unit of its own so that it compiles in
// parallel with head_dim 128 (decode_pers.cu).
#include "decode_pers.cuh"

namespace pfkv {

cudaError_t preload_split_pers_d64() { return preload_pers_hd<64>(); }

cudaError_t launch_split_pers_d64(const DecodeArgs &a, const DecodePlan &p, cudaStream_t s) {
    return launch_pers_hd<64>(a, p, s);
}

}  // namespace pfkv
