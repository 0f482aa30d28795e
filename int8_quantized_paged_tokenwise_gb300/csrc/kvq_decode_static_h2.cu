// Decode kernel instantiations for the INT8 cache with static scales, two KV heads per warp step:
// head_dim 64/128, FP16/BF16 activations, and their host-side launch helpers.
#include "kvq_decode.cuh"

namespace kvq {

const DecodeOps kDecodeStaticH2 = DecodeLaunch<true, true, 2>::ops();

}  // namespace kvq
