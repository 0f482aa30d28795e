// Decode kernel instantiations for the INT8 cache with per-token scale planes, two KV heads per warp step:
// head_dim 64/128, FP16/BF16 activations, and their host-side launch helpers.
#include "kvq_decode.cuh"

namespace kvq {

const DecodeOps kDecodeInt8H2 = DecodeLaunch<true, false, 2>::ops();

}  // namespace kvq
