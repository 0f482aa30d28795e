// Decode kernel instantiations for the INT8 cache with per-token scale planes,
// one KV head and two consecutive pages per warp step: head_dim 64/128,
// FP16/BF16 activations, and their host-side launch helpers.
#include "kvq_decode.cuh"

namespace kvq {

const DecodeOps kDecodeInt8T2 = DecodeLaunch<true, false, 1, false, 2>::ops();

}  // namespace kvq
