// Decode kernel instantiations for the native 16-bit cache (the A/B twin):
// head_dim 64/128, FP16/BF16 activations, and their host-side launch helpers.
#include "kvq_decode.cuh"

namespace kvq {

const DecodeOps kDecodeKv16 = DecodeLaunch<false, false, 1>::ops();

}  // namespace kvq
