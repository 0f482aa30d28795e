// Decode kernel instantiations for the INT8 cache with per-token scale planes:
// head_dim 64/128, FP16/BF16 activations, and their host-side launch helpers.
#include "kvq_decode.cuh"

namespace kvq {

const DecodeOps kDecodeInt8H1 = DecodeLaunch<true, false, 1>::ops();

}  // namespace kvq
