// Decode kernel instantiations for the INT8 cache with static (per-tensor, binary32) scales:
// head_dim 64/128, FP16/BF16 activations, and their host-side launch helpers.
#include "kvq_decode.cuh"

namespace kvq {

const DecodeOps kDecodeStaticH1 = DecodeLaunch<true, true, 1>::ops();

}  // namespace kvq
