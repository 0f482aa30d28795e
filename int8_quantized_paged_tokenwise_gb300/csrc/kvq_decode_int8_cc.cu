// Decode kernel instantiations for the INT8 cache with per-token scale planes
// computed on the CUDA cores (FFMA dot products instead of tensor-core MMAs):
// the A/B counterpart of kvq_decode_int8.cu, head_dim 64/128, FP16/BF16
// activations, and their host-side launch helpers.
#include "kvq_decode.cuh"

namespace kvq {

const DecodeOps kDecodeInt8Cc = DecodeLaunch<true, false, 1, true>::ops();

}  // namespace kvq
