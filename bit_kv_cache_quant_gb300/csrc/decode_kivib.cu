// Decode attention instantiated for KIVI residual-buffer keys (per-channel scales
// per closed block, full-precision tail) with affine per-token values.
#include "decode_tc.cuh"

namespace kvq {
template cudaError_t launch_decode<F_KIVIB8, F_AFF8>(const CacheView&, int, const DecodeArgs&, cudaStream_t);
template cudaError_t launch_decode<F_KIVIB4, F_AFF4>(const CacheView&, int, const DecodeArgs&, cudaStream_t);
}  // namespace kvq
