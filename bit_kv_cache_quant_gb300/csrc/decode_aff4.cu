// Decode attention instantiated for keys in AFF4 and values in AFF4.
#include "decode_tc.cuh"

namespace kvq {
template cudaError_t launch_decode<F_AFF4, F_AFF4>(const CacheView&, int, const DecodeArgs&, cudaStream_t);
}  // namespace kvq
