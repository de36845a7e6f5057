// Decode attention instantiated for keys in Q40 and values in AFF8.
#include "decode_tc.cuh"

namespace kvq {
template cudaError_t launch_decode<F_Q40, F_AFF8>(const CacheView&, int, const DecodeArgs&, cudaStream_t);
}  // namespace kvq
