// Decode attention instantiated for keys in KIVI4 and values in AFF4.
#include "decode_tc.cuh"

namespace kvq {
template cudaError_t launch_decode<F_KIVI4, F_AFF4>(const CacheView&, int, const DecodeArgs&, cudaStream_t);
}  // namespace kvq
