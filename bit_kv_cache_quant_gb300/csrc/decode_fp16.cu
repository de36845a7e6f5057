// Decode attention instantiated for keys in FP16 and values in FP16.
#include "decode_tc.cuh"

namespace kvq {
template cudaError_t launch_decode<F_FP16, F_FP16>(const CacheView&, int, const DecodeArgs&, cudaStream_t);
}  // namespace kvq
