// decode_mma.cu -- tensor-core decode attention (placeholder until written).
#include "kvarn_internal.cuh"

namespace kvarn {
bool decode_mma_supported(int) { return false; }
cudaError_t launch_decode_mma(const DecodeArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace kvarn
