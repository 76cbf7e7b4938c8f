// Chunked tensor-core prefill (placeholder until the tcgen05 kernel lands).
#include "kda_common.cuh"

namespace kda {
bool chunked_kernel_built() { return false; }
cudaError_t launch_chunked(const ChunkedArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace kda
