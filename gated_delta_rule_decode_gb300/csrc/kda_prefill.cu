// Chunked prefill (placeholder until the chunked kernels land).
#include "kda.h"
#include "kda_internal.h"

namespace kda {

size_t prefill_workspace_bytes(int, int, int, int32_t, int64_t) { return 0; }

cudaError_t launch_prefill(const PrefillParams &, int, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace kda
