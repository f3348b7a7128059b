// Chunked tensor-core prefill (placeholder until the tcgen05 kernel lands).
#include "kda_common.cuh"
namespace kda {
bool prefill_tc_supported(const kda_prefill_args&) { return false; }
size_t prefill_tc_workspace_size(const kda_prefill_args&) { return 0; }
cudaError_t launch_prefill_tc(const kda_prefill_args&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace kda
