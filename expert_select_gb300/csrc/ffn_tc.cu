// Placeholder until the tcgen05 grouped-expert kernel lands.
#include "common.cuh"

namespace moe {
bool ffn_tc_supported(const moe_layer_desc &) { return false; }
cudaError_t launch_ffn_tc(const FfnArgs &, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace moe
