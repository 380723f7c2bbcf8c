// Tensor-core paged attention (bf16): placeholder until the kernel lands.
#include "sv_internal.cuh"

namespace sv {
bool attn_tc_supported(const KV &, int, int) { return false; }
cudaError_t launch_attn_tc(const AttnArgs &, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace sv
