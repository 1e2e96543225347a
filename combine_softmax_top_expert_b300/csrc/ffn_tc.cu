// Tensor-core expert FFN (tcgen05): not yet implemented in this file.
#include "ffn.cuh"

namespace moe {
moe_status_t ffn_bf16(const FfnArgs &, cudaStream_t) { return MOE_ERR_UNSUPPORTED; }
moe_status_t ffn_e4m3(const FfnArgs &, cudaStream_t) { return MOE_ERR_UNSUPPORTED; }
}  // namespace moe
