// moe_fused_q3k.cu - fused layer kernel instantiated for routed FQ3K experts
// (shared expert in the same format or Q8_0).  One translation unit per
// routed format so the kernels compile in parallel.
#include "moe_fused.cuh"

namespace moe {

cudaError_t launch_layer_q3k(const LayerArgs &a, int sqtype, int G, size_t smem, bool pdl, cudaStream_t s) {
    if (sqtype == MOE_Q3_K || !a.shared) return launch_layer_nt<FQ3K, FQ3K>(a, G, smem, pdl, s);
    if (sqtype == MOE_Q8_0) return launch_layer_nt<FQ3K, FQ80>(a, G, smem, pdl, s);
    return cudaErrorNotSupported;
}

}  // namespace moe
