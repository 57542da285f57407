// moe_fused_q80.cu - fused layer kernel instantiated for routed FQ80 experts
// (shared expert in the same format or Q8_0).  One translation unit per
// routed format so the kernels compile in parallel.
#include "moe_fused.cuh"

namespace moe {

cudaError_t launch_layer_q80(const LayerArgs &a, int sqtype, int G, size_t smem, bool pdl, cudaStream_t s) {
    if (sqtype == MOE_Q8_0 || !a.shared) return launch_layer_nt<FQ80, FQ80>(a, G, smem, pdl, s);
    return cudaErrorNotSupported;
}

}  // namespace moe
