// moe_fused_mx4.cu - fused layer kernel instantiated for routed FMX4 experts
// (shared expert in the same format or Q8_0).  One translation unit per
// routed format so the kernels compile in parallel.
#include "moe_fused.cuh"

namespace moe {

cudaError_t launch_layer_mx4(const LayerArgs &a, int sqtype, int G, size_t smem, bool pdl, cudaStream_t s) {
    if (sqtype == MOE_MXFP4 || !a.shared) return launch_layer_nt<FMX4, FMX4>(a, G, smem, pdl, s);
    if (sqtype == MOE_Q8_0) return launch_layer_nt<FMX4, FQ80>(a, G, smem, pdl, s);
    return cudaErrorNotSupported;
}

}  // namespace moe
