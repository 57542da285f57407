// moe_noalloc.cu - moe_expert_ffn for callers that cannot allocate device
// memory.
//
// moe_expert_ffn needs a scratch workspace (h, its q8 records, tickets and
// the status word) that the caller allocates.  Some callers cannot do that:
// code that runs against a fixed device-memory plan settled at start-up
// (nothing may be allocated once serving has begun), plugin hosts that hand
// a component its inputs and outputs but no allocator, and callers on paths
// where cudaMalloc/cudaFree are off limits because they can synchronise the
// device or fail under memory pressure.  This variant keeps its scratch in a
// fixed array that lives in the library's own device image instead; it
// allocates nothing.
#include <mutex>

#include "moe_common.cuh"
#include "moe_launch.h"

namespace {

// Scratch for one call; every device that loads the library holds it until
// the process exits.
constexpr size_t kStaticScratchBytes = (size_t)2 << 20;   // 2 MiB
static __device__ __align__(256) unsigned char g_ffn_scratch[kStaticScratchBytes];

std::mutex g_setup_mu;
void *g_scratch_addr[64] = {nullptr};

// Host code must not use g_ffn_scratch directly: on the host that name is
// only a stand-in.  The device address is looked up once per device, with
// that device current.
cudaError_t scratch_for_current_device(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_ffn_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

using namespace moe;

extern "C" moe_status moe_expert_ffn_noalloc(const void *xq, int T, const int32_t *ids, const float *weights,
                                             int k, const moe_pool *pool, const moe_pool *shared,
                                             const float *shared_scale, float *y, cudaStream_t stream) {
    // every check moe_expert_ffn makes comes first, so a call it would reject
    // enqueues nothing (not even the clear of the shared scratch below)
    const moe_status v = ffn_check_args(xq, T, ids, weights, k, pool, shared, shared_scale, y);
    if (v != MOE_OK) return v;
    const FfnWs L = ffn_ws_layout(T, k, pool->H, pool->I, shared ? shared->I : 0);
    if (L.total > kStaticScratchBytes) return MOE_ERR_WORKSPACE;   // beyond the fixed scratch
    if (T == 0) return MOE_OK;
    void *scratch = nullptr;
    if (scratch_for_current_device(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
    // the array keeps the previous call's contents: the status word and the
    // tickets must start at zero
    if (cudaMemsetAsync(scratch, 0, L.h_r, stream) != cudaSuccess) return MOE_ERR_CUDA;
    return moe_expert_ffn(xq, T, ids, weights, k, pool, shared, shared_scale, y, scratch, kStaticScratchBytes,
                          stream);
}
