// moe_api.cu - the C ABI declared in include/moe.h: argument validation and
// launches.  Every check happens before anything is enqueued.
#include <string.h>

#include "moe_common.cuh"
#include "moe_launch.h"

using namespace moe;

namespace {

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

bool expert_format(int q) {
    return q == MOE_Q8_0 || q == MOE_Q4_K || q == MOE_Q2_K || q == MOE_MXFP4 || q == MOE_Q6_K || q == MOE_Q3_K;
}

// columns a packed matrix of this format accepts
bool cols_ok(int q, int cols) {
    if (cols <= 0) return false;
    if (q == MOE_MXFP4) return cols % 32 == 0;
    return cols % 256 == 0;
}

size_t packed_bytes(int q, int rows, int cols) {
    if (rows <= 0 || rows % 32 || !expert_format(q) || !cols_ok(q, cols)) return 0;
    size_t tile;
    switch (q) {
        case MOE_Q4_K: tile = FQ4K::tile_bytes(cols); break;
        case MOE_Q2_K: tile = FQ2K::tile_bytes(cols); break;
        case MOE_Q8_0: tile = FQ80::tile_bytes(cols); break;
        case MOE_Q6_K: tile = FQ6K::tile_bytes(cols); break;
        case MOE_Q3_K: tile = FQ3K::tile_bytes(cols); break;
        default: tile = FMX4::tile_bytes(cols); break;
    }
    return (size_t)(rows / 32) * tile;
}

moe_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return MOE_OK;
    if (e == cudaErrorInvalidConfiguration || e == cudaErrorNotSupported) return MOE_ERR_UNSUPPORTED;
    return MOE_ERR_CUDA;
}

size_t route_ws(int T, int E, int H) {
    const int nseg = (H + 1023) / 1024;
    return 256 + (size_t)T * E * nseg * sizeof(float);
}

bool pool_ok(const moe_pool *p, bool shared) {
    if (!p || !p->experts || !expert_format(p->qtype)) return false;
    if (p->H <= 0 || p->I <= 0 || p->H % 32 || p->I % 32) return false;
    if (shared ? p->E != 1 : (p->E < 1 || p->E > MOE_MAX_EXPERTS)) return false;
    return true;
}

// formats whose records span 256 columns need 256-blocks of activations
bool pool_shape_ok(const moe_pool *p) {
    if (!cols_ok(p->qtype, p->H) || !cols_ok(p->qtype, p->I)) return false;
    return act_block(p->H) != 0 && act_block(p->I) != 0;
}

}  // namespace

namespace moe {
moe_status ffn_check_args(const void *xq, int T, const int32_t *ids, const float *weights, int k,
                          const moe_pool *pool, const moe_pool *shared, const float *shared_scale, const float *y) {
    if (T < 0 || T > MOE_MAX_TOKENS || k < 1 || k > MOE_MAX_K) return MOE_ERR_INVALID_ARG;
    if (!pool_ok(pool, false)) return MOE_ERR_INVALID_ARG;
    if (shared && !pool_ok(shared, true)) return MOE_ERR_INVALID_ARG;
    if (!pool_shape_ok(pool)) return MOE_ERR_UNSUPPORTED;
    if (shared && (shared->H != pool->H || !pool_shape_ok(shared))) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    if (!xq || !ids || !weights || !y || !aligned16(xq) || !aligned16(y)) return MOE_ERR_INVALID_ARG;
    if (shared_scale && !shared) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}
}  // namespace moe

extern "C" {

int moe_act_block(int n) { return act_block(n); }

size_t moe_q8_row_bytes(int n) { return q8_row_bytes(n); }

size_t moe_packed_bytes(moe_qtype qtype, int rows, int cols) { return packed_bytes(qtype, rows, cols); }

moe_status moe_pack_weights(const void *blocks, moe_qtype qtype, int rows, int cols, void *packed,
                            cudaStream_t stream) {
    if (!blocks || !packed) return MOE_ERR_INVALID_ARG;
    if (rows <= 0 || cols <= 0) return MOE_ERR_INVALID_ARG;
    if (packed_bytes(qtype, rows, cols) == 0) return MOE_ERR_UNSUPPORTED;
    if (!aligned16(packed)) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_pack((const uint8_t *)blocks, qtype, rows, cols, (uint8_t *)packed, stream));
}

moe_status moe_quantize_q8K(const float *x, int T, int n, void *xq, cudaStream_t stream) {
    if (T < 0 || T > MOE_MAX_TOKENS * 64) return MOE_ERR_INVALID_ARG;
    if (!act_block(n)) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    if (!x || !xq || !aligned16(x) || !aligned16(xq)) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_quantize(x, T, n, (uint8_t *)xq, stream));
}

size_t moe_route_workspace_bytes(int T, int E, int H) {
    if (T <= 0 || E <= 0 || H <= 0) return 0;
    return route_ws(T, E, H);
}

moe_status moe_route(const float *hidden, const void *xq, int T, int H, const void *w_router, moe_qtype rtype,
                     int E, const float *router_bias, int k, moe_gating gating, int renormalize, int32_t *ids,
                     float *weights, float *logits_out, const float *shared_gate, float *shared_scale, void *ws,
                     size_t ws_bytes, cudaStream_t stream) {
    if (T < 0 || T > MOE_MAX_TOKENS || H <= 0 || H % 32 || E < 1 || E > MOE_MAX_EXPERTS) return MOE_ERR_INVALID_ARG;
    if (k < 1 || k > E || k > MOE_MAX_K) return MOE_ERR_INVALID_ARG;
    if (gating != MOE_GATE_SOFTMAX && gating != MOE_GATE_SIGMOID) return MOE_ERR_INVALID_ARG;
    if (rtype != MOE_F32 && rtype != MOE_Q8_0) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    if (!w_router || !ids || !weights) return MOE_ERR_INVALID_ARG;
    if (!aligned16(w_router)) return MOE_ERR_INVALID_ARG;
    if (rtype == MOE_F32 && (!hidden || !aligned16(hidden))) return MOE_ERR_INVALID_ARG;
    if (rtype == MOE_Q8_0) {
        if (H % 256) return MOE_ERR_UNSUPPORTED;
        if (!xq || !aligned16(xq)) return MOE_ERR_INVALID_ARG;
    }
    if ((shared_gate == nullptr) != (shared_scale == nullptr)) return MOE_ERR_INVALID_ARG;
    if (shared_gate && (!hidden || !aligned16(hidden) || !aligned16(shared_gate))) return MOE_ERR_INVALID_ARG;
    if (!ws || ws_bytes < route_ws(T, E, H) || !aligned16(ws)) return MOE_ERR_WORKSPACE;
    RouteArgs a;
    a.hidden = hidden;
    a.xq = (const uint8_t *)xq;
    a.w = w_router;
    a.bias = router_bias;
    a.ids = ids;
    a.weights = weights;
    a.logits_out = logits_out;
    a.counter = (unsigned *)ws;
    a.partial = (float *)((char *)ws + 256);
    a.T = T;
    a.H = H;
    a.E = E;
    a.k = k;
    a.nseg = (H + 1023) / 1024;
    a.gating = gating;
    a.renorm = renormalize ? 1 : 0;
    a.shared_gate = shared_gate;
    a.shared_scale = shared_scale;
    if (shared_gate) {
        const moe_status st = cuda_status(launch_shared_gate(hidden, T, H, shared_gate, shared_scale, stream));
        if (st != MOE_OK) return st;
    }
    return cuda_status(launch_route(a, rtype, stream));
}

size_t moe_ffn_workspace_bytes(int T, int k, const moe_pool *pool, const moe_pool *shared) {
    if (T < 0 || k < 1 || !pool) return 0;
    return ffn_ws_layout(T, k, pool->H, pool->I, shared ? shared->I : 0).total;
}

moe_status moe_expert_ffn(const void *xq, int T, const int32_t *ids, const float *weights, int k,
                          const moe_pool *pool, const moe_pool *shared, const float *shared_scale, float *y,
                          void *ws, size_t ws_bytes, cudaStream_t stream) {
    const moe_status v = moe::ffn_check_args(xq, T, ids, weights, k, pool, shared, shared_scale, y);
    if (v != MOE_OK || T == 0) return v;
    const FfnWs L = ffn_ws_layout(T, k, pool->H, pool->I, shared ? shared->I : 0);
    if (!ws || ws_bytes < L.total || !aligned16(ws)) return MOE_ERR_WORKSPACE;
    char *w = (char *)ws;
    FfnArgs a;
    a.xq = (const uint8_t *)xq;
    a.ids = ids;
    a.weights = weights;
    a.experts = pool->experts;
    a.shared = shared ? shared->experts : nullptr;
    a.shared_scale = shared_scale;
    a.y = y;
    a.status = (unsigned *)(w + L.status);
    a.counters = (unsigned *)(w + L.counters);
    a.h_r = (float *)(w + L.h_r);
    a.h_s = (float *)(w + L.h_s);
    a.hq_r = (uint8_t *)(w + L.hq_r);
    a.hq_s = (uint8_t *)(w + L.hq_s);
    a.T = T;
    a.k = k;
    a.H = pool->H;
    a.I = pool->I;
    a.Is = shared ? shared->I : 0;
    a.E = pool->E;
    a.qtype = pool->qtype;
    a.sqtype = shared ? shared->qtype : pool->qtype;
    return cuda_status(launch_ffn(a, stream));
}

moe_status moe_sum_partials(const float *parts, int R, size_t n, float *y, cudaStream_t stream) {
    if (R < 1 || R > MOE_MAX_RANKS || n % 4) return MOE_ERR_INVALID_ARG;
    if (n == 0) return MOE_OK;
    if (!parts || !y || !aligned16(parts) || !aligned16(y)) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_sum_partials(parts, R, n, y, stream));
}

moe_status moe_read_device_status(void *ws, int clear, uint32_t *flags, cudaStream_t stream) {
    if (!ws || !flags) return MOE_ERR_INVALID_ARG;
    uint32_t v = 0;
    if (cudaMemcpyAsync(&v, ws, sizeof v, cudaMemcpyDeviceToHost, stream) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
    if (clear && v) {
        if (cudaMemsetAsync(ws, 0, sizeof v, stream) != cudaSuccess) return MOE_ERR_CUDA;
        if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
    }
    *flags = v;
    return v ? MOE_ERR_DEVICE_STATUS : MOE_OK;
}

moe_status moe_debug_row_dots(const void *packed, moe_qtype qtype, int rows, int cols, int row, const void *xq,
                              int32_t *isums, cudaStream_t stream) {
    if (!packed || !xq || !isums) return MOE_ERR_INVALID_ARG;
    if (packed_bytes(qtype, rows, cols) == 0) return MOE_ERR_UNSUPPORTED;
    if (row < 0 || row >= rows) return MOE_ERR_INVALID_ARG;
    if (!aligned16(xq) || !aligned16(packed)) return MOE_ERR_INVALID_ARG;
    if (qtype != MOE_MXFP4 && act_block(cols) != 256) return MOE_ERR_UNSUPPORTED;
    return cuda_status(launch_row_dots((const uint8_t *)packed, qtype, cols, row, (const uint8_t *)xq, isums,
                                       stream));
}

const char *moe_status_str(moe_status s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported format or shape";
        case MOE_ERR_WORKSPACE: return "workspace missing or too small";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_DEVICE_STATUS: return "device reported a data error";
        case MOE_ERR_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

}  // extern "C"
