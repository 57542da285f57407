// moe_fused_api.cu - moe_layer_forward: validation, workspace and shared
// memory planning, dispatch of the fused layer kernel (moe_fused.cuh).
#include "moe_common.cuh"
#include "moe_launch.h"

namespace moe {

cudaError_t launch_layer_q4k(const LayerArgs &a, int sqtype, int G, size_t smem, bool pdl, cudaStream_t s);
cudaError_t launch_layer_q2k(const LayerArgs &a, int sqtype, int G, size_t smem, bool pdl, cudaStream_t s);
cudaError_t launch_layer_q80(const LayerArgs &a, int sqtype, int G, size_t smem, bool pdl, cudaStream_t s);
cudaError_t launch_layer_mx4(const LayerArgs &a, int sqtype, int G, size_t smem, bool pdl, cudaStream_t s);
cudaError_t launch_layer_q6k(const LayerArgs &a, int sqtype, int G, size_t smem, bool pdl, cudaStream_t s);
cudaError_t launch_layer_q3k(const LayerArgs &a, int sqtype, int G, size_t smem, bool pdl, cudaStream_t s);

// constants mirrored from moe_fused.cuh (kept in one place there; checked below)
constexpr int kNBAR = 32;
// consumer warps of the kernel for a launch's token count (Warps<NT> in the kernel)
static int consumer_warps(int NT) { return NT == 1 ? 16 : 8; }
constexpr uint32_t kRingDefault = 160 * 1024;

static size_t al16(size_t v) { return (v + 15) & ~(size_t)15; }

LayerWs layer_ws_layout(int T, int k, int H, int I, int Is, int E) {
    auto al = [](size_t v) { return (v + 255) & ~(size_t)255; };
    const size_t P = (size_t)T * k;
    LayerWs w;
    w.status = 0;
    w.epoch = 256;                   // one launch counter per block (G <= 256)
    w.logits = w.epoch + 4 * 256;
    w.h_r = al(w.logits + 8 * (size_t)T * E);
    w.h_s = al(w.h_r + 8 * P * I);
    w.o_r = al(w.h_s + 8 * (size_t)T * (Is > 0 ? Is : 0));
    w.o_s = al(w.o_r + 8 * P * H);
    w.total = al(w.o_s + 8 * (size_t)T * H);
    return w;
}

// largest packed record of a format for rows of `cols` columns
static uint32_t max_rec(int q, int cols) {
    switch (q) {
        case MOE_Q4_K: return 9 * 512;
        case MOE_Q2_K: return 5 * 512 + 128;
        case MOE_Q8_0: return 17 * 512;
        case MOE_Q6_K: return FQ6K::REC;
        case MOE_Q3_K: return FQ3K::REC;
        default: {
            const int nb = cols / 32 < 8 ? cols / 32 : 8;
            return (uint32_t)nb * 512 + 256;
        }
    }
}
static size_t tile_bytes_of(int q, int cols) {
    switch (q) {
        case MOE_Q4_K: return FQ4K::tile_bytes(cols);
        case MOE_Q2_K: return FQ2K::tile_bytes(cols);
        case MOE_Q8_0: return FQ80::tile_bytes(cols);
        case MOE_Q6_K: return FQ6K::tile_bytes(cols);
        case MOE_Q3_K: return FQ3K::tile_bytes(cols);
        default: return FMX4::tile_bytes(cols);
    }
}

// The kernel's work plan counts bytes in 128-byte lines with 32-bit
// integers: every expert of the call at once must stay below 2^28 lines.
static bool plan_fits(const LayerArgs &a, int qtype, int sqtype) {
    const size_t P = (size_t)a.T * a.k;
    size_t lines = P * (2 * tile_bytes_of(qtype, a.H) * (size_t)(a.I / 32) + tile_bytes_of(qtype, a.I) * (size_t)(a.H / 32));
    if (a.shared) lines += 2 * tile_bytes_of(sqtype, a.H) * (size_t)(a.Is / 32) + tile_bytes_of(sqtype, a.Is) * (size_t)(a.H / 32);
    return (lines >> 7) < ((size_t)1 << 28);   // x4 (quarter lines) stays below 2^30
}

// smallest possible ring item of a format: a gate+up record pair, or one down record
static uint32_t max_item(int q, int H, int I) {
    const uint32_t a = 2 * max_rec(q, H), b = max_rec(q, I);
    return a > b ? a : b;
}
// log2 of the records per ring item: the largest power of two (1 to 8) that
// keeps an item within a quarter of the ring (fewer, larger copies land sooner)
static int lg_recs_per_item(size_t ring, uint32_t rec_bytes) {
    const size_t r = ring / 4 / rec_bytes;
    return r >= 8 ? 3 : (r >= 4 ? 2 : (r >= 2 ? 1 : 0));
}

static long long g_exchange_wait = 0;   // 0: the kernel's default bound
void set_exchange_wait(long long cycles) { g_exchange_wait = cycles; }

cudaError_t launch_layer(LayerArgs &a, int qtype, int sqtype, bool pdl, cudaStream_t s) {
    if (!plan_fits(a, qtype, sqtype)) return cudaErrorNotSupported;
    a.wait_limit = g_exchange_wait > 0 ? g_exchange_wait : 800ll * 1000ll * 1000ll;
    a.balpha = 3;   // A bytes count three quarters (235B-A22B-style layer: measured against 0, 1/4, 1/2 and 1)
    int G = num_sms();
    if (G > 256) G = 256;
    const int nseg = (a.H + 1023) / 1024;
    const int rr = (a.E + G - 1) / G;   // router rows per block, at most
    const size_t rowb = a.rtype == MOE_F32 ? (size_t)a.H * 4 : (size_t)(a.H / 32) * 34;
    uint32_t item = max_item(qtype, a.H, a.I);
    if (a.shared) {
        const uint32_t si = max_item(sqtype, a.H, a.Is);
        if (si > item) item = si;
    }
    a.table_in_smem = (size_t)a.E * sizeof(moe_expert) <= 16 * 1024 ? 1 : 0;
    a.xrec = q8_row_bytes(a.H);
    const int Imax = a.Is > a.I ? a.Is : a.I;
    a.hrec = q8_row_bytes(Imax);
    a.NT = a.T <= 1 ? 1 : 4;   // batches above 4 tokens never reach the fused kernel
    // A units: two alternating buffers of the warps' gate and up partials;
    // B batches: per-record partials, 64 slots for one token, 32 for four
    a.bslots = a.NT == 1 ? 64 : 32;
    size_t red_bytes = (size_t)2 * consumer_warps(a.NT) * 2 * a.NT * 32 * 4;
    if ((size_t)a.bslots * a.NT * 32 * 4 > red_bytes) red_bytes = (size_t)a.bslots * a.NT * 32 * 4;

    Smem o;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = al16(off + bytes);
        return (uint32_t)at;
    };
    const size_t fixed_router = (size_t)rr * rowb;
    // everything but the ring and the hq records
    const size_t fixed_core = (2 * kNBAR + 5) * 8 + 2 * kNBAR * 4 + fixed_router +
                              (a.table_in_smem ? a.E * sizeof(moe_expert) : 0) + a.T * a.xrec +
                              4 * (size_t)a.T * a.E + 4 * (size_t)rr * nseg * a.T + 8 * (size_t)a.P +
                              4 * (5 * (size_t)a.P + 1) + red_bytes + kLayerMiscBytes + 16 * 16;
    const size_t optin = (size_t)smem_optin();
    {   // hq records: every pair when they fit in 48 KB and leave room for the
        // ring, never fewer than one expert's (T)
        const size_t want = (size_t)a.P + (a.shared ? a.T : 0);
        size_t fit = (48 * 1024) / a.hrec;
        if (fixed_core + 2 * (size_t)item < optin) {
            const size_t room = (optin - fixed_core - 2 * (size_t)item) / a.hrec;
            if (room < fit) fit = room;
        }
        if (fit < (size_t)a.T) fit = a.T;
        a.hq_slots = (int)(want < fit ? want : fit);
    }
    const size_t fixed_rest = fixed_core + (size_t)a.hq_slots * a.hrec;
    if (fixed_rest + 2 * (size_t)item > optin) return cudaErrorInvalidConfiguration;
    size_t ring = kRingDefault;
    if (ring < 2 * (size_t)item) ring = 2 * (size_t)item;
    if (fixed_rest + ring > optin) ring = (optin - fixed_rest) & ~(size_t)127;
    a.ring_bytes = (uint32_t)ring;
    // items per format: a small routed record (Q2_K) beside a large shared one
    // (Q8_0) still gets copies of several records
    a.lgra = lg_recs_per_item(ring, 2 * max_rec(qtype, a.H));
    a.lgrb = lg_recs_per_item(ring, max_rec(qtype, a.I));
    a.lgsa = a.shared ? lg_recs_per_item(ring, 2 * max_rec(sqtype, a.H)) : 0;
    a.lgsb = a.shared ? lg_recs_per_item(ring, max_rec(sqtype, a.Is)) : 0;
    o.ring = take(ring);
    o.bars = take((2 * kNBAR + 5) * 8);   // ring full/empty, fixed bytes, A partials ready/free x 2
    o.starts = take(2 * kNBAR * 4);   // item start offsets, then slot tags
    o.router = take(fixed_router);
    o.table = take(a.table_in_smem ? a.E * sizeof(moe_expert) : 0);
    o.xq = take(a.T * a.xrec);
    o.hq = take((size_t)a.hq_slots * a.hrec);
    o.lg = take(4 * (size_t)a.T * a.E);
    o.segv = take(4 * (size_t)rr * nseg * a.T);
    o.ids = take(4 * (size_t)a.P);
    o.wts = take(4 * (size_t)a.P);
    o.grp = take(4 * (5 * (size_t)a.P + 1));
    o.red = take(red_bytes);
    o.misc = take(kLayerMiscBytes);
    o.total = (uint32_t)off;
    if (o.total > optin) return cudaErrorInvalidConfiguration;
    a.sm = o;
    switch (qtype) {
        case MOE_Q4_K: return launch_layer_q4k(a, sqtype, G, o.total, pdl, s);
        case MOE_Q2_K: return launch_layer_q2k(a, sqtype, G, o.total, pdl, s);
        case MOE_Q8_0: return launch_layer_q80(a, sqtype, G, o.total, pdl, s);
        case MOE_MXFP4: return launch_layer_mx4(a, sqtype, G, o.total, pdl, s);
        case MOE_Q6_K: return launch_layer_q6k(a, sqtype, G, o.total, pdl, s);
        case MOE_Q3_K: return launch_layer_q3k(a, sqtype, G, o.total, pdl, s);
    }
    return cudaErrorNotSupported;
}

}  // namespace moe

using namespace moe;

namespace {
bool al16p(const void *p) { return ((uintptr_t)p & 15u) == 0; }
bool fmt_ok(int q) {
    return q == MOE_Q8_0 || q == MOE_Q4_K || q == MOE_Q2_K || q == MOE_MXFP4 || q == MOE_Q6_K || q == MOE_Q3_K;
}
bool cols_ok(int q, int cols) { return cols > 0 && (q == MOE_MXFP4 ? cols % 32 == 0 : cols % 256 == 0); }
}  // namespace

// Batches above this size take the three separate kernels: every record is
// then dotted with many tokens, and the persistent kernel's eight consumer
// warps per SM run out of latency hiding where the separate kernels, with
// several blocks per SM, do not.
constexpr int kFusedMaxTokens = 4;

// workspace of the separate-kernel route for larger batches: the FFN
// workspace first (its status word is the layer's), then the router's, the
// q8 activations, ids and weights
struct SplitWs {
    size_t ffn, route, xq, ids, w, sscale, total;
};
SplitWs split_ws_layout(int T, int k, const moe_pool *pool, const moe_pool *shared) {
    auto al = [](size_t v) { return (v + 255) & ~(size_t)255; };
    SplitWs s;
    s.ffn = 0;
    s.route = al(moe_ffn_workspace_bytes(T, k, pool, shared));
    s.xq = al(s.route + moe_route_workspace_bytes(T, pool->E, pool->H));
    s.ids = al(s.xq + (size_t)T * q8_row_bytes(pool->H));
    s.w = al(s.ids + 4 * (size_t)T * k);
    s.sscale = al(s.w + 4 * (size_t)T * k);
    s.total = al(s.sscale + 4 * (size_t)T);
    return s;
}

extern "C" {

moe_status moe_debug_set_exchange_wait(long long cycles) {
    if (cycles < 0) return MOE_ERR_INVALID_ARG;
    set_exchange_wait(cycles);
    return MOE_OK;
}

size_t moe_layer_workspace_bytes(int T, int k, const moe_pool *pool, const moe_pool *shared) {
    if (T < 1 || k < 1 || !pool) return 0;
    if (T > kFusedMaxTokens) return split_ws_layout(T, k, pool, shared).total;
    return layer_ws_layout(T, k, pool->H, pool->I, shared ? shared->I : 0, pool->E).total;
}

moe_status moe_layer_forward(const float *hidden, int T, const void *w_router, moe_qtype rtype,
                             const float *router_bias, int k, moe_gating gating, int renormalize,
                             const moe_pool *pool, const moe_pool *shared, const float *shared_gate, float *y,
                             int32_t *ids_out,
                             float *weights_out, float *logits_out, void *xq_out, void *ws, size_t ws_bytes,
                             unsigned flags, cudaStream_t stream) {
    if (T < 0 || T > MOE_MAX_TOKENS || k < 1 || k > MOE_MAX_K) return MOE_ERR_INVALID_ARG;
    if (!pool || !pool->experts || !fmt_ok(pool->qtype)) return MOE_ERR_INVALID_ARG;
    const int H = pool->H, I = pool->I, E = pool->E;
    if (H <= 0 || I <= 0 || H % 32 || I % 32 || E < 1 || E > MOE_MAX_EXPERTS || k > E) return MOE_ERR_INVALID_ARG;
    if (gating != MOE_GATE_SOFTMAX && gating != MOE_GATE_SIGMOID) return MOE_ERR_INVALID_ARG;
    if (shared && (!shared->experts || shared->E != 1 || !fmt_ok(shared->qtype) || shared->I <= 0 ||
                   shared->I % 32 || shared->H != H))
        return MOE_ERR_INVALID_ARG;
    if (rtype != MOE_F32 && rtype != MOE_Q8_0) return MOE_ERR_UNSUPPORTED;
    if (rtype == MOE_Q8_0 && H % 256) return MOE_ERR_UNSUPPORTED;
    if (!cols_ok(pool->qtype, H) || !cols_ok(pool->qtype, I)) return MOE_ERR_UNSUPPORTED;
    if (shared && (!cols_ok(shared->qtype, H) || !cols_ok(shared->qtype, shared->I))) return MOE_ERR_UNSUPPORTED;
    if (shared && shared->qtype != pool->qtype && shared->qtype != MOE_Q8_0) return MOE_ERR_UNSUPPORTED;
    if (shared_gate && (!shared || !al16p(shared_gate))) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!hidden || !w_router || !y || !al16p(hidden) || !al16p(w_router) || !al16p(y)) return MOE_ERR_INVALID_ARG;
    if (xq_out && !al16p(xq_out)) return MOE_ERR_INVALID_ARG;
    if (T > kFusedMaxTokens) {   // the three kernels back to back, through their own entry points
        const SplitWs S = split_ws_layout(T, k, pool, shared);
        if (!ws || ws_bytes < S.total || !al16p(ws)) return MOE_ERR_WORKSPACE;
        char *w = (char *)ws;
        void *xq = xq_out ? xq_out : (void *)(w + S.xq);
        int32_t *ids = ids_out ? ids_out : (int32_t *)(w + S.ids);
        float *wts = weights_out ? weights_out : (float *)(w + S.w);
        float *sscale = shared_gate ? (float *)(w + S.sscale) : nullptr;
        moe_status st = moe_quantize_q8K(hidden, T, H, xq, stream);
        if (st == MOE_OK)
            st = moe_route(hidden, xq, T, H, w_router, rtype, E, router_bias, k, gating, renormalize, ids, wts,
                           logits_out, shared_gate, sscale, w + S.route, S.xq - S.route, stream);
        if (st == MOE_OK)
            st = moe_expert_ffn(xq, T, ids, wts, k, pool, shared, sscale, y, w + S.ffn, S.route, stream);
        return st;
    }
    const LayerWs L = layer_ws_layout(T, k, H, I, shared ? shared->I : 0, E);
    if (!ws || ws_bytes < L.total || !al16p(ws)) return MOE_ERR_WORKSPACE;
    char *w = (char *)ws;
    LayerArgs a = {};
    a.x = hidden;
    a.w_router = w_router;
    a.rbias = router_bias;
    a.experts = pool->experts;
    a.shared = shared ? shared->experts : nullptr;
    a.shared_gate = shared_gate;
    a.y = y;
    a.ids_out = ids_out;
    a.w_out = weights_out;
    a.logits_out = logits_out;
    a.xq_out = (uint8_t *)xq_out;
    a.status = (unsigned *)(w + L.status);
    a.epoch = (unsigned *)(w + L.epoch);
    typedef unsigned long long tw;
    a.logits = (tw *)(w + L.logits);
    a.h_r = (tw *)(w + L.h_r);
    a.h_s = (tw *)(w + L.h_s);
    a.o_r = (tw *)(w + L.o_r);
    a.o_s = (tw *)(w + L.o_s);
    a.rtype = rtype;
    a.k = k;
    a.gating = gating;
    a.renorm = renormalize ? 1 : 0;
    a.T = T;
    a.H = H;
    a.I = I;
    a.Is = shared ? shared->I : 0;
    a.E = E;
    a.P = T * k;
    const cudaError_t e =
        launch_layer(a, pool->qtype, shared ? shared->qtype : pool->qtype, (flags & MOE_LAYER_OVERLAP_PREVIOUS) != 0,
                     stream);
    if (e == cudaSuccess) return MOE_OK;
    if (e == cudaErrorInvalidConfiguration || e == cudaErrorNotSupported) return MOE_ERR_UNSUPPORTED;
    return MOE_ERR_CUDA;
}

}  // extern "C"
