/*
 * moe.h - C ABI of the GB300 (sm_103a) quantized routed-expert MoE FFN.
 *
 * One decode step of a Mixture-of-Experts layer, as the pulsar README states
 * it ("MoE resolve" passage and the model table):
 *   1. moe_quantize_q8K : activations -> q8 blocks (integer dots follow,
 *                         "activations quantized to q8_0/q8_K").
 *   2. moe_route        : router GEMV, softmax or sigmoid top-k (README model
 *                         table: "softmax router", "sigmoid-gated router").
 *   3. moe_expert_ffn   : per (token, slot) the chosen expert's gate/up GEMVs
 *                         over block-quantised weights, SwiGLU, requantised h,
 *                         the down GEMV, the routing-weight scale and the
 *                         fixed-order per-token sum, plus the shared expert.
 *                         Experts arrive as explicit per-expert device
 *                         pointers and a NULL gate pointer means "not mine"
 *                         (README, "MoE resolve": the kernels receive
 *                         per-(token, slot) pointers; NULL means not mine).
 *
 * Conventions for every call:
 *  - All pointers named "device" are CUDA device pointers; the library never
 *    dereferences them on the host.  Host pointers are marked "host".
 *  - The caller owns every buffer.  The library allocates nothing, keeps no
 *    state between calls and never synchronises the host, except
 *    moe_read_device_status, which does.
 *  - Calls are asynchronous and ordered on the given stream (0 = legacy
 *    default stream).  Argument errors are returned before anything is
 *    launched; a failed launch returns MOE_ERR_CUDA.
 *  - Inputs must be finite.  Weights and expert tables are read-only for the
 *    duration of a call.
 *  - Results are deterministic: identical inputs give bit-identical outputs,
 *    whatever the batch composition (see moe_expert_ffn).
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* NULL where a buffer is required, bad size or shape */
    MOE_ERR_UNSUPPORTED = 2,   /* valid but not implemented (format/shape pairing)   */
    MOE_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required          */
    MOE_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed                */
    MOE_ERR_DEVICE_STATUS = 5, /* a kernel recorded a data error (see status word)    */
    MOE_ERR_TIMEOUT = 6        /* reserved: a bounded device-side wait gave up        */
} moe_status;

/* Weight formats (GGUF-style blocks; see moe_pack_weights for the bytes). */
typedef enum {
    MOE_F32 = 0,    /* plain fp32 (router only)                                   */
    MOE_Q8_0 = 1,   /* 32 weights: f16 d, i8 q[32]               w = d*q   (34 B)  */
    MOE_Q4_K = 2,   /* 256 weights: f16 d, f16 dmin, 6-bit sc/m x 8, 4-bit q (144 B) */
    MOE_Q2_K = 3,   /* 256 weights: 4-bit sc/m x 16, 2-bit q, f16 d, f16 dmin (84 B) */
    MOE_MXFP4 = 4,  /* 32 weights: E8M0 scale e, FP4 E2M1 q[32]  w = 2^(e-127)*q (17 B) */
    MOE_Q6_K = 5,   /* 256 weights: 4+2-bit q (offset 32), i8 sc x 16, f16 d     (210 B) */
    MOE_Q3_K = 6    /* 256 weights: 2+1-bit q (offset 4), 6-bit sc x 16, f16 d   (110 B) */
} moe_qtype;

typedef enum { MOE_GATE_SOFTMAX = 0, MOE_GATE_SIGMOID = 1 } moe_gating;

/* Device status word bits (moe_read_device_status). */
#define MOE_DEV_BAD_ID 0x1u       /* an expert id outside [0, E): that slot was skipped     */
#define MOE_DEV_DUP_ID 0x2u       /* an id repeated within one token: the repeat was skipped */
#define MOE_DEV_TIMEOUT 0x4u      /* a bounded wait in moe_layer_forward gave up: y is invalid,
                                     zero the workspace before the next call */

/* Limits of this build. */
#define MOE_MAX_TOKENS 16          /* T per call (small-batch decode)        */
#define MOE_MAX_K 32               /* top-k                                  */
#define MOE_MAX_EXPERTS 1024       /* E                                      */
#define MOE_MAX_RANKS 64           /* partial outputs summed by moe_sum_partials */

/* ------------------------------------------------------------------ sizes */

/* Activation quantisation block for a width n: 256 if n % 256 == 0, 32 if
 * n % 32 == 0 (the README's "multiple of 32 but not 256 -> q8_0" rule),
 * else 0 (unsupported). */
int moe_act_block(int n);

/* Bytes of one token's q8 activation record of width n (a multiple of 16):
 *   offset 0          : float d[n/B]        block scales, B = moe_act_block(n)
 *   offset A          : int8  q[n]          codes, A = 16-aligned 4*n/B
 *   offset A + n      : int16 bsum[n/16]    sum of each 16 consecutive codes
 * T tokens are T records back to back.  Returns 0 if n is unsupported. */
size_t moe_q8_row_bytes(int n);

/* Bytes of a packed weight matrix (rows x cols), 0 if unsupported.
 * rows % 32 == 0; cols % 256 == 0 for Q4_K, Q2_K, Q8_0, Q6_K and Q3_K;
 * cols % 32 == 0 for MXFP4.  The packed size equals the GGUF size except for
 * MXFP4 matrices whose cols/32 is not a multiple of 8, Q6_K (4 bytes per row
 * and 256 columns for d instead of 2) and Q3_K (112 bytes per row and 256
 * columns instead of 110). */
size_t moe_packed_bytes(moe_qtype qtype, int rows, int cols);

/* ------------------------------------------------------------- one-time pack */

/*
 * Lossless re-layout of a row-major matrix of GGUF-style blocks (device,
 * rows x cols/QK blocks, QK = 256 or 32) into the packed layout the FFN
 * kernels stream with 128-bit coalesced loads (device, moe_packed_bytes).
 * Same bits per weight; run once at load time.  This mirrors the README's
 * load-time tensor transforms (K-quant dense tensors are requantised when
 * loaded); here nothing is requantised, only moved.
 *
 * Packed layout: rows are cut into tiles of 32; a tile is a sequence of
 * records along the columns; a record is a set of 512-byte planes, plane p
 * holding 16 bytes for each of the 32 rows (row r of the tile at byte 16*r):
 *   Q4_K  : record = 1 block (256 cols); planes 0..8 = the block's bytes
 *           [16p, 16p+16) (plane 0: d, dmin, scales; 1..8: qs).      4608 B
 *   Q2_K  : record = 1 block; planes 0..4 = bytes [16p, 16p+16) (scales,
 *           qs), then one 128-byte plane of {d, dmin} (4 B per row). 2688 B
 *   Q8_0  : record = 8 blocks (256 cols); planes 2b, 2b+1 = q of block b,
 *           plane 16 = the 8 f16 d of the row.                       8704 B
 *   MXFP4 : record = nb <= 8 blocks (the last record of a row takes the
 *           remainder); planes 0..nb-1 = qs of block b, then a 256-byte
 *           plane of 8 scale bytes per row (unused bytes zero). nb*512+256 B
 *   Q6_K  : record = 1 block; planes 0..12 = bytes [16p, 16p+16) (ql, qh,
 *           the 16 int8 scales), then a 128-byte plane of {d, 0, 0}.  6784 B
 *   Q3_K  : record = 1 block; planes 0..5 = hmask and qs, plane 6 = the
 *           12 scale bytes, d and two zero bytes.                    3584 B
 * Errors: MOE_ERR_UNSUPPORTED for F32 or shapes outside the rules above.
 */
moe_status moe_pack_weights(const void *blocks, moe_qtype qtype, int rows, int cols,
                            void *packed, cudaStream_t stream);

/* ---------------------------------------------------------- hot-path calls */

/*
 * Activation quantisation (README "MoE resolve": activations quantised to
 * q8_0/q8_K before integer dots).  x: device fp32 [T][n]; xq: device, T
 * records of moe_q8_row_bytes(n); both 16-byte aligned.  Per block of
 * B = moe_act_block(n): amax = max|x|, d = amax/127, q = rint(x*(127/amax))
 * (round half to even; IEEE division), d = 0 and q = 0 for an all-zero
 * block; bsum = sums of 16 codes.  T in [0, MOE_MAX_TOKENS*64]; T == 0 is a
 * no-op.
 * Errors: MOE_ERR_UNSUPPORTED if moe_act_block(n) == 0; MOE_ERR_INVALID_ARG
 * for T out of range or a NULL or unaligned x or xq.
 */
moe_status moe_quantize_q8K(const float *x, int T, int n, void *xq, cudaStream_t stream);

/*
 * Router GEMV + top-k + gating (README intro: the router stays resident;
 * model table: softmax and sigmoid-gated routers, top-k of E).
 *   hidden      : device fp32 [T][H], 16-byte aligned (read by an F32 router)
 *   xq          : device q8 records of hidden (moe_quantize_q8K), required
 *                 for a Q8_0 router, ignored (may be NULL) for F32
 *   w_router    : device, F32 [E][H] row-major, or Q8_0 blocks [E][H/32]
 *                 (GGUF row-major, not packed; rows must be 16-byte aligned,
 *                 i.e. (H/32) % 8 == 0)
 *   router_bias : device fp32 [E] added to the logits, or NULL
 *   ids         : device int32 [T][k] out: the k largest logits, largest
 *                 first, the lower index first on equal logits
 *   weights     : device fp32 [T][k] out.  Softmax: exp(l - lmax) over the
 *                 chosen k, normalised to sum 1 (renormalize != 0) or over all
 *                 E (renormalize == 0).  Sigmoid: s = 1/(1+exp(-l)), divided
 *                 by the sum over the chosen k when renormalize != 0.
 *   logits_out  : device fp32 [T][E] out, or NULL
 *   shared_gate : device fp32 [H], 16-byte aligned, or NULL: the shared
 *                 expert's gate vector (the README's gate_inp_shexp, an f32
 *                 tensor; its use is not stated there, and the reading taken
 *                 is a per-token scalar gate on the shared expert's output)
 *   shared_scale: device fp32 [T] out with shared_gate (NULL without it):
 *                 sigma(shared_gate . hidden[t]), the logit in the fixed order
 *                 below (a one-row F32 router, hidden required), then
 *                 1/(1+exp(-l)); moe_expert_ffn takes it as the shared
 *                 expert's weight
 *   ws          : device workspace of moe_route_workspace_bytes(T, E, H) bytes,
 *                 zero-filled before its first use; every completed call
 *                 leaves it ready for the next one
 * Logits are fp32 in one fixed summation order, so ids are reproducible bit
 * for bit: the row is cut into 1024-element segments; in a segment, lane l of
 * 32 accumulates float4 chunks l, l+32, ... with fused multiply-adds in
 * element order; the 32 lane values are combined by an xor butterfly
 * (offsets 16, 8, 4, 2, 1); segment values are added in order, then the bias.
 * A Q8_0 router uses 32-block segments with lane l taking block l of the
 * segment, value (d_w*d_x)*isum.
 * Limits: 1 <= k <= min(E, MOE_MAX_K), E <= MOE_MAX_EXPERTS, T <= MOE_MAX_TOKENS,
 * H % 32 == 0.
 * Errors: MOE_ERR_INVALID_ARG for limits, gating, a NULL or unaligned
 * buffer, or shared_gate and shared_scale not given together (or a shared
 * gate without hidden); MOE_ERR_UNSUPPORTED for a router type other than F32/Q8_0 or a Q8_0
 * router with H % 256 != 0; MOE_ERR_WORKSPACE for a missing, short or
 * unaligned ws.
 */
moe_status moe_route(const float *hidden, const void *xq, int T, int H,
                     const void *w_router, moe_qtype rtype, int E, const float *router_bias,
                     int k, moe_gating gating, int renormalize,
                     int32_t *ids, float *weights, float *logits_out,
                     const float *shared_gate, float *shared_scale,
                     void *ws, size_t ws_bytes, cudaStream_t stream);
size_t moe_route_workspace_bytes(int T, int E, int H);

/* One expert: packed device matrices (moe_pack_weights) and optional biases.
 * A fused gate_up tensor (one [2I][H] matrix, gate rows first, as the README's
 * GGUF notes allow) packed as one matrix serves both projections: gate = its
 * start, up = gate + moe_packed_bytes(qtype, I, H), since packed tiles of 32
 * rows are stored one after another. */
typedef struct {
    const void *gate;     /* packed [I][H]; NULL: this expert is not owned here  */
    const void *up;       /* packed [I][H]                                        */
    const void *down;     /* packed [H][I]                                        */
    const float *b_gate;  /* device fp32 [I] or NULL                              */
    const float *b_up;    /* device fp32 [I] or NULL                              */
    const float *b_down;  /* device fp32 [H] or NULL (scaled by the routing weight) */
} moe_expert;

/* A set of experts of one format.  `experts` is a DEVICE array of E entries
 * (the per-expert pointer table stays on the device; the host never walks it). */
typedef struct {
    moe_qtype qtype;
    int H, I, E;
    const moe_expert *experts;
} moe_pool;

/*
 * Routed + shared expert FFN for T tokens (README "MoE resolve": integer
 * dots on q8 activations with per-block rescale; SwiGLU; per-slot weighted
 * sum; shared expert always on).
 *   xq      : device q8 records of the T hidden states (width pool->H),
 *             16-byte aligned
 *   ids     : device int32 [T][k]; weights: device fp32 [T][k]
 *   pool    : host pointer to the routed pool (qtype Q8_0, Q4_K, Q2_K, MXFP4,
 *             Q6_K or Q3_K)
 *   shared  : host pointer to a pool with E == 1 (no biases read), or NULL
 *   shared_scale: device fp32 [T], the shared expert's weight per token
 *             (moe_route's shared_scale), or NULL for weight 1; requires
 *             shared
 *   y       : device fp32 [T][H] out, 16-byte aligned, overwritten:
 *             y[t] = sum over slots s in slot order of w[t][s]*o(ids[t][s])
 *                    + g[t]*o_shared (added last; g = shared_scale or 1),
 *             o = W_down . q8(h) + b_down,  h = silu(g) * u,
 *             g = W_gate . xq + b_gate, u = W_up . xq + b_up (fp32 h is
 *             requantised with the moe_quantize_q8K rule, width I).
 *             Slots whose expert is not owned (gate == NULL) add nothing: an
 *             expert-parallel rank passes a pool with its non-owned entries
 *             NULL and receives a partial y.
 *   ws      : device workspace of moe_ffn_workspace_bytes() bytes, zero-filled
 *             before its first use.  The first 4 bytes are the device status
 *             word (MOE_DEV_* bits): an id outside [0, E) or repeated within a
 *             token is skipped and flagged there, without failing the call.
 * Every token's result is computed with the same arithmetic and order
 * whatever the other tokens of the batch, so a token's y is bit-identical
 * between T = 1 and any batch that contains it.
 * Limits: T <= MOE_MAX_TOKENS, k <= MOE_MAX_K, E <= MOE_MAX_EXPERTS;
 * H and I multiples of 32 (of 256 for Q4_K, Q2_K, Q8_0).
 * Errors: MOE_ERR_INVALID_ARG for limits, a pool with no expert table, an
 * unknown expert format, a NULL or unaligned buffer, or shared_scale without
 * a shared pool; MOE_ERR_UNSUPPORTED for widths the format cannot hold or a
 * shared pool of another H;
 * MOE_ERR_WORKSPACE for a missing, short or unaligned ws.
 */
moe_status moe_expert_ffn(const void *xq, int T, const int32_t *ids, const float *weights, int k,
                          const moe_pool *pool, const moe_pool *shared, const float *shared_scale,
                          float *y, void *ws, size_t ws_bytes, cudaStream_t stream);
size_t moe_ffn_workspace_bytes(int T, int k, const moe_pool *pool, const moe_pool *shared);

/*
 * moe_expert_ffn for callers that cannot allocate device memory: code bound
 * to a device-memory plan fixed at start-up, plugin hosts that pass inputs
 * and outputs but offer no allocator, and paths where cudaMalloc/cudaFree are
 * not allowed because they can synchronise the device or fail under memory
 * pressure.  The pages have no counterpart to this call; it exists for
 * deployment.  Arguments and results are those of moe_expert_ffn, without
 * the workspace.
 *  - Scratch is one fixed array of 2 MiB in the library's device image, held
 *    on every device that loads the library until the process exits.  A
 *    shape whose moe_ffn_workspace_bytes() exceeds 2 MiB returns
 *    MOE_ERR_WORKSPACE before anything is enqueued.
 *  - Allocates nothing.  The first call on a device looks up the array's
 *    device address; make that first call before any stream capture.
 *  - Every call uses the same array and finds the previous call's contents
 *    there (the status word and tickets are cleared by each call).  Calls
 *    that overlap on the GPU (other streams, other host threads) race and
 *    corrupt each other's results: order them.
 *  - The status word lives in that array and is not reported; out-of-range
 *    or repeated ids are still skipped.
 */
moe_status moe_expert_ffn_noalloc(const void *xq, int T, const int32_t *ids, const float *weights, int k,
                                  const moe_pool *pool, const moe_pool *shared, const float *shared_scale,
                                  float *y, cudaStream_t stream);

/*
 * The whole layer: quantise (moe_quantize_q8K's rule), route (moe_route's
 * fixed-order logits, top-k and gating) and the routed + shared expert FFN
 * (moe_expert_ffn's arithmetic), for decode where the three steps sit back to
 * back.  For T <= 4 this is one launch, described below; larger batches run
 * the three calls in turn (their kernels keep more warps per SM busy once
 * every weight record is dotted with many tokens), inside the same workspace.
 * One persistent block per SM: every block quantises x and
 * computes the logits of its own router rows, every block reads all logits,
 * selects the same top-k and streams its share of the chosen experts' packed
 * weights with TMA bulk copies into a shared-memory ring.  Logits, h and the
 * per-slot o rows pass between blocks through the workspace as 8-byte words
 * that carry the value and a per-call epoch (launch counters kept in the
 * workspace), so readers poll the data itself.  Results equal those of the
 * three calls (same arithmetic and summation orders).
 *   hidden      : device fp32 [T][H]; w_router/rtype/router_bias/k/gating/
 *                 renormalize as in moe_route; pool/shared as in moe_expert_ffn
 *   shared_gate : device fp32 [H] or NULL, as in moe_route: the shared
 *                 expert's output is scaled per token by sigma(gate . hidden)
 *                 (requires shared; 16-byte aligned)
 *                 (shared: the same format as pool or Q8_0)
 *   y           : device fp32 [T][H] out
 *   ids_out, weights_out, logits_out, xq_out: optional outputs (NULL to skip)
 *   hidden, w_router, y and xq_out must be 16-byte aligned
 *   ws          : device workspace of moe_layer_workspace_bytes() bytes,
 *                 zero-filled before its first use and after any call that set
 *                 MOE_DEV_TIMEOUT; completed calls leave it ready for the next
 *                 call with the same T (zero-fill it again before a call with
 *                 another T: the layouts differ)
 *   flags       : (T <= 4) MOE_LAYER_OVERLAP_PREVIOUS lets this launch start while the
 *                 previous kernel in the stream is still running (programmatic
 *                 dependent launch): before that kernel has finished, the call
 *                 reads only weights, router and expert tables, so none of those
 *                 may be written by the previous kernel; hidden and everything
 *                 else are read only after it completes.
 * Every device-side wait is bounded (8e8 SM cycles, under a second): on timeout the call sets
 * MOE_DEV_TIMEOUT in the status word (moe_read_device_status) and returns.
 * Limits as moe_route and moe_expert_ffn; additionally the blocks must all be
 * resident at once (checked: MOE_ERR_UNSUPPORTED otherwise).
 * Errors: as moe_route and moe_expert_ffn (argument errors before any launch),
 * and MOE_ERR_UNSUPPORTED for a shared pool whose format is neither the
 * routed pool's nor Q8_0.
 */
#define MOE_LAYER_OVERLAP_PREVIOUS 0x1u
moe_status moe_layer_forward(const float *hidden, int T, const void *w_router, moe_qtype rtype,
                             const float *router_bias, int k, moe_gating gating, int renormalize,
                             const moe_pool *pool, const moe_pool *shared, const float *shared_gate, float *y,
                             int32_t *ids_out, float *weights_out, float *logits_out, void *xq_out,
                             void *ws, size_t ws_bytes, unsigned flags, cudaStream_t stream);
size_t moe_layer_workspace_bytes(int T, int k, const moe_pool *pool, const moe_pool *shared);

/*
 * Expert-parallel reduction (README "MoE resolve": each tier card computes
 * the slots of the experts it holds and the partial outputs are summed).  An
 * expert-parallel rank passes moe_expert_ffn / moe_layer_forward a pool whose
 * non-owned entries are NULL and gets a partial y; with the R partials side
 * by side (for example gathered from every rank):
 *   parts : device fp32 [R][n], rank r's partial at parts + r*n
 *   y     : device fp32 [n] out: y[i] = ((parts[0][i] + parts[1][i]) + ...)
 *           + parts[R-1][i], added in rank order, so the result does not
 *           depend on how the partials arrived
 * Both 16-byte aligned; n % 4 == 0; 1 <= R <= MOE_MAX_RANKS.
 * Errors: MOE_ERR_INVALID_ARG for R, n or a NULL or unaligned buffer.
 */
moe_status moe_sum_partials(const float *parts, int R, size_t n, float *y, cudaStream_t stream);

/*
 * Reads (and, if clear != 0, zeroes) the device status word at the start of
 * an FFN or layer workspace (both keep it in their first 4 bytes).
 * Synchronises `stream`.  *flags receives MOE_DEV_* bits.
 * Returns MOE_ERR_DEVICE_STATUS if any bit was set, MOE_OK otherwise.
 */
moe_status moe_read_device_status(void *ws, int clear, uint32_t *flags, cudaStream_t stream);

/*
 * Test hook: the exact int32 sub-block dots of one row of a packed matrix
 * with one q8 activation record, computed by the same device code the FFN
 * uses (the README's one-row GPU-vs-CPU arbiter idea).  Q4_K: 8 per
 * 256-block; Q2_K: 16; Q8_0 and MXFP4: 1 per 32-block.
 *   packed: device (moe_pack_weights); xq: device, one record of width cols;
 *   isums: device int32 out, cols/256*8, cols/256*16 or cols/32 entries.
 */
moe_status moe_debug_row_dots(const void *packed, moe_qtype qtype, int rows, int cols, int row,
                              const void *xq, int32_t *isums, cudaStream_t stream);

/*
 * Test hook: the bound, in SM clock cycles, on how long a moe_layer_forward
 * launch made after this call waits for another block's exchange words
 * (logits, h, o) before it gives up with MOE_DEV_TIMEOUT; 0 restores the
 * default (8e8 cycles).  A short bound makes the timeout path run without
 * any fault: the launch skips the remaining work, lets its own bulk copies
 * land (those waits keep the long bound) and returns.  Host-side setting of
 * this process, read when a layer launch is made (a captured graph keeps the
 * value it was captured with).  Errors: MOE_ERR_INVALID_ARG for cycles < 0.
 */
moe_status moe_debug_set_exchange_wait(long long cycles);

const char *moe_status_str(moe_status s);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H */
