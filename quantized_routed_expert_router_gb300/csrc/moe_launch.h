// moe_launch.h - internal launcher declarations shared by the translation
// units of the library (not part of the public C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

constexpr int MAXP = MOE_MAX_TOKENS * MOE_MAX_K;   // (token, slot) pairs per call
constexpr size_t kLayerMiscBytes = 4096;          // shared-memory block state of the fused kernel

struct RouteArgs {
    const float *hidden;
    const uint8_t *xq;
    const void *w;
    const float *bias;
    int32_t *ids;
    float *weights;
    float *logits_out;
    float *partial;      // ws: [T][E][nseg]
    unsigned *counter;   // ws
    const float *shared_gate;   // [H] or nullptr
    float *shared_scale;        // [T] out (with shared_gate)
    int T, H, E, k, nseg, gating, renorm;
};

struct FfnArgs {
    const uint8_t *xq;           // [T] records of width H
    const int32_t *ids;          // [T][k]
    const float *weights;        // [T][k]
    const moe_expert *experts;   // device [E]
    const moe_expert *shared;    // device [1] or nullptr
    const float *shared_scale;   // [T] weight of the shared expert, or nullptr (1)
    float *y;                    // [T][H]
    unsigned *status;            // ws
    unsigned *counters;          // ws [MAXP + 1]
    float *h_r;                  // ws [T*k][I]
    float *h_s;                  // ws [T][Is]
    uint8_t *hq_r;               // ws [T*k] records of width I
    uint8_t *hq_s;               // ws [T] records of width Is
    int T, k, H, I, Is, E;
    int qtype, sqtype;
};

// fused layer kernel: shared-memory carve-up (byte offsets) and arguments
struct Smem {
    uint32_t ring, bars, starts, router, table, xq, hq, lg, segv, ids, wts, grp, red, misc, total;
};

struct LayerArgs {
    const float *x;                 // [T][H]
    const void *w_router;
    const float *rbias;
    const moe_expert *experts;      // device [E]
    const moe_expert *shared;       // device [1] or nullptr
    const float *shared_gate;       // [H] gate vector of the shared expert, or nullptr
    float *y;                       // [T][H]
    int32_t *ids_out;               // optional outputs
    float *w_out;
    float *logits_out;
    uint8_t *xq_out;
    unsigned *status, *epoch;   // workspace: status word, per-block launch counters [G]
    // tagged words (value bits | epoch << 32): logits [T][E], h [T*k][I],
    // shared h [T][Is], o [T*k][H], shared o [T][H]
    unsigned long long *logits, *h_r, *h_s, *o_r, *o_s;
    int rtype, k, gating, renorm;
    int T, H, I, Is, E, P, NT;
    int table_in_smem;
    int hq_slots;                   // q8 records of requantised h the block can hold
    int bslots;                     // B-record partial-sum slots of the reduction buffer
    uint32_t ring_bytes;
    int lgra, lgrb, lgsa, lgsb;     // log2 of the records per ring item: routed A (gate + up runs),
                                    // routed B (down run), shared A, shared B
    long long wait_limit;           // cycles a wait for another block's exchange words may take
    int balpha;                     // weight of A bytes in the B-range balance, in quarters (0..4)
    size_t xrec, hrec;
    Smem sm;
};

struct LayerWs {
    size_t status, epoch, logits, h_r, h_s, o_r, o_s, total;
};
LayerWs layer_ws_layout(int T, int k, int H, int I, int Is, int E);
// plans shared memory and launches the fused layer kernel for the pool's formats
cudaError_t launch_layer(LayerArgs &a, int qtype, int sqtype, bool pdl, cudaStream_t s);
// the exchange-wait bound of later layer launches (0: the default)
void set_exchange_wait(long long cycles);

// every argument check of moe_expert_ffn except the workspace's (MOE_OK for
// T == 0 once the shapes are valid)
moe_status ffn_check_args(const void *xq, int T, const int32_t *ids, const float *weights, int k,
                          const moe_pool *pool, const moe_pool *shared, const float *shared_scale, const float *y);

// workspace layout of moe_expert_ffn (offsets in bytes)
struct FfnWs {
    size_t status, counters, h_r, h_s, hq_r, hq_s, total;
};
FfnWs ffn_ws_layout(int T, int k, int H, int I, int Is);

int num_sms();
int smem_optin();

cudaError_t launch_quantize(const float *x, int T, int n, uint8_t *xq, cudaStream_t s);
cudaError_t launch_route(const RouteArgs &a, int rtype, cudaStream_t s);
// per-token weight of the shared expert (shared_gate_weight) into scale[T]
cudaError_t launch_shared_gate(const float *hidden, int T, int H, const float *w, float *scale, cudaStream_t s);
cudaError_t launch_sum_partials(const float *parts, int R, size_t n, float *y, cudaStream_t s);
cudaError_t launch_pack(const uint8_t *src, int qtype, int rows, int cols, uint8_t *dst, cudaStream_t s);
cudaError_t launch_row_dots(const uint8_t *packed, int qtype, int cols, int row, const uint8_t *xq,
                            int32_t *out, cudaStream_t s);
// returns cudaErrorInvalidConfiguration if the shape needs more shared memory than a block has
cudaError_t launch_ffn(const FfnArgs &a, cudaStream_t s);

}  // namespace moe
