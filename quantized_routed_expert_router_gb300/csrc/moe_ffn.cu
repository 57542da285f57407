// moe_ffn.cu - routed + shared expert FFN for small-batch decode.
//
// pulsar README, "MoE resolve": per (token, slot) the chosen expert's
// gate/up/down run as integer dots on q8 activations with per-block rescale
// ("ds4's exact math"), experts are handed over as explicit device pointers
// with NULL meaning "not mine", and the per-slot outputs are summed; the
// shared expert is always on.  Two kernels, stream ordered:
//
//  gateup_kernel : work item = (unique expert, 32-row tile of I).  The block
//      streams that tile of W_gate and W_up once (128-bit coalesced loads,
//      one lane per row, the K dimension split over the 8 warps) and applies
//      it to every token that chose the expert; h = silu(g) * u goes to the
//      workspace.  The last block to finish an expert (atomic ticket)
//      requantises that expert's h rows to q8 for the down projection.
//  down_kernel   : one block per 32-row tile of H.  It streams that tile of
//      W_down for every chosen expert and the shared expert, then sums the
//      slots of each token in slot order (w * o), adds the shared expert last
//      and writes y.  No atomics touch y.
//
// Both kernels derive the expert grouping (unique experts in ascending id,
// the tokens of each) from ids in every block: a few hundred integer ops that
// spare a separate launch and a host round trip.
#include "moe_common.cuh"
#include "moe_launch.h"

namespace moe {

constexpr int FW = 8;                 // warps per block
constexpr int FT = FW * 32;           // threads per block

struct Group {
    int U;
    uint32_t bitmap[MOE_MAX_EXPERTS / 32];
    int wpre[MOE_MAX_EXPERTS / 32];
    int ue[MAXP];          // expert id of unique index u (ascending)
    uint32_t umask[MAXP];  // tokens that chose unique u
    int uoff[MAXP + 1];    // start of u's pairs in plist
    int plist[MAXP];       // pair ids (t*k + s) grouped by u, tokens ascending
    int pu[MAXP];          // unique index of pair p, -1: skipped
};

// Grouping of the (token, slot) pairs by expert; identical in every block.
__device__ void build_group(const FfnArgs &a, Group &g) {
    const int tid = threadIdx.x, P = a.T * a.k;
    const int nw = (a.E + 31) >> 5;
    for (int i = tid; i < MOE_MAX_EXPERTS / 32; i += FT) g.bitmap[i] = 0;
    for (int i = tid; i < MAXP; i += FT) g.umask[i] = 0;
    __syncthreads();
    for (int p = tid; p < P; p += FT) {
        const int t = p / a.k, s = p - t * a.k;
        const int e = a.ids[p];
        const bool valid = e >= 0 && e < a.E;
        bool dup = false;
        if (valid)
            for (int s2 = 0; s2 < s; ++s2) dup |= (a.ids[t * a.k + s2] == e);
        const bool owned = valid && a.experts[e].gate != nullptr;
        if (blockIdx.x == 0 && (!valid || dup)) atomicOr(a.status, (!valid ? MOE_DEV_BAD_ID : 0u) | (dup ? MOE_DEV_DUP_ID : 0u));
        const bool keep = valid && !dup && owned;
        g.pu[p] = keep ? e : -1;
        if (keep) atomicOr(&g.bitmap[e >> 5], 1u << (e & 31));
    }
    __syncthreads();
    if (tid < 32) {
        int carry = 0;
        for (int base = 0; base < nw; base += 32) {
            const int w = base + tid;
            const int c = w < nw ? __popc(g.bitmap[w]) : 0;
            int inc = c;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xFFFFFFFFu, inc, off);
                if (tid >= off) inc += o;
            }
            if (w < nw) g.wpre[w] = carry + inc - c;
            carry += __shfl_sync(0xFFFFFFFFu, inc, 31);
        }
        if (tid == 0) g.U = carry;
    }
    __syncthreads();
    for (int p = tid; p < P; p += FT) {
        const int e = g.pu[p];
        if (e < 0) continue;
        const int u = g.wpre[e >> 5] + __popc(g.bitmap[e >> 5] & ((1u << (e & 31)) - 1u));
        g.ue[u] = e;
        atomicOr(&g.umask[u], 1u << (p / a.k));
        g.pu[p] = u;
    }
    __syncthreads();
    if (tid < 32) {
        int carry = 0;
        for (int base = 0; base < g.U; base += 32) {
            const int u = base + tid;
            const int c = u < g.U ? __popc(g.umask[u]) : 0;
            int inc = c;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xFFFFFFFFu, inc, off);
                if (tid >= off) inc += o;
            }
            if (u < g.U) g.uoff[u] = carry + inc - c;
            carry += __shfl_sync(0xFFFFFFFFu, inc, 31);
        }
        if (tid == 0) g.uoff[g.U] = carry;
    }
    __syncthreads();
    for (int p = tid; p < P; p += FT) {
        const int u = g.pu[p];
        if (u < 0) continue;
        const int t = p / a.k;
        g.plist[g.uoff[u] + __popc(g.umask[u] & ((1u << t) - 1u))] = p;
    }
    __syncthreads();
}

// ------------------------------------------------------------ gate / up

template <class F, int NT>
__device__ void gateup_dots(const uint8_t *gtile, const uint8_t *utile, int H, int nt, const uint8_t *xs,
                            size_t xrec, float *red) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float ag[NT], au[NT];
#pragma unroll
    for (int i = 0; i < NT; ++i) { ag[i] = 0.f; au[i] = 0.f; }
    const int nrec = F::nrec(H);
    for (int r = warp; r < nrec; r += FW) {
        const int nb = F::rec_blocks(H, r);
        typename F::W wg, wu;
        F::load(wg, gtile + F::rec_off(H, r), nb, lane);
        F::load(wu, utile + F::rec_off(H, r), nb, lane);
        const int k0 = r * F::QK;
#pragma unroll
        for (int i = 0; i < NT; ++i) {
            if (i < nt) {
                const Act x = act_view(xs + i * xrec, H);
                int is[F::NSUB];
                F::isums(wg, x, k0, nb, is);
                ag[i] = __fadd_rn(ag[i], F::combine(wg, x, k0, nb, is));
                F::isums(wu, x, k0, nb, is);
                au[i] = __fadd_rn(au[i], F::combine(wu, x, k0, nb, is));
            }
        }
    }
#pragma unroll
    for (int i = 0; i < NT; ++i) {
        if (i < nt) {
            red[((warp * 2 + 0) * NT + i) * 32 + lane] = ag[i];
            red[((warp * 2 + 1) * NT + i) * 32 + lane] = au[i];
        }
    }
}

template <class F, int NT>
__device__ void gateup_finish(const moe_expert &ex, int rt, int nt, const int *dest, float *hbase, int Irows,
                              const float *red) {
    for (int idx = threadIdx.x; idx < nt * 32; idx += FT) {
        const int i = idx >> 5, l = idx & 31;
        float g = 0.f, u = 0.f;
#pragma unroll
        for (int w = 0; w < FW; ++w) {
            g += red[((w * 2 + 0) * NT + i) * 32 + l];
            u += red[((w * 2 + 1) * NT + i) * 32 + l];
        }
        const int row = rt * 32 + l;
        if (ex.b_gate) g += ex.b_gate[row];
        if (ex.b_up) u += ex.b_up[row];
        const float h = g / (1.f + expf(-g)) * u;
        hbase[(size_t)dest[i] * Irows + row] = h;
    }
}

// quantise rows of h (written by other blocks of this grid) into q8 records
__device__ void requant_rows(const float *hbase, uint8_t *hqbase, int Irows, int nt, const int *dest);

template <class F, class FS>
__global__ void __launch_bounds__(FT) gateup_kernel(FfnArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    Group &g = *reinterpret_cast<Group *>(smem);
    __shared__ int s_dest[MOE_MAX_TOKENS];
    __shared__ int s_tok[MOE_MAX_TOKENS];
    __shared__ unsigned s_last;
    const size_t xrec = q8_row_bytes(a.H);
    uint8_t *xs = smem + ((sizeof(Group) + 15) & ~(size_t)15);
    float *red = reinterpret_cast<float *>(xs + ((a.T * xrec + 15) & ~(size_t)15));

    build_group(a, g);
    const int tiles = a.I / 32;
    const int tiles_s = a.shared ? a.Is / 32 : 0;
    const int nitems = g.U * tiles + tiles_s;
    for (int it = blockIdx.x; it < nitems; it += gridDim.x) {
        const bool sh = it >= g.U * tiles;
        const int u = sh ? -1 : it / tiles;
        const int rt = sh ? it - g.U * tiles : it - u * tiles;
        int nt;
        if (!sh) {
            nt = g.uoff[u + 1] - g.uoff[u];
            if (threadIdx.x < nt) {
                const int p = g.plist[g.uoff[u] + threadIdx.x];
                s_dest[threadIdx.x] = p;
                s_tok[threadIdx.x] = p / a.k;
            }
        } else {
            nt = a.T;
            if (threadIdx.x < nt) { s_dest[threadIdx.x] = threadIdx.x; s_tok[threadIdx.x] = threadIdx.x; }
        }
        __syncthreads();
        // stage the q8 records of this item's tokens
        const int n16 = (int)(xrec / 16);
        for (int i = threadIdx.x; i < nt * n16; i += FT) {
            const int j = i / n16, c = i - j * n16;
            reinterpret_cast<uint4 *>(xs + j * xrec)[c] =
                reinterpret_cast<const uint4 *>(a.xq + (size_t)s_tok[j] * xrec)[c];
        }
        __syncthreads();
        const moe_expert &ex = sh ? a.shared[0] : a.experts[g.ue[u]];
        const int Irows = sh ? a.Is : a.I;
        float *hbase = sh ? a.h_s : a.h_r;
        if (!sh) {
            const size_t tb = F::tile_bytes(a.H);
            const uint8_t *gt = reinterpret_cast<const uint8_t *>(ex.gate) + rt * tb;
            const uint8_t *ut = reinterpret_cast<const uint8_t *>(ex.up) + rt * tb;
            if (nt <= 1) gateup_dots<F, 1>(gt, ut, a.H, nt, xs, xrec, red);
            else if (nt <= 4) gateup_dots<F, 4>(gt, ut, a.H, nt, xs, xrec, red);
            else gateup_dots<F, 16>(gt, ut, a.H, nt, xs, xrec, red);
        } else {
            const size_t tb = FS::tile_bytes(a.H);
            const uint8_t *gt = reinterpret_cast<const uint8_t *>(ex.gate) + rt * tb;
            const uint8_t *ut = reinterpret_cast<const uint8_t *>(ex.up) + rt * tb;
            if (nt <= 1) gateup_dots<FS, 1>(gt, ut, a.H, nt, xs, xrec, red);
            else if (nt <= 4) gateup_dots<FS, 4>(gt, ut, a.H, nt, xs, xrec, red);
            else gateup_dots<FS, 16>(gt, ut, a.H, nt, xs, xrec, red);
        }
        __syncthreads();
        if (nt <= 1) gateup_finish<F, 1>(ex, rt, nt, s_dest, hbase, Irows, red);
        else if (nt <= 4) gateup_finish<F, 4>(ex, rt, nt, s_dest, hbase, Irows, red);
        else gateup_finish<F, 16>(ex, rt, nt, s_dest, hbase, Irows, red);
        __threadfence();
        __syncthreads();
        // ticket: the block finishing the last tile of this expert requantises h
        unsigned *ctr = a.counters + (sh ? MAXP : u);
        if (threadIdx.x == 0) {
            __threadfence();
            const unsigned ntiles = sh ? (unsigned)tiles_s : (unsigned)tiles;
            s_last = (atomicAdd(ctr, 1u) == ntiles - 1u);
        }
        __syncthreads();
        if (s_last) {
            __threadfence();
            uint8_t *hq = sh ? a.hq_s : a.hq_r;
            requant_rows(hbase, hq, Irows, nt, s_dest);
            __syncthreads();
            if (threadIdx.x == 0) *ctr = 0u;
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------------ down

template <class F>
__device__ void down_item(const uint8_t *tile, int I, int r, int npairs, const int *pairs, int pair_base,
                          const uint8_t *hq, size_t hrec, float *part, int nrec_max) {
    const int lane = threadIdx.x & 31;
    const int nb = F::rec_blocks(I, r);
    typename F::W w;
    F::load(w, tile + F::rec_off(I, r), nb, lane);
    const int k0 = r * F::QK;
    for (int i = 0; i < npairs; ++i) {
        const int p = pairs ? pairs[i] : i;
        const Act h = act_view(hq + (size_t)p * hrec, I);
        int is[F::NSUB];
        F::isums(w, h, k0, nb, is);
        part[((size_t)(pair_base + p) * nrec_max + r) * 32 + lane] = F::combine(w, h, k0, nb, is);
    }
}

template <class F, class FS>
__global__ void __launch_bounds__(FT) down_kernel(FfnArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    Group &g = *reinterpret_cast<Group *>(smem);
    float *part = reinterpret_cast<float *>(smem + ((sizeof(Group) + 15) & ~(size_t)15));
    build_group(a, g);
    const int rt = blockIdx.x;
    const int warp = threadIdx.x >> 5;
    const int P = a.T * a.k;
    const int nr = F::nrec(a.I);
    const int ns = a.shared ? FS::nrec(a.Is) : 0;
    const int nrec_max = nr > ns ? nr : ns;
    const size_t hrec = q8_row_bytes(a.I), hrec_s = a.shared ? q8_row_bytes(a.Is) : 0;
    const int nitems = g.U * nr + ns;
    for (int it = warp; it < nitems; it += FW) {
        if (it < g.U * nr) {
            const int u = it / nr, r = it - u * nr;
            const moe_expert &ex = a.experts[g.ue[u]];
            const uint8_t *tile = reinterpret_cast<const uint8_t *>(ex.down) + (size_t)rt * F::tile_bytes(a.I);
            down_item<F>(tile, a.I, r, g.uoff[u + 1] - g.uoff[u], g.plist + g.uoff[u], 0, a.hq_r, hrec, part,
                         nrec_max);
        } else {
            const int r = it - g.U * nr;
            const uint8_t *tile = reinterpret_cast<const uint8_t *>(a.shared[0].down) + (size_t)rt * FS::tile_bytes(a.Is);
            down_item<FS>(tile, a.Is, r, a.T, nullptr, P, a.hq_s, hrec_s, part, nrec_max);
        }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < a.T * 32; idx += FT) {
        const int t = idx >> 5, l = idx & 31;
        const int row = rt * 32 + l;
        float y = 0.f;
        for (int s = 0; s < a.k; ++s) {
            const int p = t * a.k + s;
            const int u = g.pu[p];
            if (u < 0) continue;
            float o = 0.f;
            for (int r = 0; r < nr; ++r) o += part[((size_t)p * nrec_max + r) * 32 + l];
            const float *bd = a.experts[g.ue[u]].b_down;
            if (bd) o += bd[row];
            y += a.weights[p] * o;
        }
        if (a.shared) {
            float o = 0.f;
            for (int r = 0; r < ns; ++r) o += part[((size_t)(P + t) * nrec_max + r) * 32 + l];
            y += a.shared_scale ? a.shared_scale[t] * o : o;
        }
        a.y[(size_t)t * a.H + row] = y;
    }
}

// ------------------------------------------------------- requantisation

__device__ void requant_rows(const float *hbase, uint8_t *hqbase, int Irows, int nt, const int *dest) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int chunks = (Irows + 255) / 256;
    const size_t rec = q8_row_bytes(Irows);
    for (int w = warp; w < nt * chunks; w += FW) {
        const int i = w / chunks, c = w - i * chunks;
        quant_chunk256<true>(hbase + (size_t)dest[i] * Irows, Irows, 256 * c, hqbase + (size_t)dest[i] * rec,
                                 lane);
    }
}

// --------------------------------------------------------------- launch

FfnWs ffn_ws_layout(int T, int k, int H, int I, int Is) {
    (void)H;
    auto al = [](size_t v) { return (v + 255) & ~(size_t)255; };
    FfnWs w;
    w.status = 0;
    w.counters = 256;
    w.h_r = al(w.counters + sizeof(unsigned) * (MAXP + 1));
    w.h_s = al(w.h_r + sizeof(float) * (size_t)T * k * I);
    w.hq_r = al(w.h_s + sizeof(float) * (size_t)T * (Is > 0 ? Is : 0));
    w.hq_s = al(w.hq_r + (size_t)T * k * q8_row_bytes(I));
    w.total = al(w.hq_s + (Is > 0 ? (size_t)T * q8_row_bytes(Is) : 0));
    return w;
}

template <class F, class FS>
static cudaError_t launch_ffn_t(const FfnArgs &a, cudaStream_t s) {
    const size_t gsz = (sizeof(Group) + 15) & ~(size_t)15;
    const size_t xrec = q8_row_bytes(a.H);
    const int ntmax = a.T <= 1 ? 1 : (a.T <= 4 ? 4 : 16);
    const size_t smem_gu = gsz + ((a.T * xrec + 15) & ~(size_t)15) + (size_t)FW * 2 * ntmax * 32 * 4;
    const int nr = F::nrec(a.I), ns = a.shared ? FS::nrec(a.Is) : 0;
    const int nrec_max = nr > ns ? nr : ns;
    const size_t smem_dn = gsz + (size_t)(a.T * a.k + a.T) * nrec_max * 32 * 4;
    if (smem_gu > (size_t)smem_optin() || smem_dn > (size_t)smem_optin()) return cudaErrorInvalidConfiguration;
    cudaError_t err = ensure_smem<gateup_kernel<F, FS>>(smem_gu);
    if (err != cudaSuccess) return err;
    err = ensure_smem<down_kernel<F, FS>>(smem_dn);
    if (err != cudaSuccess) return err;
    const int umax = a.T * a.k < a.E ? a.T * a.k : a.E;
    const long long items = (long long)umax * (a.I / 32) + (a.shared ? a.Is / 32 : 0);
    long long grid = 2LL * num_sms();
    if (items < grid) grid = items;
    if (grid < 1) grid = 1;
    gateup_kernel<F, FS><<<(unsigned)grid, FT, smem_gu, s>>>(a);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    down_kernel<F, FS><<<a.H / 32, FT, smem_dn, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_ffn(const FfnArgs &a, cudaStream_t s) {
    const int q = a.qtype, sq = a.shared ? a.sqtype : a.qtype;
    if (q == MOE_Q8_0 && sq == MOE_Q8_0) return launch_ffn_t<FQ80, FQ80>(a, s);
    if (q == MOE_Q4_K && sq == MOE_Q4_K) return launch_ffn_t<FQ4K, FQ4K>(a, s);
    if (q == MOE_Q4_K && sq == MOE_Q8_0) return launch_ffn_t<FQ4K, FQ80>(a, s);
    if (q == MOE_Q2_K && sq == MOE_Q2_K) return launch_ffn_t<FQ2K, FQ2K>(a, s);
    if (q == MOE_Q2_K && sq == MOE_Q8_0) return launch_ffn_t<FQ2K, FQ80>(a, s);
    if (q == MOE_MXFP4 && sq == MOE_MXFP4) return launch_ffn_t<FMX4, FMX4>(a, s);
    if (q == MOE_MXFP4 && sq == MOE_Q8_0) return launch_ffn_t<FMX4, FQ80>(a, s);
    if (q == MOE_Q6_K && sq == MOE_Q6_K) return launch_ffn_t<FQ6K, FQ6K>(a, s);
    if (q == MOE_Q6_K && sq == MOE_Q8_0) return launch_ffn_t<FQ6K, FQ80>(a, s);
    if (q == MOE_Q3_K && sq == MOE_Q3_K) return launch_ffn_t<FQ3K, FQ3K>(a, s);
    if (q == MOE_Q3_K && sq == MOE_Q8_0) return launch_ffn_t<FQ3K, FQ80>(a, s);
    return cudaErrorNotSupported;
}

}  // namespace moe
