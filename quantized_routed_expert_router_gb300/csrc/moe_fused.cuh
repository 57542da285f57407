// moe_fused.cuh - one persistent launch per MoE layer: quantise, route, expert
// FFN (pulsar README, "MoE resolve" passage: router, integer dots on q8
// activations with per-block rescale, explicit expert pointers with NULL =
// "not mine", per-slot sum, shared expert always on).
//
// Grid: one block per SM, all co-resident; 8 consumer warps + 1 producer warp.
//
//  1. Before the previous kernel in the stream has finished (programmatic
//     dependent launch), the producer bulk-copies input-independent bytes
//     into shared memory: this block's router rows, the expert pointer table
//     and the first shared-expert gate/up records.
//  2. After griddepcontrol.wait every block quantises x itself (no exchange),
//     computes logits for its router rows in the fixed summation order and
//     publishes them; while the other blocks finish, it runs its share of the
//     shared expert's gate/up.
//  3. A release/acquire ticket over all blocks makes every logit visible;
//     each block selects the same top-k, groups the (token, slot) pairs by
//     expert and derives the same work plan:
//       A units = (expert, 32-row tile of I): gate + up records,
//       B units = (expert, 32-row tile of H): down records.
//     A units are dealt out in a snake over blocks; B units are contiguous
//     ranges sized so every block streams about the same number of bytes.
//  4. The producer streams each unit's records (TMA bulk copies, complete_tx
//     mbarriers) through a byte ring; consumer warp r % 8 takes record r of a
//     unit, so every sum has a fixed order whatever the batch.
//  5. An A unit ends with h = silu(g) * u rows in global scratch and a
//     release on its expert's ticket; a B unit first waits for the tickets of
//     its expert, requantises that expert's h locally, and ends with o rows
//     plus a ticket on its row tile; the block that completes a row tile sums
//     the slots of each token in slot order (shared expert last) into y.
//  Every wait is bounded by the global timer; a timeout sets MOE_DEV_TIMEOUT,
//  drains this block's copies in flight and returns.
#pragma once

#include "moe_common.cuh"
#include "moe_launch.h"

namespace moe {

constexpr int LW = 8;                  // consumer warps
constexpr int LT = (LW + 1) * 32;      // threads per block (with the producer warp)
constexpr int NBAR = 32;               // ring items in flight (barrier slots)
constexpr unsigned long long WAIT_NS = 400ull * 1000ull * 1000ull;   // 0.4 s per wait

// ------------------------------------------------------------ PTX helpers

__device__ __forceinline__ unsigned long long gtimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_arm(uint64_t *b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(b)) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t *b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(saddr(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
// bounded wait on an mbarrier phase; false on timeout
__device__ __forceinline__ bool mbar_wait(uint64_t *b, uint32_t parity) {
    if (mbar_test(b, parity)) return true;
    const unsigned long long t0 = gtimer();
    while (!mbar_test(b, parity))
        if (gtimer() - t0 > WAIT_NS) return false;
    return true;
}
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            saddr(dst)),
        "l"(src), "r"(bytes), "r"(saddr(bar))
        : "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void red_release(unsigned *p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned atom_acqrel(unsigned *p, unsigned v) {
    unsigned o;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(o) : "l"(p), "r"(v) : "memory");
    return o;
}
__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// bounded spin until *p >= target; false on timeout
__device__ __forceinline__ bool spin_geq(const unsigned *p, unsigned target) {
    if (ld_acquire(p) >= target) return true;
    const unsigned long long t0 = gtimer();
    while (ld_acquire(p) < target)
        if (gtimer() - t0 > WAIT_NS) return false;
    return true;
}
__device__ __forceinline__ void cbar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }   // consumers only

// ------------------------------------------------------------- block state

struct Misc {
    volatile int abort;
    int U, n_sa, n_ra, nA, n_sb, n_rb, nB, jb0, jb1;
    int tilesI, tilesIs, tilesH;
    int hq_key;          // expert whose h is requantised in hq (-1 none, MAXP shared)
    int nc;              // contributions per row tile of y
    uint32_t bitmap[MOE_MAX_EXPERTS / 32];
    int wpre[MOE_MAX_EXPERTS / 32];
    double bsum[LW];
};

// Snake over blocks: unit j -> block, pass by pass, reversing every other pass.
__device__ __forceinline__ int snake_unit(int pass, int c, int G) {
    return pass * G + ((pass & 1) ? (G - 1 - c) : c);
}

template <class F, class FS, int NT>
struct LayerKernel {
    const LayerArgs &a;
    unsigned char *sm;
    Smem o;
    Misc *m;
    int c, G, warp, lane;

    __device__ LayerKernel(const LayerArgs &args, unsigned char *smem) : a(args), sm(smem), o(args.sm) {
        m = reinterpret_cast<Misc *>(sm + o.misc);
        c = blockIdx.x;
        G = gridDim.x;
        warp = threadIdx.x >> 5;
        lane = threadIdx.x & 31;
    }

    __device__ uint64_t *full_bar(int i) { return reinterpret_cast<uint64_t *>(sm + o.bars) + (i % NBAR); }
    __device__ uint64_t *empty_bar(int i) { return reinterpret_cast<uint64_t *>(sm + o.bars) + NBAR + (i % NBAR); }
    __device__ uint64_t *fixed_bar() { return reinterpret_cast<uint64_t *>(sm + o.bars) + 2 * NBAR; }
    __device__ uint32_t *starts() { return reinterpret_cast<uint32_t *>(sm + o.starts); }
    __device__ const moe_expert *table() {
        return a.table_in_smem ? reinterpret_cast<const moe_expert *>(sm + o.table) : a.experts;
    }
    __device__ int *ue() { return reinterpret_cast<int *>(sm + o.grp); }
    __device__ uint32_t *umask() { return reinterpret_cast<uint32_t *>(ue() + a.P); }
    __device__ int *uoff() { return reinterpret_cast<int *>(umask() + a.P); }
    __device__ int *plist() { return uoff() + a.P + 1; }
    __device__ int *pu() { return plist() + a.P; }
    __device__ int *ids() { return reinterpret_cast<int *>(sm + o.ids); }
    __device__ float *wts() { return reinterpret_cast<float *>(sm + o.wts); }
    __device__ uint8_t *xq(int t) { return sm + o.xq + (size_t)t * a.xrec; }
    __device__ uint8_t *hq(int i) { return sm + o.hq + (size_t)i * a.hrec; }

    __device__ void fail() {
        m->abort = 1;
        atomicOr(a.status, MOE_DEV_TIMEOUT);
    }

    // ------------------------------------------------------------ units
    // kind: 0 shared A, 1 routed A, 2 shared B, 3 routed B
    struct Unit {
        int kind, u, rt, nrec, nt;
        const uint8_t *g, *up, *d;   // tile bases (A: gate/up, B: down)
        const moe_expert *ex;
    };

    __device__ void unit_of(int j, Unit &U) {
        const moe_expert *T = table();
        if (j < m->n_sa) {
            U.kind = 0; U.u = MAXP; U.rt = j;
            U.ex = a.shared;
            U.nrec = FS::nrec(a.H);
            U.nt = a.T;
            const size_t tb = FS::tile_bytes(a.H);
            U.g = (const uint8_t *)a.shared->gate + (size_t)U.rt * tb;
            U.up = (const uint8_t *)a.shared->up + (size_t)U.rt * tb;
        } else if (j < m->nA) {
            const int q = j - m->n_sa;
            U.kind = 1; U.u = q / m->tilesI; U.rt = q - U.u * m->tilesI;
            U.ex = T + ue()[U.u];
            U.nrec = F::nrec(a.H);
            U.nt = uoff()[U.u + 1] - uoff()[U.u];
            const size_t tb = F::tile_bytes(a.H);
            U.g = (const uint8_t *)U.ex->gate + (size_t)U.rt * tb;
            U.up = (const uint8_t *)U.ex->up + (size_t)U.rt * tb;
        } else if (j < m->nA + m->n_sb) {
            U.kind = 2; U.u = MAXP; U.rt = j - m->nA;
            U.ex = a.shared;
            U.nrec = FS::nrec(a.Is);
            U.nt = a.T;
            U.d = (const uint8_t *)a.shared->down + (size_t)U.rt * FS::tile_bytes(a.Is);
        } else {
            const int q = j - m->nA - m->n_sb;
            U.kind = 3; U.u = q / m->tilesH; U.rt = q - U.u * m->tilesH;
            U.ex = T + ue()[U.u];
            U.nrec = F::nrec(a.I);
            U.nt = uoff()[U.u + 1] - uoff()[U.u];
            U.d = (const uint8_t *)U.ex->down + (size_t)U.rt * F::tile_bytes(a.I);
        }
    }

    __device__ uint32_t item_bytes(const Unit &U, int r) {
        switch (U.kind) {
            case 0: return 2 * FS::rec_bytes(a.H, r);
            case 1: return 2 * F::rec_bytes(a.H, r);
            case 2: return FS::rec_bytes(a.Is, r);
            default: return F::rec_bytes(a.I, r);
        }
    }

    // -------------------------------------------------------- producer
    struct Ring {
        uint32_t head;
        int issued, tail;   // items issued so far; oldest item not yet reclaimed
    };

    __device__ bool reclaim_oldest(Ring &R) {
        const int t = R.tail;
        if (!mbar_wait(empty_bar(t), (uint32_t)((t / NBAR) & 1))) return false;
        ++R.tail;
        return true;
    }

    // place an item of `bytes` bytes; returns false on timeout.  In-flight
    // items occupy [start(tail), head) in ring order (possibly wrapped).
    __device__ bool ring_place(Ring &R, uint32_t bytes, uint32_t &start) {
        for (;;) {
            if (R.issued - R.tail >= NBAR) {
                if (!reclaim_oldest(R)) return false;
                continue;
            }
            if (R.issued == R.tail) { R.head = 0; start = 0; return true; }
            const uint32_t ts = starts()[R.tail % NBAR];
            if (R.head > ts) {
                if (a.ring_bytes - R.head >= bytes) { start = R.head; return true; }
                if (ts >= bytes) { start = 0; return true; }
            } else if (R.head < ts) {
                if (ts - R.head >= bytes) { start = R.head; return true; }
            }
            if (!reclaim_oldest(R)) return false;
        }
    }

    __device__ bool issue(Ring &R, const Unit &U, int r) {
        const uint32_t bytes = item_bytes(U, r);
        uint32_t start;
        if (!ring_place(R, bytes, start)) return false;
        const int i = R.issued;
        starts()[i % NBAR] = start;
        uint8_t *dst = sm + o.ring + start;
        uint64_t *fb = full_bar(i);
        mbar_arm(fb, bytes);
        if (U.kind == 0 || U.kind == 1) {
            const uint32_t half = bytes / 2;
            const size_t off = U.kind == 0 ? FS::rec_off(a.H, r) : F::rec_off(a.H, r);
            bulk_g2s(dst, U.g + off, half, fb);
            bulk_g2s(dst + half, U.up + off, half, fb);
        } else {
            const size_t off = U.kind == 2 ? FS::rec_off(a.Is, r) : F::rec_off(a.I, r);
            bulk_g2s(dst, U.d + off, bytes, fb);
        }
        R.head = start + bytes;
        ++R.issued;
        return true;
    }

    __device__ bool issue_unit(Ring &R, int j) {
        Unit U;
        unit_of(j, U);
        for (int r = 0; r < U.nrec; ++r) {
            if (m->abort) return false;
            if (!issue(R, U, r)) { fail(); return false; }
        }
        return true;
    }

    // ------------------------------------------------------- consumers
    // one record of a unit: wait for it, pull it into registers, free the slot
    // wait for item i (a record, or a gate+up record pair) to land in the ring
    __device__ const uint8_t *wait_item(int i) {
        if (m->abort) return nullptr;
        if (!mbar_wait(full_bar(i), (uint32_t)((i / NBAR) & 1))) { fail(); return nullptr; }
        return sm + o.ring + starts()[i % NBAR];
    }
    __device__ void free_item(int i) {
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(i));
    }

    // A unit: g and u partial sums of this warp's records, then h rows
    template <class FF>
    __device__ void run_A(const Unit &U, int &item, int &rbuf) {
        float ag[NT], au[NT];
#pragma unroll
        for (int i = 0; i < NT; ++i) { ag[i] = 0.f; au[i] = 0.f; }
        int tok[NT];
#pragma unroll
        for (int i = 0; i < NT; ++i)
            tok[i] = (i < U.nt) ? (U.kind == 0 ? i : plist()[uoff()[U.u] + i] / a.k) : 0;
        for (int r = 0; r < U.nrec; ++r, ++item) {
            if ((r & (LW - 1)) != warp) continue;
            const uint8_t *rec = wait_item(item);
            if (!rec) continue;
            const int nb = FF::rec_blocks(a.H, r);
            const int k0 = r * FF::QK;
            {   // gate record, then up record: one record's registers live at a time
                typename FF::W w;
                FF::load_s(w, rec, nb, lane);
#pragma unroll
                for (int i = 0; i < NT; ++i) {
                    if (i < U.nt) {
                        const Act x = act_view(xq(tok[i]), a.H);
                        int is[FF::NSUB];
                        FF::isums(w, x, k0, nb, is);
                        ag[i] += FF::combine(w, x, k0, nb, is);
                    }
                }
            }
            {
                typename FF::W w;
                FF::load_s(w, rec + FF::rec_bytes(a.H, r), nb, lane);
                free_item(item);
#pragma unroll
                for (int i = 0; i < NT; ++i) {
                    if (i < U.nt) {
                        const Act x = act_view(xq(tok[i]), a.H);
                        int is[FF::NSUB];
                        FF::isums(w, x, k0, nb, is);
                        au[i] += FF::combine(w, x, k0, nb, is);
                    }
                }
            }
        }
        float *red = reinterpret_cast<float *>(sm + o.red) + rbuf * (LW * 2 * NT * 32);
#pragma unroll
        for (int i = 0; i < NT; ++i) {
            red[((warp * 2 + 0) * NT + i) * 32 + lane] = ag[i];
            red[((warp * 2 + 1) * NT + i) * 32 + lane] = au[i];
        }
        cbar();
        if (warp == 0) {
            const int row = U.rt * 32 + lane;
            const int Irows = U.kind == 0 ? a.Is : a.I;
            float *hb = U.kind == 0 ? a.h_s : a.h_r;
            for (int i = 0; i < U.nt && i < NT; ++i) {
                float g = 0.f, uu = 0.f;
#pragma unroll
                for (int w = 0; w < LW; ++w) {
                    g += red[((w * 2 + 0) * NT + i) * 32 + lane];
                    uu += red[((w * 2 + 1) * NT + i) * 32 + lane];
                }
                if (U.ex->b_gate) g += U.ex->b_gate[row];
                if (U.ex->b_up) uu += U.ex->b_up[row];
                const float h = g / (1.f + expf(-g)) * uu;
                const int dest = U.kind == 0 ? i : plist()[uoff()[U.u] + i];
                hb[(size_t)dest * Irows + row] = h;
            }
            __threadfence();
            __syncwarp();
            if (lane == 0) red_release(a.hctr + U.u, 1u);
        }
        rbuf ^= 1;
    }

    // requantise the h rows of unit U's expert into the block's hq records
    __device__ bool load_hq(const Unit &U) {
        const int key = U.kind == 2 ? MAXP : U.u;
        if (m->hq_key == key) return true;
        const int Irows = U.kind == 2 ? a.Is : a.I;
        const unsigned need = (unsigned)(U.kind == 2 ? m->tilesIs : m->tilesI);
        cbar();   // everyone is done with the previous hq
        if (threadIdx.x == 0 && !m->abort)
            if (!spin_geq(a.hctr + key, need)) fail();
        cbar();
        const float *hb = U.kind == 2 ? a.h_s : a.h_r;
        const int chunks = (Irows + 255) / 256;
        const bool ok = !m->abort;
        for (int w = warp; ok && w < U.nt * chunks; w += LW) {
            const int i = w / chunks, ch = w - i * chunks;
            const int dest = U.kind == 2 ? i : plist()[uoff()[U.u] + i];
            quant_chunk256<true>(hb + (size_t)dest * Irows, Irows, 256 * ch, hq(i), lane);
        }
        if (threadIdx.x == 0) m->hq_key = key;
        cbar();
        return true;
    }

    // B unit: o rows of the down projection, then (last block of the tile) y
    template <class FF>
    __device__ void run_B(const Unit &U, int &item, int &rbuf) {
        const int Irows = U.kind == 2 ? a.Is : a.I;
        float ao[NT];
#pragma unroll
        for (int i = 0; i < NT; ++i) ao[i] = 0.f;
        for (int r = 0; r < U.nrec; ++r, ++item) {
            if ((r & (LW - 1)) != warp) continue;
            const uint8_t *rec = wait_item(item);
            if (!rec) continue;
            typename FF::W wd;
            const int nb = FF::rec_blocks(Irows, r);
            FF::load_s(wd, rec, nb, lane);
            free_item(item);
            const int k0 = r * FF::QK;
#pragma unroll
            for (int i = 0; i < NT; ++i) {
                if (i < U.nt) {
                    const Act h = act_view(hq(i), Irows);
                    int is[FF::NSUB];
                    FF::isums(wd, h, k0, nb, is);
                    ao[i] += FF::combine(wd, h, k0, nb, is);
                }
            }
        }
        float *red = reinterpret_cast<float *>(sm + o.red) + rbuf * (LW * 2 * NT * 32);
#pragma unroll
        for (int i = 0; i < NT; ++i) red[(warp * NT + i) * 32 + lane] = ao[i];
        cbar();
        if (warp == 0) {
            const int row = U.rt * 32 + lane;
            for (int i = 0; i < U.nt && i < NT; ++i) {
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < LW; ++w) v += red[(w * NT + i) * 32 + lane];
                if (U.kind == 3) {
                    if (U.ex->b_down) v += U.ex->b_down[row];
                    const int p = plist()[uoff()[U.u] + i];
                    a.o_r[(size_t)p * a.H + row] = v;
                } else {
                    a.o_s[(size_t)i * a.H + row] = v;
                }
            }
            __threadfence();
            __syncwarp();
            unsigned old = 0;
            if (lane == 0) old = atom_acqrel(a.yticket + U.rt, 1u);
            old = __shfl_sync(0xFFFFFFFFu, old, 0);
            if (old == (unsigned)m->nc - 1u) {
                __syncwarp();
                write_y(U.rt);
                if (lane == 0) a.yticket[U.rt] = 0u;
            }
        }
        rbuf ^= 1;
    }

    // y rows of one 32-row tile: slots in slot order, shared expert last
    __device__ void write_y(int rt) {
        const int row = rt * 32 + lane;
        for (int t = 0; t < a.T; ++t) {
            float y = 0.f;
            for (int s = 0; s < a.k; ++s) {
                const int p = t * a.k + s;
                if (pu()[p] < 0) continue;
                y += wts()[p] * __ldcg(a.o_r + (size_t)p * a.H + row);
            }
            if (a.shared) y += __ldcg(a.o_s + (size_t)t * a.H + row);
            a.y[(size_t)t * a.H + row] = y;
        }
    }

    // ------------------------------------------------------ phases
    __device__ void init() {
        if (threadIdx.x == 0) {
            for (int i = 0; i < 2 * NBAR; ++i) mbar_init(reinterpret_cast<uint64_t *>(sm + o.bars) + i, 1);
            mbar_init(fixed_bar(), 1);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            m->abort = 0;
            m->hq_key = -1;
        }
        __syncthreads();
    }

    // router rows of this block (balanced contiguous range)
    __device__ void router_range(int &e0, int &e1) {
        e0 = (int)(((long long)c * a.E) / G);
        e1 = (int)(((long long)(c + 1) * a.E) / G);
    }

    __device__ void quantise_x() {
        const int chunks = (a.H + 255) / 256;
        for (int w = warp; w < a.T * chunks; w += LW) {
            const int t = w / chunks, ch = w - t * chunks;
            quant_chunk256<false>(a.x + (size_t)t * a.H, a.H, 256 * ch, xq(t), lane);
        }
    }

    __device__ void router_logits() {
        int e0, e1;
        router_range(e0, e1);
        const int nr = e1 - e0;
        const int nseg = (a.H + 1023) / 1024;
        float *segv = reinterpret_cast<float *>(sm + o.segv);   // [row][seg][T]
        if (nr > 0 || a.table_in_smem) {
            if (!mbar_wait(fixed_bar(), 0)) fail();
        }
        cbar();
        if (!m->abort) {
            for (int it = warp; it < nr * nseg; it += LW) {
                const int r = it / nseg, s = it - r * nseg;
                const int s0 = s * 1024, seglen = min(1024, a.H - s0);
                if (a.rtype == MOE_F32) {
                    const float *wr = reinterpret_cast<const float *>(sm + o.router) + (size_t)r * a.H + s0;
                    float4 wv[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int cc = lane + 32 * j;
                        if (4 * cc < seglen) {
                            const uint4 u = lds_u4(wr + 4 * cc);
                            wv[j] = make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z),
                                                __uint_as_float(u.w));
                        }
                    }
                    for (int t = 0; t < a.T; ++t) {
                        const float *xt = a.x + (size_t)t * a.H + s0;
                        float v = 0.f;
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int cc = lane + 32 * j;
                            if (4 * cc < seglen) {
                                const float4 xv = *reinterpret_cast<const float4 *>(xt + 4 * cc);
                                v = __fmaf_rn(wv[j].x, xv.x, v);
                                v = __fmaf_rn(wv[j].y, xv.y, v);
                                v = __fmaf_rn(wv[j].z, xv.z, v);
                                v = __fmaf_rn(wv[j].w, xv.w, v);
                            }
                        }
#pragma unroll
                        for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
                        if (lane == 0) segv[(r * nseg + s) * a.T + t] = v;
                    }
                } else {
                    const int nblk = a.H / 32;
                    const int b = s * 32 + lane;
                    const bool has = b < nblk;
                    const uint8_t *row = sm + o.router + (size_t)r * (nblk * 34);
                    uint32_t qw[8];
                    float dw = 0.f;
                    if (has) {
                        const uint16_t *hp = reinterpret_cast<const uint16_t *>(row + 34 * b);
                        dw = h2f(hp[0]);
#pragma unroll
                        for (int mm = 0; mm < 8; ++mm) qw[mm] = (uint32_t)hp[1 + 2 * mm] | ((uint32_t)hp[2 + 2 * mm] << 16);
                    }
                    for (int t = 0; t < a.T; ++t) {
                        float v = 0.f;
                        if (has) {
                            const Act x = act_view(xq(t), a.H);
                            const int4 x0 = lds128(x.q + 32 * b), x1 = lds128(x.q + 32 * b + 16);
                            int acc = 0;
                            acc = dp4a(qw[0], (uint32_t)x0.x, acc);
                            acc = dp4a(qw[1], (uint32_t)x0.y, acc);
                            acc = dp4a(qw[2], (uint32_t)x0.z, acc);
                            acc = dp4a(qw[3], (uint32_t)x0.w, acc);
                            acc = dp4a(qw[4], (uint32_t)x1.x, acc);
                            acc = dp4a(qw[5], (uint32_t)x1.y, acc);
                            acc = dp4a(qw[6], (uint32_t)x1.z, acc);
                            acc = dp4a(qw[7], (uint32_t)x1.w, acc);
                            v = __fmul_rn(__fmul_rn(dw, x.d[(32 * b) >> x.lgB]), (float)acc);
                        }
#pragma unroll
                        for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
                        if (lane == 0) segv[(r * nseg + s) * a.T + t] = v;
                    }
                }
            }
        }
        cbar();
        for (int it = threadIdx.x; it < nr * a.T; it += LW * 32) {
            const int r = it / a.T, t = it - r * a.T;
            float l = segv[(r * nseg) * a.T + t];
            for (int s = 1; s < nseg; ++s) l = __fadd_rn(l, segv[(r * nseg + s) * a.T + t]);
            if (a.rbias) l = __fadd_rn(l, a.rbias[e0 + r]);
            a.logits[(size_t)t * a.E + e0 + r] = l;
        }
        __threadfence();
        cbar();
        if (threadIdx.x == 0) red_release(a.route_ctr, 1u);
    }

    __device__ void topk_and_group() {
        if (threadIdx.x == 0 && !m->abort)
            if (!spin_geq(a.route_ctr, (unsigned)G)) fail();
        cbar();
        float *lgs = reinterpret_cast<float *>(sm + o.lg);
        for (int i = threadIdx.x; i < a.T * a.E; i += LW * 32) lgs[i] = __ldcg(a.logits + i);
        cbar();
        if (c == 0 && a.logits_out)
            for (int i = threadIdx.x; i < a.T * a.E; i += LW * 32) a.logits_out[i] = lgs[i];
        for (int t = warp; t < a.T; t += LW) {
            const float *lg = lgs + (size_t)t * a.E;
            uint32_t taken = 0;
            float mysel = 0.f;
            for (int s = 0; s < a.k; ++s) {
                float bv = 0.f;
                int bi = 0x7FFFFFFF;
                for (int j = 0, e = lane; e < a.E; ++j, e += 32) {
                    if (taken & (1u << j)) continue;
                    const float v = lg[e];
                    if (bi == 0x7FFFFFFF || v > bv) { bv = v; bi = e; }
                }
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) {
                    const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
                    const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, off);
                    if (oi != 0x7FFFFFFF && (bi == 0x7FFFFFFF || ov > bv || (ov == bv && oi < bi))) { bv = ov; bi = oi; }
                }
                if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
                if (lane == s) mysel = bv;
                if (lane == 0) ids()[t * a.k + s] = bi;
            }
            const float l0 = __shfl_sync(0xFFFFFFFFu, mysel, 0);
            float w;
            if (a.gating == MOE_GATE_SOFTMAX) {
                w = lane < a.k ? expf(mysel - l0) : 0.f;
                float z;
                if (a.renorm) {
                    z = w;
                } else {
                    z = 0.f;
                    for (int e = lane; e < a.E; e += 32) z += expf(lg[e] - l0);
                }
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) z = __fadd_rn(z, __shfl_xor_sync(0xFFFFFFFFu, z, off));
                w = w / z;
            } else {
                w = lane < a.k ? 1.f / (1.f + expf(-mysel)) : 0.f;
                if (a.renorm) {
                    float z = w;
#pragma unroll
                    for (int off = 16; off >= 1; off >>= 1) z = __fadd_rn(z, __shfl_xor_sync(0xFFFFFFFFu, z, off));
                    w = w / z;
                }
            }
            if (lane < a.k) wts()[t * a.k + lane] = w;
        }
        cbar();
        if (c == 0) {
            for (int i = threadIdx.x; i < a.P; i += LW * 32) {
                if (a.ids_out) a.ids_out[i] = ids()[i];
                if (a.w_out) a.w_out[i] = wts()[i];
            }
        }
        group();
    }

    // (token, slot) pairs grouped by owned expert, ascending ids, tokens ascending
    __device__ void group() {
        const int tid = threadIdx.x, P = a.P;
        const int nw = (a.E + 31) >> 5;
        for (int i = tid; i < MOE_MAX_EXPERTS / 32; i += LW * 32) m->bitmap[i] = 0;
        for (int i = tid; i < P; i += LW * 32) umask()[i] = 0;
        cbar();
        const moe_expert *T = table();
        for (int p = tid; p < P; p += LW * 32) {
            const int t = p / a.k, s = p - t * a.k;
            const int e = ids()[p];
            bool dup = false;
            for (int s2 = 0; s2 < s; ++s2) dup |= (ids()[t * a.k + s2] == e);
            const bool keep = !dup && T[e].gate != nullptr;
            pu()[p] = keep ? e : -1;
            if (keep) atomicOr(&m->bitmap[e >> 5], 1u << (e & 31));
        }
        cbar();
        if (tid < 32) {
            int carry = 0;
            for (int base = 0; base < nw; base += 32) {
                const int w = base + tid;
                const int cnt = w < nw ? __popc(m->bitmap[w]) : 0;
                int inc = cnt;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int v = __shfl_up_sync(0xFFFFFFFFu, inc, off);
                    if (tid >= off) inc += v;
                }
                if (w < nw) m->wpre[w] = carry + inc - cnt;
                carry += __shfl_sync(0xFFFFFFFFu, inc, 31);
            }
            if (tid == 0) m->U = carry;
        }
        cbar();
        for (int p = tid; p < P; p += LW * 32) {
            const int e = pu()[p];
            if (e < 0) continue;
            const int u = m->wpre[e >> 5] + __popc(m->bitmap[e >> 5] & ((1u << (e & 31)) - 1u));
            ue()[u] = e;
            atomicOr(&umask()[u], 1u << (p / a.k));
            pu()[p] = u;
        }
        cbar();
        if (tid < 32) {
            int carry = 0;
            for (int base = 0; base < m->U; base += 32) {
                const int u = base + tid;
                const int cnt = u < m->U ? __popc(umask()[u]) : 0;
                int inc = cnt;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int v = __shfl_up_sync(0xFFFFFFFFu, inc, off);
                    if (tid >= off) inc += v;
                }
                if (u < m->U) uoff()[u] = carry + inc - cnt;
                carry += __shfl_sync(0xFFFFFFFFu, inc, 31);
            }
            if (tid == 0) uoff()[m->U] = carry;
        }
        cbar();
        for (int p = tid; p < P; p += LW * 32) {
            const int u = pu()[p];
            if (u < 0) continue;
            const int t = p / a.k;
            plist()[uoff()[u] + __popc(umask()[u] & ((1u << t) - 1u))] = p;
        }
        cbar();
        plan();
    }

    // unit counts and this block's B range (bytes balanced against the A deal)
    __device__ void plan() {
        const int tid = threadIdx.x;
        if (tid == 0) {
            m->tilesI = a.I / 32;
            m->tilesIs = a.shared ? a.Is / 32 : 0;
            m->tilesH = a.H / 32;
            m->n_ra = m->U * m->tilesI;
            m->nA = m->n_sa + m->n_ra;
            m->n_sb = a.shared ? m->tilesH : 0;
            m->n_rb = m->U * m->tilesH;
            m->nB = m->n_sb + m->n_rb;
            m->nc = m->U + (a.shared ? 1 : 0);
        }
        cbar();
        const double sa = 2.0 * FS::tile_bytes(a.H), ra = 2.0 * F::tile_bytes(a.H);
        const double sb = a.shared ? (double)FS::tile_bytes(a.Is) : 0.0, rb = (double)F::tile_bytes(a.I);
        const double totB = m->n_sb * sb + m->n_rb * rb;
        double totA = m->n_sa * sa + m->n_ra * ra;
        // A bytes of block tid (tid < G), then budgets, scan
        double my_a = 0.0;
        if (tid < G) {
            for (int p = 0;; ++p) {
                const int j = snake_unit(p, tid, G);
                if (p * G >= m->nA) break;
                if (j < m->n_sa) my_a += sa;
                else if (j < m->nA) my_a += ra;
            }
        }
        const double target = (totA + totB) / G;
        double b = (tid < G) ? fmax(0.0, target - my_a) : 0.0;
        // block-exclusive scan of b over the first G threads (8 warps x 32)
        double inc = b;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const double v = __shfl_up_sync(0xFFFFFFFFu, inc, off);
            if (lane >= off) inc += v;
        }
        if (lane == 31) m->bsum[warp] = inc;
        cbar();
        double before = 0.0, total = 0.0;
        for (int w = 0; w < LW; ++w) {
            if (w < warp) before += m->bsum[w];
            total += m->bsum[w];
        }
        const double excl = before + inc - b;
        // block c's range [P_c, P_{c+1}) scaled to totB
        __shared__ double s_lo, s_hi;
        const double scale = total > 0.0 ? totB / total : 0.0;
        if (tid == c) s_lo = excl * scale;
        if (tid == c + 1 || (c + 1 == G && tid == 0)) s_hi = (c + 1 == G) ? totB : excl * scale;
        cbar();
        if (tid == 0) {
            m->jb0 = first_b_unit(s_lo, sb, rb);
            m->jb1 = (c + 1 == G) ? m->nB : first_b_unit(s_hi, sb, rb);
            if (m->jb1 < m->jb0) m->jb1 = m->jb0;
        }
        cbar();
    }

    // first B unit whose byte midpoint is >= X
    __device__ int first_b_unit(double X, double sb, double rb) {
        const int n_sb = m->n_sb, n_rb = m->n_rb;
        if (n_sb > 0) {
            double jj = ceil((X - 0.5 * sb) / sb);
            if (jj < 0) jj = 0;
            if (jj < n_sb) return (int)jj;
        }
        const double base = n_sb * sb;
        double jj = ceil((X - base - 0.5 * rb) / rb);
        if (jj < 0) jj = 0;
        if (jj > n_rb) jj = n_rb;
        return n_sb + (int)jj;
    }

    // ------------------------------------------------------- main body
    __device__ void run() {
        init();
        pdl_trigger();
        if (threadIdx.x == 0) {
            m->n_sa = a.shared ? a.Is / 32 : 0;
            m->nA = m->n_sa;
        }
        __syncthreads();
        if (warp == LW) {
            producer();
        } else {
            consumer();
        }
        __syncthreads();
        finish();
    }

    __device__ void producer() {
        Ring R{0, 0, 0};
        if (lane == 0) {
            // input-independent bytes: router rows, expert table, shared gate/up
            int e0, e1;
            router_range(e0, e1);
            const size_t rowb = a.rtype == MOE_F32 ? (size_t)a.H * 4 : (size_t)(a.H / 32) * 34;
            const uint32_t rbytes = (uint32_t)((e1 - e0) * rowb);
            const uint32_t tb = a.table_in_smem ? (uint32_t)(a.E * sizeof(moe_expert)) : 0u;
            if (rbytes + tb > 0) {
                mbar_arm(fixed_bar(), rbytes + tb);
                if (rbytes) bulk_g2s(sm + o.router, (const uint8_t *)a.w_router + (size_t)e0 * rowb, rbytes, fixed_bar());
                if (tb) bulk_g2s(sm + o.table, a.experts, tb, fixed_bar());
            }
            for (int p = 0; !m->abort; ++p) {
                const int j = snake_unit(p, c, G);
                if (p * G >= m->n_sa) break;
                if (j < m->n_sa && !issue_unit(R, j)) break;
            }
        }
        __syncthreads();   // routing handoff: the plan is ready
        if (lane == 0 && !m->abort) {
            for (int p = 0;; ++p) {
                const int j = snake_unit(p, c, G);
                if (p * G >= m->nA) break;
                if (j >= m->n_sa && j < m->nA && !issue_unit(R, j)) break;
            }
            for (int j = m->nA + m->jb0; j < m->nA + m->jb1 && !m->abort; ++j)
                if (!issue_unit(R, j)) break;
        }
        // drain: no copy may still be writing this block's shared memory at exit
        if (lane == 0) {
            for (int i = R.tail; i < R.issued; ++i) mbar_wait(full_bar(i), (uint32_t)((i / NBAR) & 1));
        }
        __syncwarp();
    }

    __device__ void consumer() {
        pdl_wait();
        quantise_x();
        cbar();
        if (c == 0 && a.xq_out) {
            const int n16 = (int)(a.xrec / 16);
            for (int i = threadIdx.x; i < a.T * n16; i += LW * 32)
                reinterpret_cast<uint4 *>(a.xq_out)[i] = reinterpret_cast<const uint4 *>(sm + o.xq)[i];
        }
        router_logits();
        // shared-expert gate/up while the other blocks publish their logits
        int item = 0, rbuf = 0;
        for (int p = 0;; ++p) {
            const int j = snake_unit(p, c, G);
            if (p * G >= m->n_sa) break;
            if (j < m->n_sa) {
                Unit U;
                unit_of(j, U);
                run_A<FS>(U, item, rbuf);
            }
        }
        topk_and_group();
        bar_handoff();
        for (int p = 0;; ++p) {
            const int j = snake_unit(p, c, G);
            if (p * G >= m->nA) break;
            if (j >= m->n_sa && j < m->nA) {
                Unit U;
                unit_of(j, U);
                run_A<F>(U, item, rbuf);
            }
        }
        // no loop below leaves early: every consumer thread must reach every
        // named barrier; after a timeout only waits and sums are skipped
        for (int j = m->nA + m->jb0; j < m->nA + m->jb1; ++j) {
            Unit U;
            unit_of(j, U);
            load_hq(U);
            if (U.kind == 2) run_B<FS>(U, item, rbuf);
            else run_B<F>(U, item, rbuf);
        }
        if (m->nB == 0 && c == 0) {   // nothing owned: y = 0
            for (int i = threadIdx.x; i < a.T * a.H; i += LW * 32) a.y[i] = 0.f;
        }
    }

    // the handoff barrier pairs with the producer's __syncthreads
    __device__ void bar_handoff() { __syncthreads(); }

    __device__ void finish() {
        if (threadIdx.x == 0) {
            __threadfence();
            const unsigned old = atom_acqrel(a.done_ctr, 1u);
            if (old == (unsigned)G - 1u) {
                *a.route_ctr = 0u;
                for (int i = 0; i <= a.P; ++i) a.hctr[i] = 0u;
                a.hctr[MAXP] = 0u;
                for (int i = 0; i < a.H / 32; ++i) a.yticket[i] = 0u;
                __threadfence();
                *a.done_ctr = 0u;
            }
        }
    }
};

template <class F, class FS, int NT>
__global__ void __launch_bounds__(LT, 1) layer_kernel(const __grid_constant__ LayerArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    LayerKernel<F, FS, NT> K(a, smem);
    K.run();
}

template <class F, class FS, int NT>
cudaError_t launch_layer_t(const LayerArgs &a, int G, size_t smem, bool pdl, cudaStream_t s) {
    static int occ_ok[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = ensure_smem<layer_kernel<F, FS, NT>>(smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && occ_ok[dev] < (int)smem + 1) {
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, layer_kernel<F, FS, NT>, LT, smem);
        if (e != cudaSuccess) return e;
        if (n < 1) return cudaErrorInvalidConfiguration;   // every block must be resident at once
        occ_ok[dev] = (int)smem + 1;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)G);
    cfg.blockDim = dim3(LT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, layer_kernel<F, FS, NT>, a);
}

template <class F, class FS>
cudaError_t launch_layer_nt(const LayerArgs &a, int G, size_t smem, bool pdl, cudaStream_t s) {
    if (a.NT == 1) return launch_layer_t<F, FS, 1>(a, G, smem, pdl, s);
    if (a.NT == 4) return launch_layer_t<F, FS, 4>(a, G, smem, pdl, s);
    return launch_layer_t<F, FS, 16>(a, G, smem, pdl, s);
}

}  // namespace moe
