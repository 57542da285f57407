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
//  2. After griddepcontrol.wait every block computes the logits of its
//     router rows in the fixed summation order and publishes them, then
//     quantises x itself (a Q8_0 router dots the quantised x, so it
//     quantises first); while the other blocks finish, it runs its share of
//     the shared expert's gate/up.
//  3. Every block reads every logit and selects the same top-k, groups the
//     (token, slot) pairs by expert and derives the same work plan:
//       A units = (expert, 32-row tile of I): gate + up records,
//       B units = (expert, 32-row tile of H): down records.
//     A units are dealt out in a snake over blocks; B units go in
//     contiguous ranges sized so every block streams about the same number
//     of bytes (so a block's B units need the h of one or two experts).
//  4. The producer streams the units' records (TMA bulk copies, complete_tx
//     mbarriers) through a byte ring, up to eight records per copy; consumer
//     warp r % 8 takes record r of an A unit, and a batch's B records are
//     spread over the warps with per-record partial sums added in record
//     order, so every sum has a fixed order whatever the batch.
//  5. An A unit ends with h = silu(g) * u rows in global scratch; a B
//     batch's block first requantises its experts' h locally, and each B
//     unit ends with o rows; row tile rt of y is written by block rt % G,
//     which sums the slots of each token in slot order (shared expert last).
//  Exchanges between blocks (logits, h, o) carry no separate flag: every
//  value is stored with this launch's epoch in one 8-byte word, and a reader
//  polls the words it needs, re-reading all the missing ones each round,
//  until they carry the epoch.  An 8-byte aligned
//  access is single-copy atomic, so a word with the right epoch holds the
//  right value and no fence is needed on either side.  The epoch comes
//  from one counter per block in the workspace: block c reads its own after
//  the dependency wait and writes it back (+1) as it ends.  Every block
//  advances its counter once per launch, so all blocks agree on the epoch, and
//  no block touches another's counter.
//  Every wait is bounded (SM cycle counter); a timeout sets MOE_DEV_TIMEOUT,
//  drains this block's copies in flight and returns.
#pragma once

#include <type_traits>

#include "moe_common.cuh"
#include "moe_launch.h"

namespace moe {

// consumer warps: 16 for one token (four per SM sub-partition keep the
// integer dots' latencies covered), 8 for four tokens (four times the dot
// work per record and per register)
template <int NT>
struct Warps {
    static constexpr int LW = NT == 1 ? 16 : 8;
    static constexpr int LT = (LW + 1) * 32;   // threads per block (with the producer warp)
};
constexpr int MAX_LW = 16;
constexpr int NBAR = 32;               // ring items in flight (barrier slots)
constexpr int MAX_ITEM_RECS = 16;      // records per ring item, at most (also the empty-barrier count)
// bound on every device-side wait, in SM clock cycles (about 0.4-1 s at the
// clocks this part runs at); the cycle counter is cheap to poll.  Waits for
// another block's exchange words use the launch's wait_limit instead (this
// value unless a test sets a shorter one); waits for this block's own bulk
// copies always use this bound, so no block leaves with a copy in flight.
constexpr long long WAIT_CYCLES = 800ll * 1000ll * 1000ll;

// ------------------------------------------------------------ PTX helpers

__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_arm(uint64_t *b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive_n(uint64_t *b, uint32_t n) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(b)), "r"(n) : "memory");
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
// bounded wait on an mbarrier phase; false on timeout (the loop is out of line)
static __device__ __noinline__ bool mbar_wait_slow(uint64_t *b, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_test(b, parity))
        if (clock64() - t0 > WAIT_CYCLES) return false;
    return true;
}
__device__ __forceinline__ bool mbar_wait(uint64_t *b, uint32_t parity) {
    return mbar_test(b, parity) || mbar_wait_slow(b, parity);
}
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            saddr(dst)),
        "l"(src), "r"(bytes), "r"(saddr(bar))
        : "memory");
}
// Weight records and router rows are read once per launch: their L2 lines
// are marked evict-first, so the stream does not push out what the launch
// re-reads (exchange words, activations, expert tables, the kernel's code).
__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void bulk_g2s_stream(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                                uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(saddr(dst)),
        "l"(src), "r"(bytes), "r"(saddr(bar)), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// tagged word: the value's bits in the low half, the epoch in the high half
typedef unsigned long long tword;
__device__ __forceinline__ void st_tag(tword *p, float v, uint32_t ep) {
    const tword w = ((tword)ep << 32) | __float_as_uint(v);
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ tword ld_tag(const tword *p) {
    tword w;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
    return w;
}
// two adjacent tagged words (16-byte aligned); each word is read atomically
__device__ __forceinline__ void ld_tag2(const tword *p, tword &w0, tword &w1) {
    asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(w0), "=l"(w1) : "l"(p) : "memory");
}
__device__ __forceinline__ uint32_t tag_of(tword w) { return (uint32_t)(w >> 32); }
__device__ __forceinline__ float tag_value(tword w) { return __uint_as_float((uint32_t)w); }
__device__ __forceinline__ uint32_t ld_relaxed_u32(const unsigned *p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_u32(unsigned *p, uint32_t v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// A line of global memory into L2 (no value comes back, so it may run before
// the dependency wait: the later loads still read L2, the point of coherence)
__device__ __forceinline__ void prefetch_l2(const void *p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }
template <int LW>
__device__ __forceinline__ void cbar_n() { asm volatile("bar.sync 1, %0;" ::"n"(LW * 32) : "memory"); }   // consumers only

// ------------------------------------------------------------- block state

// The work plan's counts and this block's B range for U owned experts.
struct SpecPlan {
    int tilesI, tilesIs, tilesH, n_ra, nA, n_sb, n_rb, nB, brev, closed, jb0, jb1, nb;
    uint32_t target, lo, hi;
};

struct Misc {
    volatile int abort;
    volatile int spec_ready;   // one token: the producer's plan for U = k is in spec
    int use_spec;
    SpecPlan spec;
    int U, n_sa, n_ra, nA, n_sb, n_rb, nB, jb0, jb1;
    int tilesI, tilesIs, tilesH;
    uint32_t ep;         // this launch's epoch
    moe_expert shx;      // the shared expert's table entry, copied before the routing handoff
    uint32_t bitmap[MOE_MAX_EXPERTS / 32];
    int wpre[MOE_MAX_EXPERTS / 32];
    int nkeys, kkey[64], kslot[64];   // experts of the current B batch and their hq slots
    int nb, bend;                      // this block's B units: [jb0, jb1), nb of them; end of the hq batch
    // the current hq batch's B units (at most 64): unit index, first ring
    // item and first record (relative to the batch; entry [n] holds the
    // totals) and hq slot
    int bt_j[64], bt_it[65], bt_rec[65], bt_slot[64];
    uint32_t bsum[MAX_LW], target, lo, hi;   // B shares, in quarters of 128-byte lines
    int closed;          // the B shares need no clamping (closed form)
    float sgate[4];      // per-token weight of the shared expert (with a gate vector)
    int brev;            // B ranges are given to blocks G-1 first
};

static_assert(sizeof(Misc) <= kLayerMiscBytes, "fused kernel block state outgrew its shared-memory region");

// Slow paths, out of line and free of the kernel object: every launch runs
// this kernel's code once per phase, and fetching cold instructions costs
// about as much as the work, so each inlined copy of a rarely taken loop is
// paid for on every launch.
static __device__ __noinline__ void fail_dev(Misc *m, unsigned *status) {
    m->abort = 1;
    atomicOr(status, MOE_DEV_TIMEOUT);
}
// p re-read until it carries epoch ep (bounded; on timeout the value is not used)
static __device__ __noinline__ tword wait_tag_slow(const tword *p, uint32_t ep, Misc *m, unsigned *status,
                                                   long long limit) {
    const long long t0 = clock64();
    for (;;) {
        const tword w = ld_tag(p);
        if (tag_of(w) == ep) return w;
        if (m->abort || clock64() - t0 > limit) {
            fail_dev(m, status);
            return w;
        }
    }
}
// ring item i: its slot tag set by the producer (a consumer ahead of the
// producer sleeps between polls: a tight loop of shared-memory loads by eight
// warps slows the producer), then its full barrier; false on abort or timeout
static __device__ __noinline__ bool wait_item_slow(int i, volatile uint32_t *tags, uint64_t *full, Misc *m,
                                                   unsigned *status) {
    if (m->abort) return false;
    const long long t0 = clock64();
    while (tags[i % NBAR] != (uint32_t)i) {
        __nanosleep(64);
        if (clock64() - t0 > WAIT_CYCLES || m->abort) { fail_dev(m, status); return false; }
    }
    if (!mbar_wait(full, (uint32_t)((i / NBAR) & 1))) { fail_dev(m, status); return false; }
    return true;
}

// Compute steps shared by several phases.
//
// The block's dynamic shared memory.  Code that gets byte offsets into it
// (rather than generic pointers) compiles to shared-memory loads.
extern __shared__ __align__(128) unsigned char moe_smem[];

// One packed record (at shared offset rec) dotted with nt activation records
// (record i at shared offset abase + aidx[i] * astride): integer sub-block
// dots, accumulated in record order into acc[i].  Used by the gate, up and
// down projections.
// The record is pulled into registers (w) first, so its ring slot can be
// released before the dots run (rec_load, then rec_dot_w).
template <class FF>
static __device__ __forceinline__ void rec_load(typename FF::W &w, uint32_t rec, int nb, int lane) {
    FF::load_s(w, moe_smem + rec, nb, lane);
}
template <class FF, int NT>
static __device__ __forceinline__ void rec_dot_w(const typename FF::W &w, int nb, int k0, int cols, uint32_t abase,
                                              uint32_t astride, const int *aidx, int nt, float *acc) {
#pragma unroll
    for (int i = 0; i < NT; ++i) {
        if (i < nt) {
            const Act x = act_view(moe_smem + abase + (uint32_t)aidx[i] * astride, cols);
            int is[FF::NSUB];
            FF::isums(w, x, k0, nb, is);
            acc[i] = __fadd_rn(acc[i], FF::combine(w, x, k0, nb, is));
        }
    }
}
// monotone unsigned key of a float (larger float -> larger key); -0 and +0
// share the key of +0 so equal logits tie and the lower index wins
__device__ __forceinline__ uint32_t fkey(float v) {
    if (v == 0.f) v = 0.f;
    const uint32_t b = __float_as_uint(v);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float fkey_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Snake over blocks: unit j -> block, pass by pass, reversing every other pass.
__device__ __forceinline__ int snake_unit(int pass, int c, int G) {
    return pass * G + ((pass & 1) ? (G - 1 - c) : c);
}

// The work plan every thread keeps in registers once it is known (thread 0
// derives it in shared memory; re-reading those words and dividing by the
// tile counts on every use cost hundreds of cycles per unit).
struct Plan {
    int n_sa, nA, n_sb, nB;      // A units: shared then routed; B units: shared then routed
    int tilesI, tilesIs, tilesH; // 32-row tiles of I, of the shared expert's I, of H
    float invI, invH;            // 1 / tilesI, 1 / tilesH (quotients corrected exactly)
    int nb, jb0;                 // this block's B units: [jb0, jb0 + nb)
};

// q / t for 0 <= q < 2^22, t >= 1, from a float estimate corrected exactly
__device__ __forceinline__ int div_tiles(int q, int t, float inv) {
    int u = (int)((float)q * inv);
    if (u * t > q) --u;
    if ((u + 1) * t <= q) ++u;
    return u;
}

template <class F, class FS, int NT>
struct LayerKernel {
    static constexpr int LW = Warps<NT>::LW, LT = Warps<NT>::LT;
    __device__ static void cbar() { cbar_n<LW>(); }
    const LayerArgs &a;
    unsigned char *sm;
    Smem o;
    Misc *m;
    int c, G, warp, lane;
    uint32_t ep = 0;   // consumers: this launch's epoch (after the dependency wait)
    Plan p;            // loaded by load_plan once the plan is in shared memory
    // the shared expert's table entry: the caller's device table until the
    // routing handoff, then the block's shared-memory copy of it
    const moe_expert *shp;

    __device__ LayerKernel(const LayerArgs &args, unsigned char *smem) : a(args), sm(smem), o(args.sm) {
        m = reinterpret_cast<Misc *>(sm + o.misc);
        c = blockIdx.x;
        G = gridDim.x;
        warp = threadIdx.x >> 5;
        lane = threadIdx.x & 31;
        shp = args.shared;
    }

    __device__ uint64_t *full_bar(int i) { return reinterpret_cast<uint64_t *>(sm + o.bars) + (i % NBAR); }
    __device__ uint64_t *empty_bar(int i) { return reinterpret_cast<uint64_t *>(sm + o.bars) + NBAR + (i % NBAR); }
    __device__ uint64_t *fixed_bar() { return reinterpret_cast<uint64_t *>(sm + o.bars) + 2 * NBAR; }
    // A-unit partial sums, two buffers: ready (every consumer warp has
    // written its partials) and free (the unit's reducing warp has read them)
    __device__ uint64_t *ready_bar(int b) { return reinterpret_cast<uint64_t *>(sm + o.bars) + 2 * NBAR + 1 + b; }
    __device__ uint64_t *free_bar(int b) { return reinterpret_cast<uint64_t *>(sm + o.bars) + 2 * NBAR + 3 + b; }
    __device__ uint32_t *starts() { return reinterpret_cast<uint32_t *>(sm + o.starts); }
    // item index currently owning each ring slot (set by the producer once the
    // slot's previous item is reclaimed); lets a consumer that is many items
    // ahead of the ring wait for its own item instead of an earlier phase of
    // the same barrier with the same parity
    __device__ volatile uint32_t *tags() { return reinterpret_cast<volatile uint32_t *>(sm + o.starts) + NBAR; }
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

    __device__ void fail() { fail_dev(m, a.status); }

    __device__ void load_plan() {
        p.n_sa = m->n_sa;
        p.nA = m->nA;
        p.n_sb = m->n_sb;
        p.nB = m->nB;
        p.tilesI = a.I / 32;
        p.tilesIs = a.shared ? a.Is / 32 : 0;
        p.tilesH = a.H / 32;
        p.invI = 1.f / (float)p.tilesI;
        p.invH = 1.f / (float)p.tilesH;
        p.nb = m->nb;
        p.jb0 = m->jb0;
    }

    // w, already loaded from p, if it carries this launch's epoch, else p re-read
    __device__ __forceinline__ tword wait_tag(const tword *p, tword w) {
        return tag_of(w) == ep ? w : wait_tag_slow(p, ep, m, a.status, a.wait_limit);
    }

    // ------------------------------------------------------------ units
    // kind: 0 shared A, 1 routed A, 2 shared B, 3 routed B
    struct Unit {
        int kind, u, rt, nrec, nt, nitems;
        const uint8_t *g, *up, *d;   // tile bases (A: gate/up, B: down)
        const moe_expert *ex;
    };

    // log2 of the records per ring item of a unit kind (each format sizes its own)
    __device__ __forceinline__ int lg_of(int kind) const {
        return kind == 0 ? a.lgsa : (kind == 1 ? a.lgra : (kind == 2 ? a.lgsb : a.lgrb));
    }
    __device__ void unit_of(int j, Unit &U) {
        unit_of0(j, U);
        const int lg = lg_of(U.kind);
        U.nitems = (U.nrec + (1 << lg) - 1) >> lg;
    }
    __device__ void unit_of0(int j, Unit &U) {
        const moe_expert *T = table();
        if (j < p.n_sa) {
            U.kind = 0; U.u = MAXP; U.rt = j;
            U.ex = shp;
            U.nrec = FS::nrec(a.H);
            U.nt = a.T;
            const size_t tb = FS::tile_bytes(a.H);
            U.g = (const uint8_t *)shp->gate + (size_t)U.rt * tb;
            U.up = (const uint8_t *)shp->up + (size_t)U.rt * tb;
        } else if (j < p.nA) {
            const int q = j - p.n_sa;
            U.kind = 1; U.u = div_tiles(q, p.tilesI, p.invI); U.rt = q - U.u * p.tilesI;
            U.ex = T + ue()[U.u];
            U.nrec = F::nrec(a.H);
            U.nt = uoff()[U.u + 1] - uoff()[U.u];
            const size_t tb = F::tile_bytes(a.H);
            U.g = (const uint8_t *)U.ex->gate + (size_t)U.rt * tb;
            U.up = (const uint8_t *)U.ex->up + (size_t)U.rt * tb;
        } else if (j < p.nA + p.n_sb) {
            U.kind = 2; U.u = MAXP; U.rt = j - p.nA;
            U.ex = shp;
            U.nrec = FS::nrec(a.Is);
            U.nt = a.T;
            U.d = (const uint8_t *)shp->down + (size_t)U.rt * FS::tile_bytes(a.Is);
        } else {
            const int q = j - p.nA - p.n_sb;
            U.kind = 3; U.u = div_tiles(q, p.tilesH, p.invH); U.rt = q - U.u * p.tilesH;
            U.ex = T + ue()[U.u];
            U.nrec = F::nrec(a.I);
            U.nt = uoff()[U.u + 1] - uoff()[U.u];
            U.d = (const uint8_t *)U.ex->down + (size_t)U.rt * F::tile_bytes(a.I);
        }
    }

    // Ring item q of a unit: records [r0, r1) with r0 = q R (R = 2^lg_of(kind)).
    // An A item holds the gate run, then the up run of the same records; a B
    // item holds the down run.
    __device__ void item_recs(const Unit &U, int q, int &r0, int &r1) {
        const int lg = lg_of(U.kind);
        r0 = q << lg;
        r1 = min(r0 + (1 << lg), U.nrec);
    }
    // byte offset of record r within its run (a run starts at record r0)
    template <class FF>
    __device__ static size_t run_off(int cols, int r0, int r) { return FF::rec_off(cols, r) - FF::rec_off(cols, r0); }
    __device__ uint32_t run_bytes(const Unit &U, int r0, int r1) {
        switch (U.kind) {
            case 0: return (uint32_t)run_off<FS>(a.H, r0, r1);
            case 1: return (uint32_t)run_off<F>(a.H, r0, r1);
            case 2: return (uint32_t)run_off<FS>(a.Is, r0, r1);
            default: return (uint32_t)run_off<F>(a.I, r0, r1);
        }
    }

    // -------------------------------------------------------- producer
    struct Ring {
        uint32_t head;
        int issued, tail;   // items issued so far; oldest item not yet reclaimed
        uint64_t pol;       // L2 policy of the weight stream
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

    __device__ bool issue(Ring &R, const Unit &U, int q) {
        int r0, r1;
        item_recs(U, q, r0, r1);
        const uint32_t run = run_bytes(U, r0, r1);
        const uint32_t bytes = U.kind <= 1 ? 2 * run : run;
        uint32_t start;
        if (!ring_place(R, bytes, start)) return false;
        const int i = R.issued;
        starts()[i % NBAR] = start;
        tags()[i % NBAR] = (uint32_t)i;
        uint8_t *dst = sm + o.ring + start;
        uint64_t *fb = full_bar(i);
        mbar_arm(fb, bytes);
        // consumers arrive once per record of the item (an A item holds a
        // gate and an up record per row range)
        const uint32_t users = (uint32_t)((U.kind <= 1 ? 2 : 1) * (r1 - r0));
        if (users < MAX_ITEM_RECS) mbar_arrive_n(empty_bar(i), MAX_ITEM_RECS - users);
        if (U.kind == 0 || U.kind == 1) {
            const size_t off = U.kind == 0 ? FS::rec_off(a.H, r0) : F::rec_off(a.H, r0);
            bulk_g2s_stream(dst, U.g + off, run, fb, R.pol);
            bulk_g2s_stream(dst + run, U.up + off, run, fb, R.pol);
        } else {
            const size_t off = U.kind == 2 ? FS::rec_off(a.Is, r0) : F::rec_off(a.I, r0);
            bulk_g2s_stream(dst, U.d + off, run, fb, R.pol);
        }
        R.head = start + bytes;
        ++R.issued;
        return true;
    }

    __device__ bool issue_unit(Ring &R, int j, int q0 = 0) {
        Unit U;
        unit_of(j, U);
        for (int q = q0; q < U.nitems; ++q) {
            if (m->abort) return false;
            if (!issue(R, U, q)) { fail(); return false; }
        }
        return true;
    }

    // ------------------------------------------------------- consumers
    // one record of a unit: wait for it, pull it into registers, free the slot
    // wait for item i (a record, or a gate+up record pair) to land in the ring
    // (a consumer ahead of the producer sleeps between polls of the tag: a
    // tight loop of shared-memory loads by eight warps slows the producer's
    // own shared-memory and barrier operations)
    __device__ __forceinline__ const uint8_t *wait_item(int i) {
        const bool ok = (!m->abort && tags()[i % NBAR] == (uint32_t)i && mbar_test(full_bar(i), (uint32_t)((i / NBAR) & 1))) ||
                        wait_item_slow(i, tags(), full_bar(i), m, a.status);
        return ok ? sm + o.ring + starts()[i % NBAR] : nullptr;
    }
    // n consumer arrivals on item i's empty barrier (one per record used)
    __device__ void free_item(int i, uint32_t n = 1) {
        __syncwarp();
        if (lane == 0) mbar_arrive_n(empty_bar(i), n);
    }

    // A unit: g and u partial sums of this warp's records, then h rows.  No
    // block-wide barrier per unit: each warp leaves its partials in buffer
    // ua % 2 and goes on to its next unit; the unit's reducing warp (ua % LW)
    // waits for all of them, writes h and hands the buffer back.  A warp
    // reuses a buffer only after the reducer of its previous use is done.
    template <class FF>
    __device__ void run_A(const Unit &U, int &item, int &ua) {
        float ag[NT], au[NT];
#pragma unroll
        for (int i = 0; i < NT; ++i) { ag[i] = 0.f; au[i] = 0.f; }
        int tok[NT];
#pragma unroll
        for (int i = 0; i < NT; ++i)
            tok[i] = (i < U.nt) ? (U.kind == 0 ? i : plist()[uoff()[U.u] + i] / a.k) : 0;
        // Record r's gate and up records both go to warp r % LW, which frees
        // the ring slot once it has read them both (during the up dot).
        const int lg = lg_of(U.kind);
        for (int r = warp; r < U.nrec; r += LW) {
            int r0, r1;
            item_recs(U, r >> lg, r0, r1);
            const int it = item + (r >> lg);
            const uint8_t *base = wait_item(it);
            if (!base) continue;
            const uint8_t *rec = base + run_off<FF>(a.H, r0, r);
            const uint8_t *rec_up = base + run_off<FF>(a.H, r0, r1) + run_off<FF>(a.H, r0, r);
            const int nb = FF::rec_blocks(a.H, r);
            const int k0 = r * FF::QK;
            typename FF::W w;
            rec_load<FF>(w, (uint32_t)(rec - sm), nb, lane);
            rec_dot_w<FF, NT>(w, nb, k0, a.H, o.xq, (uint32_t)a.xrec, tok, U.nt, ag);
            rec_load<FF>(w, (uint32_t)(rec_up - sm), nb, lane);
            free_item(it, 2);
            rec_dot_w<FF, NT>(w, nb, k0, a.H, o.xq, (uint32_t)a.xrec, tok, U.nt, au);
        }
        item += U.nitems;
        const int b = ua & 1, use = ua >> 1;
        float *red = reinterpret_cast<float *>(sm + o.red) + b * (LW * 2 * NT * 32);
        if (use > 0 && !m->abort && !mbar_wait(free_bar(b), (uint32_t)((use - 1) & 1))) fail();
#pragma unroll
        for (int i = 0; i < NT; ++i) {
            red[((warp * 2 + 0) * NT + i) * 32 + lane] = ag[i];
            red[((warp * 2 + 1) * NT + i) * 32 + lane] = au[i];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_n(ready_bar(b), 1);
        if (warp == ua % LW) {
            if (!m->abort && !mbar_wait(ready_bar(b), (uint32_t)(use & 1))) fail();
            const int row = U.rt * 32 + lane;
            const int Irows = U.kind == 0 ? a.Is : a.I;
            tword *hb = U.kind == 0 ? a.h_s : a.h_r;
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
                st_tag(hb + (size_t)dest * Irows + row, h, ep);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_n(free_bar(b), 1);
        }
        ++ua;
    }

    // ---------------------------------------------------------- B phase
    // The block's B units run in batches of consecutive units whose experts'
    // requantised h fit the hq buffer together.  Per batch: read those
    // experts' h (polling the tagged words) and requantise every pair of them
    // into hq (all warps), then unit b of the batch goes to warp b % 8, which
    // streams its records in order and writes the o rows itself.

    // expert key of B unit j: MAXP for the shared expert, else its unique index
    __device__ int b_key(int j) {
        if (j < p.nA + p.n_sb) return MAXP;
        return div_tiles(j - p.nA - p.n_sb, p.tilesH, p.invH);
    }
    __device__ int key_pairs(int key) { return key == MAXP ? a.T : uoff()[key + 1] - uoff()[key]; }

    // From list entry n0, the longest run of B units whose distinct experts'
    // pairs fit the hq buffer together (at most 64 experts, chosen by thread
    // 0): requantise those experts' h into hq.  Returns the end of the run.
    // lane's 8 h values (8 lane .. 8 lane + 7 of the 256-chunk at c0) from
    // tagged words: four 16-byte loads, repeated (bounded) until all carry
    // this launch's epoch; false past the row
    __device__ bool load8_tagged(const tword *x, int n, int c0, float v[8]) {
        const int e0 = c0 + 8 * lane;
        if (e0 >= n || m->abort) {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = 0.f;
            return false;
        }
        tword w[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) ld_tag2(x + e0 + 2 * i, w[2 * i], w[2 * i + 1]);
        // one warp store wrote all eight words, so they turn up together:
        // re-read all of them per round (one round trip), not word by word
        bool all = true;
#pragma unroll
        for (int i = 0; i < 8; ++i) all &= tag_of(w[i]) == ep;
        if (!all) {
            const long long t0 = clock64();
            for (;;) {
#pragma unroll
                for (int i = 0; i < 4; ++i) ld_tag2(x + e0 + 2 * i, w[2 * i], w[2 * i + 1]);
                all = true;
#pragma unroll
                for (int i = 0; i < 8; ++i) all &= tag_of(w[i]) == ep;
                if (all) break;
                if (m->abort || clock64() - t0 > a.wait_limit) {
                    fail();
                    break;
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = tag_value(w[i]);
        return true;
    }

    __device__ int load_hq_batch(int n0, int nend) {
        int *kbase = m->kslot;
        int *keys = m->kkey;
        if (warp == 0) {
            // units from n0 in order: a unit whose expert differs from the
            // previous unit's brings that expert (B ranges are contiguous, so
            // each expert's units are consecutive); the batch ends before the
            // first new expert whose pairs would overflow the hq slots or
            // that would be the 65th, and after 64 units.  Lane l takes unit
            // base + l; prefix sums over the lanes stand in for a serial walk.
            int nk = 0, used = 0, n = n0, prev_key = -1;
            for (int base = n0; base < nend && base - n0 < 64; base += 32) {
                const int i = base + lane;
                const bool valid = i < nend && i - n0 < 64;
                const int key = valid ? b_key(b_unit(i)) : -2;
                const int up = __shfl_up_sync(0xFFFFFFFFu, key, 1);
                const bool isnew = valid && key != (lane == 0 ? prev_key : up);
                const int need = isnew ? key_pairs(key) : 0;
                int cn = need, ck = isnew ? 1 : 0;   // inclusive prefix sums
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int vn = __shfl_up_sync(0xFFFFFFFFu, cn, off), vk = __shfl_up_sync(0xFFFFFFFFu, ck, off);
                    if (lane >= off) { cn += vn; ck += vk; }
                }
                const bool brk = isnew && i > n0 && (used + cn > a.hq_slots || nk + ck > 64);
                const unsigned stop = __ballot_sync(0xFFFFFFFFu, brk || !valid);
                const int first = stop ? __ffs(stop) - 1 : 32;   // units base .. base + first - 1 join
                if (lane < first && isnew) {
                    keys[nk + ck - 1] = key;
                    kbase[nk + ck - 1] = used + cn - need;
                }
                if (first > 0) {
                    used += __shfl_sync(0xFFFFFFFFu, cn, first - 1);
                    nk += __shfl_sync(0xFFFFFFFFu, ck, first - 1);
                    prev_key = __shfl_sync(0xFFFFFFFFu, key, first - 1);
                }
                n = base + first;
                if (first < 32) break;
            }
            if (lane == 0) {
                m->nkeys = nk;
                m->bend = n;
            }
        }
        cbar();
        if (warp == 0) b_table(n0, m->bend);   // the batch's unit table, while h is still arriving
        const int nk = m->nkeys;
        const bool ok = !m->abort;
        // tasks (key, pair, 256-chunk), flattened; a warp loads the h of up to
        // two tasks before quantising them (each load is an L2 trip)
        int ntask = 0;
        for (int kk = 0; kk < nk; ++kk) {
            const int key = keys[kk];
            const int Irows = key == MAXP ? a.Is : a.I;
            ntask += key_pairs(key) * ((Irows + 255) / 256);
        }
        for (int w0 = warp; ok && w0 < ntask; w0 += 2 * LW) {
            float v[2][8];
            bool act[2];
            const tword *src[2];
            uint8_t *dst[2];
            int cidx[2], nrow[2];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int w = w0 + q * LW;
                act[q] = false;
                if (w >= ntask) continue;
                int rem = w, kk = 0;
                for (;; ++kk) {   // locate the task's expert
                    const int Ir = keys[kk] == MAXP ? a.Is : a.I;
                    const int nt = key_pairs(keys[kk]) * ((Ir + 255) / 256);
                    if (rem < nt) break;
                    rem -= nt;
                }
                const int key = keys[kk];
                const int Irows = key == MAXP ? a.Is : a.I;
                const int chunks = (Irows + 255) / 256;
                const int i = rem / chunks, ch = rem - i * chunks;
                const int dest = key == MAXP ? i : plist()[uoff()[key] + i];
                src[q] = (key == MAXP ? a.h_s : a.h_r) + (size_t)dest * Irows;
                dst[q] = hq(kbase[kk] + i);
                cidx[q] = 256 * ch;
                nrow[q] = Irows;
                act[q] = load8_tagged(src[q], Irows, cidx[q], v[q]);
            }
#pragma unroll
            for (int q = 0; q < 2; ++q)
                if (w0 + q * LW < ntask) quant_store8(v[q], act[q], nrow[q], cidx[q], dst[q], lane);
        }
        cbar();
        return m->bend;
    }

    __device__ int key_slot(int key) {
        for (int q = 0; q < m->nkeys; ++q)
            if (m->kkey[q] == key) return m->kslot[q];
        return 0;
    }

    // one B unit by one warp: records in order, then its o rows
    template <class FF>
    __device__ void run_B_warp(const Unit &U, int item, int slot0) {
        const int Irows = U.kind == 2 ? a.Is : a.I;
        float ao[NT];
        int sidx[NT];   // hq slots of the unit's pairs
#pragma unroll
        for (int i = 0; i < NT; ++i) { ao[i] = 0.f; sidx[i] = slot0 + i; }
        for (int q = 0; q < U.nitems; ++q) {
            int r0, r1;
            item_recs(U, q, r0, r1);
            const uint8_t *base = wait_item(item + q);
            if (!base) continue;
            for (int r = r0; r < r1; ++r) {
                typename FF::W w;
                rec_load<FF>(w, (uint32_t)(base - sm + run_off<FF>(Irows, r0, r)), FF::rec_blocks(Irows, r), lane);
                if (r + 1 == r1) free_item(item + q, (uint32_t)(r1 - r0));
                rec_dot_w<FF, NT>(w, FF::rec_blocks(Irows, r), r * FF::QK, Irows, o.hq, (uint32_t)a.hrec, sidx, U.nt, ao);
            }
        }
        store_o(U, ao);
    }

    // o rows of a B unit (its expert's down bias added), as tagged words
    __device__ void store_o(const Unit &U, const float *ao) {
        const int row = U.rt * 32 + lane;
        const float bd = (U.kind == 3 && U.ex->b_down) ? U.ex->b_down[row] : 0.f;
#pragma unroll
        for (int i = 0; i < NT; ++i) {
            if (i < U.nt) {
                if (U.kind == 3) {
                    const int p = plist()[uoff()[U.u] + i];
                    st_tag(a.o_r + (size_t)p * a.H + row, U.ex->b_down ? ao[i] + bd : ao[i], ep);
                } else {
                    st_tag(a.o_s + (size_t)i * a.H + row, ao[i], ep);
                }
            }
        }
    }

    // One record of a B unit into partial slot t: o-row partial sums of that
    // record alone (fresh accumulators, so the later in-order sum of the
    // slots equals the unit's sequential sum bit for bit).
    template <class FF>
    __device__ void run_B_record(const Unit &U, int it0, int slot0, int r, int t) {
        const int Irows = U.kind == 2 ? a.Is : a.I;
        const int lg = lg_of(U.kind);
        const int q = r >> lg, r0 = q << lg;
        float pt[NT];
        int sidx[NT];
#pragma unroll
        for (int i = 0; i < NT; ++i) { pt[i] = 0.f; sidx[i] = slot0 + i; }
        const uint8_t *base = wait_item(it0 + q);
        if (base) {
            typename FF::W w;
            rec_load<FF>(w, (uint32_t)(base - sm + run_off<FF>(Irows, r0, r)), FF::rec_blocks(Irows, r), lane);
            free_item(it0 + q);
            rec_dot_w<FF, NT>(w, FF::rec_blocks(Irows, r), r * FF::QK, Irows, o.hq, (uint32_t)a.hrec, sidx, U.nt, pt);
        }
        float *part = reinterpret_cast<float *>(sm + o.red);
#pragma unroll
        for (int i = 0; i < NT; ++i) part[(t * NT + i) * 32 + lane] = pt[i];
    }

    // warp 0: the unit table of B units [n, n1) (at most 64), built while the
    // batch's h is requantised
    __device__ void b_table(int n, int n1) {
        int nr[2], ni[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int k = lane + 32 * h, q = n + k;
            nr[h] = ni[h] = 0;
            if (q < n1) {
                const int j = b_unit(q), key = b_key(j);
                nr[h] = key == MAXP ? FS::nrec(a.Is) : F::nrec(a.I);
                const int lg = key == MAXP ? a.lgsb : a.lgrb;
                ni[h] = (nr[h] + (1 << lg) - 1) >> lg;
                m->bt_j[k] = j;
                m->bt_slot[k] = key_slot(key);
            }
        }
        int carry_r = 0, carry_i = 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            int sr = nr[h], si = ni[h];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int vr = __shfl_up_sync(0xFFFFFFFFu, sr, off), vi = __shfl_up_sync(0xFFFFFFFFu, si, off);
                if (lane >= off) { sr += vr; si += vi; }
            }
            const int k = lane + 32 * h;
            m->bt_rec[k] = carry_r + sr - nr[h];
            m->bt_it[k] = carry_i + si - ni[h];
            carry_r += __shfl_sync(0xFFFFFFFFu, sr, 31);
            carry_i += __shfl_sync(0xFFFFFFFFu, si, 31);
        }
        // entries past the batch hold the totals (their counts are zero)
        if (lane == 0) { m->bt_rec[64] = carry_r; m->bt_it[64] = carry_i; }
    }

    // B units of one hq batch.  Groups of whole units with at most a.bslots
    // records in all (or one unit) are spread record by record over the
    // warps (record t of the group to warp t % 8, each warp in record order):
    // each record's partial sums go to a slot of the reduction buffer, then
    // one warp per unit adds its slots in record order and writes the o rows.
    // A unit with more records than the buffer has slots runs on one warp.
    __device__ void run_B_batch(int n, int n1, int &item) {
        const int CAP = a.bslots;   // record slots in the reduction buffer
        const int nu = n1 - n;   // the unit table was built by load_hq_batch
        const int *brec = m->bt_rec;
        for (int k = 0; k < nu;) {
            int ke = k + 1;
            while (ke < nu && brec[ke + 1] - brec[k] <= CAP) ++ke;
            const int recs = brec[ke] - brec[k];
            if (recs > CAP) {   // one long unit: the warp-per-unit path
                if (warp == 0) {
                    Unit U;
                    unit_of(m->bt_j[k], U);
                    if (std::is_same<F, FS>::value || U.kind == 3) run_B_warp<F>(U, item + m->bt_it[k], m->bt_slot[k]);
                    else run_B_warp<FS>(U, item + m->bt_it[k], m->bt_slot[k]);
                }
                k = ke;
                continue;
            }
            int kk = k;
            for (int t = warp; t < recs; t += LW) {
                while (brec[kk + 1] - brec[k] <= t) ++kk;
                Unit U;
                unit_of(m->bt_j[kk], U);
                const int r = t - (brec[kk] - brec[k]);
                if (std::is_same<F, FS>::value || U.kind == 3) run_B_record<F>(U, item + m->bt_it[kk], m->bt_slot[kk], r, t);
                else run_B_record<FS>(U, item + m->bt_it[kk], m->bt_slot[kk], r, t);
            }
            cbar();
            const float *part = reinterpret_cast<const float *>(sm + o.red);
            for (int kk = k + warp; kk < ke; kk += LW) {
                Unit U;
                unit_of(m->bt_j[kk], U);
                float ao[NT];
#pragma unroll
                for (int i = 0; i < NT; ++i) ao[i] = 0.f;
                for (int s = brec[kk] - brec[k]; s < brec[kk + 1] - brec[k]; ++s) {
#pragma unroll
                    for (int i = 0; i < NT; ++i) ao[i] = __fadd_rn(ao[i], part[(s * NT + i) * 32 + lane]);
                }
                store_o(U, ao);
            }
            cbar();   // the next group reuses the slots
            k = ke;
        }
        item += m->bt_it[nu];
    }

    __device__ void run_B_phase(int &item) {
        const int nend = p.nb;
        int n = 0;
        while (n < nend) {
            const int n1 = load_hq_batch(n, nend);
            run_B_batch(n, n1, item);
            cbar();   // the next batch overwrites hq
            n = n1;
        }
    }

    // Row tile rt of y belongs to block rt % G; its n-th tile goes to warp
    // n % 8.  Runs after the block's own B units.
    __device__ void finish_tiles() {
        int n = 0;
        for (int rt = c; rt < a.H / 32; rt += G, ++n)
            if ((n % LW) == warp) write_y(rt);
    }

    // y rows of one 32-row tile: slots in slot order, shared expert last.
    // A token's tagged o words are loaded, and re-read, together.
    __device__ void write_y(int rt) {
        const int row = rt * 32 + lane;
        for (int t = 0; t < a.T; ++t) {
            float y = 0.f;
            for (int s0 = 0; s0 < a.k; s0 += 8) {
                const int n = min(8, a.k - s0);
                tword w[8];
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {   // slots not owned here count as present
                    const int p = t * a.k + s0 + jj;
                    if (jj < n) w[jj] = pu()[p] >= 0 ? ld_tag(a.o_r + (size_t)p * a.H + row) : ((tword)ep << 32);
                }
                {   // re-read every missing word per round: one round trip each
                    bool all = true;
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj)
                        if (jj < n) all &= tag_of(w[jj]) == ep;
                    const long long t0 = clock64();
                    while (!all) {
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj) {
                            const int p = t * a.k + s0 + jj;
                            if (jj < n && tag_of(w[jj]) != ep) w[jj] = ld_tag(a.o_r + (size_t)p * a.H + row);
                        }
                        all = true;
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj)
                            if (jj < n) all &= tag_of(w[jj]) == ep;
                        if (!all && (m->abort || clock64() - t0 > a.wait_limit)) {
                            fail();
                            break;
                        }
                    }
                }
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const int p = t * a.k + s0 + jj;
                    if (jj < n && pu()[p] >= 0) y += wts()[p] * tag_value(w[jj]);
                }
            }
            if (a.shared) {
                const tword *ps = a.o_s + (size_t)t * a.H + row;
                const float os = tag_value(wait_tag(ps, ld_tag(ps)));
                y += a.shared_gate ? m->sgate[t] * os : os;
            }
            a.y[(size_t)t * a.H + row] = y;
        }
    }

    // ------------------------------------------------------ phases
    __device__ void init() {
        if (threadIdx.x == 0) {
            for (int i = 0; i < NBAR; ++i) mbar_init(full_bar(i), 1);
            for (int i = 0; i < NBAR; ++i) mbar_init(empty_bar(i), MAX_ITEM_RECS);
            mbar_init(fixed_bar(), 1);
            for (int b = 0; b < 2; ++b) {
                mbar_init(ready_bar(b), LW);
                mbar_init(free_bar(b), 1);
            }
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            m->abort = 0;
            m->spec_ready = 0;
        }
        for (int i = threadIdx.x; i < NBAR; i += LT) tags()[i] = 0xFFFFFFFFu;
        __syncthreads();
    }

    // router rows of this block (balanced contiguous range)
    __device__ void router_range(int &e0, int &e1) {
        e0 = (int)(((long long)c * a.E) / G);
        e1 = (int)(((long long)(c + 1) * a.E) / G);
    }

    // x into q8 records by consumer warps w0 .. LW-1
    __device__ void quantise_x(int w0) {
        const int chunks = (a.H + 255) / 256;
        for (int w = warp - w0; w < a.T * chunks; w += LW - w0) {
            const int t = w / chunks, ch = w - t * chunks;
            float v[8];
            const bool act = quant_load8<false>(a.x + (size_t)t * a.H, a.H, 256 * ch, lane, v);
            quant_store8(v, act, a.H, 256 * ch, xq(t), lane);
        }
    }

    // ep0: the block's launch counter as loaded by thread 0 (in flight until
    // the dots are done)
    __device__ void router_logits(uint32_t ep0) {
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
        if (threadIdx.x == 0) m->ep = ep0 + 1u;
        cbar();
        ep = m->ep;
        for (int it = threadIdx.x; it < nr * a.T; it += LW * 32) {
            const int r = it / a.T, t = it - r * a.T;
            float l = segv[(r * nseg) * a.T + t];
            for (int s = 1; s < nseg; ++s) l = __fadd_rn(l, segv[(r * nseg + s) * a.T + t]);
            if (a.rbias) l = __fadd_rn(l, a.rbias[e0 + r]);
            st_tag(a.logits + (size_t)t * a.E + e0 + r, l, ep);
        }
    }

    // k largest of E logits (largest first, lower index on equal logits) by one
    // warp: lane l holds keys of experts l + 32 j in registers; each round takes
    // the warp maximum key, then the lowest index holding it, and clears that
    // key.  No branch depends on the data (rounds are unrolled for the usual
    // k), which keeps the warp converged.  Writes the ids to out[0..k) and
    // returns, in lane s < k, the s-th selected logit.
    template <int JN>
    __device__ __forceinline__ void topk_round(uint32_t (&key)[JN], int s, int &myid, uint32_t &mykey) {
        uint32_t best = key[0];
        int bj = 0;
#pragma unroll
        for (int j = 1; j < JN; ++j) {
            const bool more = key[j] > best;
            best = more ? key[j] : best;
            bj = more ? j : bj;
        }
        const uint32_t mx = __reduce_max_sync(0xFFFFFFFFu, best);
        const int win = __reduce_min_sync(0xFFFFFFFFu, best == mx ? lane + 32 * bj : 0x7FFFFFFF);
        const bool mine = (win & 31) == lane;
#pragma unroll
        for (int j = 0; j < JN; ++j) key[j] = (mine && j == bj) ? 0u : key[j];
        myid = lane == s ? win : myid;
        mykey = lane == s ? mx : mykey;
    }
    template <int JN>
    __device__ float select_topk(const float *lg, int *out) {
        uint32_t key[JN];   // 0 marks padding (every real logit's key is > 0)
#pragma unroll
        for (int j = 0; j < JN; ++j) {
            const int e = lane + 32 * j;
            key[j] = e < a.E ? fkey(lg[e]) : 0u;
        }
        int myid = 0;
        uint32_t mykey = 0u;
        // rounds as a loop, not unrolled: this code runs once per launch and
        // fetching it cold costs more than the loop's own instructions
#pragma unroll 1
        for (int s = 0; s < a.k; ++s) topk_round<JN>(key, s, myid, mykey);
        if (lane < a.k) out[lane] = myid;
        return fkey_value(mykey);
    }

    // every logit into shared memory: thread i of n loads words i, i + n, ...
    // (up to 8 per round trip) and re-reads the ones not yet published
    __device__ void poll_logits(int i, int n) {
        float *lgs = reinterpret_cast<float *>(sm + o.lg);
        const int TE = a.T * a.E;
        for (int i0 = i; i0 < TE; i0 += 8 * n) {
            const int cnt = min(8, (TE - i0 + n - 1) / n);
            tword w[8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (q < cnt) w[q] = ld_tag(a.logits + i0 + q * n);
            {   // re-read every missing word per round: one round trip each
                bool all = true;
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (q < cnt) all &= tag_of(w[q]) == ep;
                const long long t0 = clock64();
                while (!all) {
                    __nanosleep(128);   // many blocks poll the same few lines: ease off between rounds
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        if (q < cnt && tag_of(w[q]) != ep) w[q] = ld_tag(a.logits + i0 + q * n);
                    all = true;
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        if (q < cnt) all &= tag_of(w[q]) == ep;
                    if (!all && (m->abort || clock64() - t0 > a.wait_limit)) {
                        fail();
                        break;
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (q < cnt) lgs[i0 + q * n] = tag_value(w[q]);
        }
    }
    // token t's top-k by the calling warp
    __device__ void topk_token(int t) {
        const float *lg = reinterpret_cast<const float *>(sm + o.lg) + (size_t)t * a.E;
        const float mysel = a.E <= 256 ? select_topk<8>(lg, ids() + t * a.k) : select_topk<32>(lg, ids() + t * a.k);
        if (lane < a.k) wts()[t * a.k + lane] = mysel;   // the weights replace these later
    }

    // After the logits are published: every logit read back, the top-k of
    // each token, x quantised (fp32 router; a Q8_0 router quantised it
    // before), then the grouping and the work plan.  One token: warp 0 reads
    // the logits and selects while the other warps quantise x.
    __device__ void route_tail(bool x_done) {
        // (one call site per step: every inlined copy is code each launch fetches)
        const bool split = NT == 1 && !x_done;
        if (!x_done && (!split || warp > 0)) quantise_x(split ? 1 : 0);
        if (a.shared_gate && warp == LW - 1)
            for (int t = 0; t < a.T; ++t) {
                const float s = shared_gate_weight(a.shared_gate, a.x + (size_t)t * a.H, a.H, lane);
                if (lane == 0) m->sgate[t] = s;
            }
        if (!split || warp == 0) poll_logits(split ? lane : threadIdx.x, split ? 32 : LW * 32);
        if (split) __syncwarp();
        else cbar();
        for (int t = warp; t < a.T; t += LW) topk_token(t);
        cbar();
        group();
    }

    // gating weights from the selected logits (after the expert streams started)
    __device__ void gating_weights() {
        const float *lgs = reinterpret_cast<const float *>(sm + o.lg);
        for (int t = warp; t < a.T; t += LW) {
            const float *lg = lgs + (size_t)t * a.E;
            const float mysel = lane < a.k ? wts()[t * a.k + lane] : 0.f;
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
            if (a.logits_out)
                for (int i = threadIdx.x; i < a.T * a.E; i += LW * 32) a.logits_out[i] = lgs[i];
            for (int i = threadIdx.x; i < a.P; i += LW * 32) {
                if (a.ids_out) a.ids_out[i] = ids()[i];
                if (a.w_out) a.w_out[i] = wts()[i];
            }
        }
    }

    // (token, slot) pairs grouped by owned expert, ascending ids, tokens
    // ascending; built by warp 0 alone (warp-synchronous, no block barriers)
    __device__ void group() {
        if (NT == 1 && warp == 0) {   // NT == 1: the launch has one token
            // one token: the k ids are distinct, each expert has one pair; the
            // unique list is the owned ids in ascending order
            const moe_expert *T = table();
            const int e = lane < a.k ? ids()[lane] : 0x7FFFFFFF;
            const bool own = lane < a.k && T[e].gate != nullptr;
            const unsigned ownm = __ballot_sync(0xFFFFFFFFu, own);
            int rank = 0;
            for (int j = 0; j < a.k; ++j) {
                const int ej = __shfl_sync(0xFFFFFFFFu, e, j);
                rank += ((ownm >> j) & 1u) && ej < e;
            }
            const int U = __popc(ownm);
            if (lane < a.k) pu()[lane] = own ? rank : -1;
            if (own) {
                ue()[rank] = e;
                umask()[rank] = 1u;
                uoff()[rank] = rank;
                plist()[rank] = lane;
            }
            if (lane == 0) { uoff()[U] = U; m->U = U; }
        } else if (NT != 1 && warp == 0) {
            const int nw = (a.E + 31) >> 5;
            m->bitmap[lane] = 0u;   // MOE_MAX_EXPERTS / 32 == 32 words
            __syncwarp();
            const moe_expert *T = table();
            // the selection gives k distinct ids per token: only ownership filters
            for (int t = 0; t < a.T; ++t)
                for (int s = lane; s < a.k; s += 32) {
                    const int p = t * a.k + s;
                    const int e = ids()[p];
                    const bool keep = T[e].gate != nullptr;
                    pu()[p] = keep ? e : -1;
                    if (keep) atomicOr(&m->bitmap[e >> 5], 1u << (e & 31));
                }
            __syncwarp();
            const int cnt = lane < nw ? __popc(m->bitmap[lane]) : 0;
            int inc = cnt;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int v = __shfl_up_sync(0xFFFFFFFFu, inc, off);
                if (lane >= off) inc += v;
            }
            m->wpre[lane] = inc - cnt;
            const int U = __shfl_sync(0xFFFFFFFFu, inc, 31);
            for (int u = lane; u < U; u += 32) umask()[u] = 0u;
            __syncwarp();
            for (int t = 0; t < a.T; ++t)
                for (int s = lane; s < a.k; s += 32) {
                    const int p = t * a.k + s;
                    const int e = pu()[p];
                    if (e < 0) continue;
                    const int u = m->wpre[e >> 5] + __popc(m->bitmap[e >> 5] & ((1u << (e & 31)) - 1u));
                    ue()[u] = e;
                    atomicOr(&umask()[u], 1u << t);
                    pu()[p] = u;
                }
            __syncwarp();
            int carry = 0;
            for (int base = 0; base < U; base += 32) {
                const int u = base + lane;
                const int c2 = u < U ? __popc(umask()[u]) : 0;
                int in2 = c2;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int v = __shfl_up_sync(0xFFFFFFFFu, in2, off);
                    if (lane >= off) in2 += v;
                }
                if (u < U) uoff()[u] = carry + in2 - c2;
                carry += __shfl_sync(0xFFFFFFFFu, in2, 31);
            }
            if (lane == 0) { uoff()[U] = carry; m->U = U; }
            __syncwarp();
            for (int t = 0; t < a.T; ++t)
                for (int s = lane; s < a.k; s += 32) {
                    const int p = t * a.k + s;
                    const int u = pu()[p];
                    if (u < 0) continue;
                    plist()[uoff()[u] + __popc(umask()[u] & ((1u << t) - 1u))] = p;
                }
        }
        cbar();
        // one token, every chosen expert owned: the producer made this plan
        // while the routing ran
        if (threadIdx.x == 0) {
            const bool use = NT == 1 && m->U == a.k && m->spec_ready;
            if (use) {
                __threadfence_block();   // the flag before the plan it publishes
                put_plan(m->spec);
            }
            m->use_spec = use ? 1 : 0;
        }
        cbar();
        if (!m->use_spec) plan();
        load_plan();
    }

    // unit counts and this block's B range: every block's A bytes follow from
    // the snake deal; block c gets the B units whose byte midpoints fall in
    // its share of what is left to reach the mean (integer bytes throughout,
    // so every block computes the same boundaries).  B ranges are contiguous,
    // so a block's B units need the h of one or two experts.  The blocks that
    // run the last A pass (one unit more than the rest) take the B units at
    // the end of the list, whose experts' h that pass completes; the others
    // take the experts finished by earlier passes, which their own earlier
    // finish lets them start at once.  So the B order over blocks runs
    // backwards when the last pass is a forward one.
    __device__ void plan() {
        const uint32_t sa = 2u * (uint32_t)(FS::tile_bytes(a.H) >> 7), ra = 2u * (uint32_t)(F::tile_bytes(a.H) >> 7);
        const uint32_t sb = a.shared ? (uint32_t)(FS::tile_bytes(a.Is) >> 7) : 0u, rb = (uint32_t)(F::tile_bytes(a.I) >> 7);
        const int tid = threadIdx.x;
        if (tid == 0) {
            SpecPlan s;
            closed_plan(m->U, s);
            put_plan(s);
        }
        cbar();
        if (!m->closed) {   // a block-wide scan of the clamped shares
            uint32_t my_a = 0;
            const int bc = m->brev ? G - 1 - tid : tid;   // the block at B position tid
            if (tid < G) {
                for (int pass = 0; pass * G < m->nA; ++pass) {
                    const int j = snake_unit(pass, bc, G);
                    if (j < m->n_sa) my_a += (uint32_t)a.balpha * sa;
                    else if (j < m->nA) my_a += (uint32_t)a.balpha * ra;
                }
            }
            const uint32_t b = (tid < G && m->target > my_a) ? m->target - my_a : 0u;
            uint32_t inc = b;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, inc, off);
                if (lane >= off) inc += v;
            }
            if (lane == 31) m->bsum[warp] = inc;
            cbar();
            uint32_t before = 0;
            for (int w = 0; w < warp; ++w) before += m->bsum[w];
            const uint32_t excl = before + inc - b;
            const int pos = m->brev ? G - 1 - c : c;   // this block's B position
            if (tid == pos) m->lo = excl;
            if (tid == pos + 1) m->hi = excl;
            cbar();
        }
        if (tid == 0 && !m->closed) {   // the range from the scanned shares
            const bool last = m->brev ? c == 0 : c + 1 == G;   // last in B order
            m->jb0 = first_b_unit(m->lo >> 2, sb, rb, m->n_sb, m->nB);
            m->jb1 = last ? m->nB : first_b_unit(m->hi >> 2, sb, rb, m->n_sb, m->nB);
            if (m->jb1 < m->jb0) m->jb1 = m->jb0;
            m->nb = m->jb1 - m->jb0;
        }
        cbar();
    }

    // The plan for U owned experts, by one thread: unit counts, the B order,
    // and - when no block's weighted A bytes exceed the mean share, so no
    // share needs clamping (s.closed) - this block's B range in closed form.
    // Bytes in 128-byte lines (every packed tile is a whole number of them),
    // shares in quarter lines: 32-bit integers throughout (the host refuses
    // shapes whose layer could reach 2^28 lines).
    __device__ void closed_plan(int U, SpecPlan &s) {
        const uint32_t sa = 2u * (uint32_t)(FS::tile_bytes(a.H) >> 7), ra = 2u * (uint32_t)(F::tile_bytes(a.H) >> 7);
        const uint32_t sb = a.shared ? (uint32_t)(FS::tile_bytes(a.Is) >> 7) : 0u, rb = (uint32_t)(F::tile_bytes(a.I) >> 7);
        const int n_sa = a.shared ? a.Is / 32 : 0;
        s.tilesI = a.I / 32;
        s.tilesIs = a.shared ? a.Is / 32 : 0;
        s.tilesH = a.H / 32;
        s.n_ra = U * s.tilesI;
        s.nA = n_sa + s.n_ra;
        s.n_sb = a.shared ? s.tilesH : 0;
        s.n_rb = U * s.tilesH;
        s.nB = s.n_sb + s.n_rb;
        // A bytes count a.balpha quarters in the balance: a block's B
        // records wait in its ring until its own A work is done, so its B
        // work lands mostly after its A work however the bytes are split
        const uint32_t aq = (uint32_t)a.balpha;
        const uint32_t tot = aq * ((uint32_t)n_sa * sa + (uint32_t)s.n_ra * ra) +
                             4u * ((uint32_t)s.n_sb * sb + (uint32_t)s.n_rb * rb);
        const uint32_t target = tot / (uint32_t)G + 1u;   // any fixed rule works: all blocks agree
        s.target = target;
        // block c's share starts at c * target - (weighted A bytes of blocks < c)
        const int npass = (s.nA + G - 1) / G;
        const uint32_t amax = aq * (uint32_t)npass * (sa > ra ? sa : ra);
        s.brev = npass > 0 && ((npass - 1) & 1) == 0;
        s.closed = amax <= target;
        s.lo = s.hi = 0u;
        s.jb0 = s.jb1 = s.nb = 0;
        if (!s.closed) return;
        if (s.brev) {   // B order G-1, ..., 0: the blocks above c come first
            const uint32_t atot = aq * a_before(G, sa, ra, n_sa, s.nA);
            s.lo = (uint32_t)(G - 1 - c) * target - (atot - aq * a_before(c + 1, sa, ra, n_sa, s.nA));
            s.hi = (uint32_t)(G - c) * target - (atot - aq * a_before(c, sa, ra, n_sa, s.nA));
        } else {
            s.lo = (uint32_t)c * target - aq * a_before(c, sa, ra, n_sa, s.nA);
            s.hi = (uint32_t)(c + 1) * target - aq * a_before(c + 1, sa, ra, n_sa, s.nA);
        }
        const bool last = s.brev ? c == 0 : c + 1 == G;   // last in B order
        s.jb0 = first_b_unit(s.lo >> 2, sb, rb, s.n_sb, s.nB);
        s.jb1 = last ? s.nB : first_b_unit(s.hi >> 2, sb, rb, s.n_sb, s.nB);
        if (s.jb1 < s.jb0) s.jb1 = s.jb0;
        s.nb = s.jb1 - s.jb0;
    }
    __device__ void put_plan(const SpecPlan &s) {
        m->tilesI = s.tilesI;
        m->tilesIs = s.tilesIs;
        m->tilesH = s.tilesH;
        m->n_ra = s.n_ra;
        m->nA = s.nA;
        m->n_sb = s.n_sb;
        m->n_rb = s.n_rb;
        m->nB = s.nB;
        m->brev = s.brev;
        m->closed = s.closed;
        m->target = s.target;
        m->lo = s.lo;
        m->hi = s.hi;
        m->jb0 = s.jb0;
        m->jb1 = s.jb1;
        m->nb = s.nb;
    }

    // A lines of blocks [0, c) under the snake deal: pass p gives them units
    // [pG, pG + c) (even p) or [pG + G - c, pG + G) (odd p); units below
    // n_sa are shared-expert units of sa lines, the rest up to nA routed of ra
    __device__ uint32_t a_before(int cc, uint32_t sa, uint32_t ra, int n_sa, int nA) {
        if (n_sa < G) {
            // closed form: every full pass gives each block one unit; the last,
            // partial pass (rem units) goes to blocks 0.. (forward) or ..G-1
            // (backward); the shared units are the first n_sa of pass 0
            const int P = nA / G, rem = nA - P * G;
            const int part = (P & 1) == 0 ? min(cc, rem) : max(0, cc - (G - rem));
            const int units = cc * P + part, sh = min(cc, n_sa);
            return sa * (uint32_t)sh + ra * (uint32_t)(units - sh);
        }
        auto span = [](int lo, int hi, int a0, int a1) -> uint32_t {
            const int l = lo > a0 ? lo : a0, h = hi < a1 ? hi : a1;
            return h > l ? (uint32_t)(h - l) : 0u;
        };
        uint32_t s = 0;
        for (int p = 0; p * G < nA; ++p) {
            const int lo = (p & 1) ? p * G + G - cc : p * G;
            s += sa * span(lo, lo + cc, 0, n_sa) + ra * span(lo, lo + cc, n_sa, nA);
        }
        return s;
    }

    // the n-th B unit of this block (global unit index)
    __device__ int b_unit(int n) {
        return p.nA + p.jb0 + n;
    }

    // first B unit whose midpoint is >= X (B list: shared units of sb lines,
    // then routed units of rb lines; midpoints in half lines)
    __device__ int first_b_unit(uint32_t X, uint32_t sb, uint32_t rb, int n_sb, int nB) {
        const uint32_t X2 = 2u * X;
        auto mid2 = [&](int j) -> uint32_t {
            return j < n_sb ? (2u * (uint32_t)j + 1u) * sb : 2u * (uint32_t)n_sb * sb + (2u * (uint32_t)(j - n_sb) + 1u) * rb;
        };
        int j;
        if (n_sb > 0 && X2 <= mid2(n_sb - 1)) j = (int)(X / sb);
        else j = n_sb + (int)((X > (uint32_t)n_sb * sb ? X - (uint32_t)n_sb * sb : 0u) / rb);
        if (j > nB) j = nB;
        while (j < nB && mid2(j) < X2) ++j;
        while (j > 0 && mid2(j - 1) >= X2) --j;
        return j;
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
        load_plan();   // the shared-expert A units; the rest follows the routing plan
        if (warp == LW) {
            producer();
        } else {
            consumer();
        }
        __syncthreads();
        finish();
    }

    __device__ void producer() {
        Ring R{0, 0, 0, evict_first_policy()};
        if (lane == 0) {
            // input-independent bytes: router rows, expert table, shared gate/up
            int e0, e1;
            router_range(e0, e1);
            const size_t rowb = a.rtype == MOE_F32 ? (size_t)a.H * 4 : (size_t)(a.H / 32) * 34;
            const uint32_t rbytes = (uint32_t)((e1 - e0) * rowb);
            const uint32_t tb = a.table_in_smem ? (uint32_t)(a.E * sizeof(moe_expert)) : 0u;
            if (rbytes + tb > 0) {
                mbar_arm(fixed_bar(), rbytes + tb);
                if (rbytes)
                    bulk_g2s_stream(sm + o.router, (const uint8_t *)a.w_router + (size_t)e0 * rowb, rbytes, fixed_bar(),
                                    R.pol);
                if (tb) bulk_g2s(sm + o.table, a.experts, tb, fixed_bar());
            }
        }
        // this block's shared-expert units (its first snake passes): the
        // consumers run them while the routing completes, freeing the ring
        if (lane == 0) {
            for (int pass = 0; pass * G < p.n_sa && !m->abort; ++pass) {
                const int j = snake_unit(pass, c, G);
                if (j < p.n_sa && !issue_unit(R, j)) break;
            }
        }
        if (NT == 1 && lane == 0 && !m->abort) {   // the plan for U = k, off the routing path
            SpecPlan s;
            closed_plan(a.k, s);
            if (s.closed) {
                m->spec = s;
                __threadfence_block();
                m->spec_ready = 1;
            }
        }
        if (lane == 0 && a.shared) m->shx = *a.shared;   // for units after the handoff
        __syncthreads();   // routing handoff: the plan is ready
        shp = &m->shx;
        load_plan();
        if (lane == 0 && !m->abort) {
            for (int pass = 0; pass * G < p.nA; ++pass) {   // the routed units
                const int j = snake_unit(pass, c, G);
                if (j >= p.n_sa && j < p.nA && !issue_unit(R, j)) break;
            }
            for (int n = 0; n < p.nb && !m->abort; ++n)
                if (!issue_unit(R, b_unit(n))) break;
        }
        // drain: no copy may still be writing this block's shared memory at exit
        if (lane == 0) {
            for (int i = R.tail; i < R.issued; ++i) mbar_wait(full_bar(i), (uint32_t)((i / NBAR) & 1));
        }
        __syncwarp();
    }

    __device__ void consumer() {
        // the block's launch counter and (one block) the hidden rows into L2
        // while the previous kernel runs
        if (threadIdx.x == 0) prefetch_l2(a.epoch + c);
        if (c == 0)
            for (int i = 32 * threadIdx.x; i < a.T * a.H; i += 32 * 32 * LW) prefetch_l2(a.x + i);
        pdl_wait();
        // This launch's epoch: the block's own counter + 1.  Every block
        // advances its counter once per launch (finish), so all blocks agree
        // without a shared count; the next launch reads it only after this
        // grid is done.  The load is consumed after the router dots.
        uint32_t ep0 = 0;
        if (threadIdx.x == 0) ep0 = ld_relaxed_u32(a.epoch + c);
        // an fp32 router needs only x: its logits go out first and x is
        // quantised while the other blocks publish theirs; a Q8_0 router dots
        // the quantised x (router_logits' barrier orders it before the dots)
        const bool xq_first = a.rtype == MOE_Q8_0;
        if (xq_first) quantise_x(0);
        router_logits(ep0);
        // the shared expert's gate/up units while the other blocks publish
        // their logits (x quantised first)
        bool x_done = xq_first;
        int item = 0, ua = 0;
        if (p.n_sa > 0) {
            if (!x_done) {
                quantise_x(0);
                cbar();
                x_done = true;
            }
            for (int pass = 0; pass * G < p.n_sa; ++pass) {
                const int j = snake_unit(pass, c, G);
                if (j < p.n_sa) {
                    Unit U;
                    unit_of(j, U);
                    run_A<FS>(U, item, ua);
                }
            }
        }
        route_tail(x_done);
        if (c == 0 && a.xq_out) {
            const int n16 = (int)(a.xrec / 16);
            for (int i = threadIdx.x; i < a.T * n16; i += LW * 32)
                reinterpret_cast<uint4 *>(a.xq_out)[i] = reinterpret_cast<const uint4 *>(sm + o.xq)[i];
        }
        bar_handoff();
        gating_weights();
        for (int pass = 0; pass * G < p.nA; ++pass) {   // the routed A units
            const int j = snake_unit(pass, c, G);
            if (j >= p.n_sa && j < p.nA) {
                Unit U;
                unit_of(j, U);
                run_A<F>(U, item, ua);
            }
        }
        // no loop below leaves early: every consumer thread must reach every
        // named barrier; after a timeout only waits and sums are skipped
        run_B_phase(item);
        finish_tiles();
    }

    // the handoff barrier pairs with the producer's __syncthreads
    __device__ void bar_handoff() {
        __syncthreads();
        shp = &m->shx;
    }

    __device__ void finish() {
        if (threadIdx.x == 0) st_relaxed_u32(a.epoch + c, m->ep);
    }
};

// one block per SM: the whole register file is the block's (17 warps: five
// share one SM sub-partition's 16K registers, so 96 per thread; 9 warps: 224)
template <class F, class FS, int NT>
__global__ void __launch_bounds__(Warps<NT>::LT, 1) layer_kernel(const __grid_constant__ LayerArgs a) {
    LayerKernel<F, FS, NT> K(a, moe_smem);
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
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, layer_kernel<F, FS, NT>, Warps<NT>::LT, smem);
        if (e != cudaSuccess) return e;
        if (n < 1) return cudaErrorInvalidConfiguration;   // one block per SM must fit
        occ_ok[dev] = (int)smem + 1;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)G);
    cfg.blockDim = dim3(Warps<NT>::LT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    // Not a cooperative launch: with that attribute a launch starts only once
    // the previous kernel has left every SM, which undoes the overlap below.
    // Co-residency of the blocks is assumed (one block per SM fits, checked
    // above); a block kept off its SM by other work makes the others' waits
    // run into their bound (MOE_DEV_TIMEOUT), it does not hang.
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
    return cudaErrorNotSupported;
}

}  // namespace moe
