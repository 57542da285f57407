// moe_common.cuh - device-side building blocks shared by the MoE kernels:
// q8 activation record geometry, the packed weight formats (one lane = one
// row of a 32-row tile) and their exact integer sub-block dots.
//
// Formats follow the pulsar README's list of routed-expert quant types
// (q8_0, q4_K, q2_K) and gpt-oss's MXFP4 experts (model table); the block
// fields are the GGUF ones.  The integer dots are the README's "ds4 exact
// math": int8 activation codes times integer weight codes, rescaled per
// block ("MoE resolve" passage; the mmq note on per-quant-block rescale).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>
#include <stddef.h>

#include "moe.h"

namespace moe {

constexpr int WARP = 32;

// Raises a kernel's dynamic shared memory limit only when a launch needs more
// than the last value set (per device), so steady-state launches, including
// those recorded into a CUDA graph, make no attribute calls.
template <auto kernel>
inline cudaError_t ensure_smem(size_t bytes) {
    static int set_bytes[64] = {0};   // one table per kernel
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if ((int)bytes <= set_bytes[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) set_bytes[dev] = (int)bytes;
    return e;
}

// ----------------------------------------------------- activation records

__host__ __device__ inline int act_block(int n) {
    return (n > 0 && n % 256 == 0) ? 256 : ((n > 0 && n % 32 == 0) ? 32 : 0);
}
__host__ __device__ inline size_t q8_q_off(int n) {
    return ((size_t)4 * (n / act_block(n)) + 15) & ~(size_t)15;
}
__host__ __device__ inline size_t q8_bs_off(int n) { return q8_q_off(n) + (size_t)n; }
__host__ __device__ inline size_t q8_row_bytes(int n) {
    if (!act_block(n)) return 0;
    return (q8_bs_off(n) + 2 * (size_t)(n / 16) + 15) & ~(size_t)15;
}

// One token's q8 record as seen by a dot: codes q[n], per-block d, per-16 sums.
struct Act {
    const float *d;
    const int8_t *q;
    const int16_t *bs;
    int lgB;  // log2 of the activation block (8 or 5)
};

__device__ __forceinline__ Act act_view(const uint8_t *rec, int n) {
    Act a;
    a.d = reinterpret_cast<const float *>(rec);
    a.q = reinterpret_cast<const int8_t *>(rec + q8_q_off(n));
    a.bs = reinterpret_cast<const int16_t *>(rec + q8_bs_off(n));
    a.lgB = act_block(n) == 256 ? 8 : 5;
    return a;
}

// ------------------------------------------------------------ primitives

__device__ __forceinline__ float h2f(uint32_t bits) {
    return __half2float(__ushort_as_half((unsigned short)(bits & 0xFFFFu)));
}

// streaming 128-bit load of weight bytes (read once per call: no L1 allocation)
__device__ __forceinline__ uint4 ldg_stream(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg_stream32(const void *p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ldg_stream64(const void *p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

// generic-mode byte permute: a selector nibble with bit 3 set replicates the
// sign bit of the selected byte instead of copying it
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ int dp4a(uint32_t a, uint32_t b, int c) {
    return __dp4a((int)a, (int)b, c);
}
// c + sum over the four byte lanes of a (unsigned) times b (signed): lets a
// code field be masked in place (the dot of 2^s x code) instead of shifted
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// c + a.lo16 * b.byte0 + a.hi16 * b.byte1 (lo), or times b.byte2, b.byte3 (hi);
// a's halves signed, b's bytes unsigned.  Two int16 block sums of the
// activation record times two unsigned scale bytes in one instruction.
__device__ __forceinline__ int dp2a_lo(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp2a_hi(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.hi.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ int4 lds128(const int8_t *p) { return *reinterpret_cast<const int4 *>(p); }

__device__ __forceinline__ uint32_t saddr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint4 lds_u4(const void *p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(saddr(p)));
    return v;
}
__device__ __forceinline__ uint2 lds_u2(const void *p) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(saddr(p)));
    return v;
}
__device__ __forceinline__ uint32_t lds_u1(const void *p) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(saddr(p)));
    return v;
}

__device__ __forceinline__ uint32_t byte_of(uint32_t w, int i) { return (w >> (8 * i)) & 0xFFu; }

// ------------------------------------------------------------------ Q4_K
// record = one 256-column block per row; 9 planes of 16 B (the GGUF block
// cut into 16-byte chunks: chunk 0 = d, dmin, 12 scale bytes; 1..8 = qs).
struct FQ4K {
    static constexpr int QK = 256;
    static constexpr int NSUB = 8;
    static constexpr int REC = 9 * 512;
    struct W { uint4 c[9]; };
    __host__ __device__ static int nrec(int cols) { return cols / 256; }
    __host__ __device__ static size_t rec_off(int, int r) { return (size_t)r * REC; }
    __host__ __device__ static size_t tile_bytes(int cols) { return (size_t)(cols / 256) * REC; }
    __device__ static void load(W &w, const uint8_t *rec, int, int lane) {
#pragma unroll
        for (int p = 0; p < 9; ++p) w.c[p] = ldg_stream(rec + p * 512 + lane * 16);
    }
    __device__ static void load_s(W &w, const uint8_t *rec, int, int lane) {
#pragma unroll
        for (int p = 0; p < 9; ++p) w.c[p] = lds_u4(rec + p * 512 + lane * 16);
    }
    __host__ __device__ static uint32_t rec_bytes(int, int) { return REC; }
    // exact sub-block dots: is[j] = sum over the 32 elements of sub-block j
    __host__ __device__ static int rec_blocks(int, int) { return 8; }
    __device__ static void isums(const W &w, const Act &a, int k0, int, int *is) {
        const int8_t *x = a.q + k0;
#pragma unroll
        for (int j = 0; j < 8; ++j) is[j] = 0;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const int g = c >> 1, h = c & 1;
            const int4 xl = lds128(x + 64 * g + 16 * h);
            const int4 xh = lds128(x + 64 * g + 32 + 16 * h);
            const uint4 q = w.c[1 + c];
            is[2 * g] = dp4a(q.x & 0x0F0F0F0Fu, (uint32_t)xl.x, is[2 * g]);
            is[2 * g] = dp4a(q.y & 0x0F0F0F0Fu, (uint32_t)xl.y, is[2 * g]);
            is[2 * g] = dp4a(q.z & 0x0F0F0F0Fu, (uint32_t)xl.z, is[2 * g]);
            is[2 * g] = dp4a(q.w & 0x0F0F0F0Fu, (uint32_t)xl.w, is[2 * g]);
            // high nibbles masked in place: the bytes are 16 x code
            is[2 * g + 1] = dp4a_us(q.x & 0xF0F0F0F0u, (uint32_t)xh.x, is[2 * g + 1]);
            is[2 * g + 1] = dp4a_us(q.y & 0xF0F0F0F0u, (uint32_t)xh.y, is[2 * g + 1]);
            is[2 * g + 1] = dp4a_us(q.z & 0xF0F0F0F0u, (uint32_t)xh.z, is[2 * g + 1]);
            is[2 * g + 1] = dp4a_us(q.w & 0xF0F0F0F0u, (uint32_t)xh.w, is[2 * g + 1]);
        }
#pragma unroll
        for (int g = 0; g < 4; ++g) is[2 * g + 1] >>= 4;   // exact: a multiple of 16
    }
    // d_x * (d * sum_j sc_j is_j - dmin * sum_j m_j bsum32_j)
    __device__ static float combine(const W &w, const Act &a, int k0, int, const int *is) {
        const uint32_t s0 = w.c[0].y, s1 = w.c[0].z, s2 = w.c[0].w;
        const uint32_t sc03 = s0 & 0x3F3F3F3Fu, m03 = s1 & 0x3F3F3F3Fu;
        const uint32_t sc47 = (s2 & 0x0F0F0F0Fu) | ((s0 >> 2) & 0x30303030u);
        const uint32_t m47 = ((s2 >> 4) & 0x0F0F0F0Fu) | ((s1 >> 2) & 0x30303030u);
        int P = 0, M = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) P += (int)byte_of(sc03, j) * is[j] + (int)byte_of(sc47, j) * is[4 + j];
        // sum_j m_j * (the two 16-element block sums of sub-block j): word j
        // of the block-sum array holds that pair as int16, so one dp2a takes
        // a sub-block against its min byte, replicated into the byte pair
        const int8_t *bs = reinterpret_cast<const int8_t *>(a.bs + (k0 >> 4));
        const int4 b03 = lds128(bs), b47 = lds128(bs + 16);
        const uint32_t m01 = prmt(m03, 0, 0x1100u), m23 = prmt(m03, 0, 0x3322u);
        const uint32_t m45 = prmt(m47, 0, 0x1100u), m67 = prmt(m47, 0, 0x3322u);
        M = dp2a_lo((uint32_t)b03.x, m01, M);
        M = dp2a_hi((uint32_t)b03.y, m01, M);
        M = dp2a_lo((uint32_t)b03.z, m23, M);
        M = dp2a_hi((uint32_t)b03.w, m23, M);
        M = dp2a_lo((uint32_t)b47.x, m45, M);
        M = dp2a_hi((uint32_t)b47.y, m45, M);
        M = dp2a_lo((uint32_t)b47.z, m67, M);
        M = dp2a_hi((uint32_t)b47.w, m67, M);
        const float d = h2f(w.c[0].x), dmin = h2f(w.c[0].x >> 16);
        const float dx = a.d[k0 >> a.lgB];
        return dx * (d * (float)P - dmin * (float)M);
    }
};

// ------------------------------------------------------------------ Q2_K
// record = one 256-column block per row: planes 0..4 = bytes [16p, 16p+16)
// (scales, qs), then a 128-byte plane holding {d, dmin} per row.
struct FQ2K {
    static constexpr int QK = 256;
    static constexpr int NSUB = 16;
    static constexpr int REC = 5 * 512 + 128;
    struct W { uint4 s; uint4 q[4]; uint32_t dd; };
    __host__ __device__ static int nrec(int cols) { return cols / 256; }
    __host__ __device__ static size_t rec_off(int, int r) { return (size_t)r * REC; }
    __host__ __device__ static size_t tile_bytes(int cols) { return (size_t)(cols / 256) * REC; }
    __device__ static void load(W &w, const uint8_t *rec, int, int lane) {
        w.s = ldg_stream(rec + lane * 16);
#pragma unroll
        for (int p = 0; p < 4; ++p) w.q[p] = ldg_stream(rec + (1 + p) * 512 + lane * 16);
        w.dd = ldg_stream32(rec + 5 * 512 + lane * 4);
    }
    __device__ static void load_s(W &w, const uint8_t *rec, int, int lane) {
        w.s = lds_u4(rec + lane * 16);
#pragma unroll
        for (int p = 0; p < 4; ++p) w.q[p] = lds_u4(rec + (1 + p) * 512 + lane * 16);
        w.dd = lds_u1(rec + 5 * 512 + lane * 4);
    }
    __host__ __device__ static uint32_t rec_bytes(int, int) { return REC; }
    __host__ __device__ static int rec_blocks(int, int) { return 8; }
    __device__ static void isums(const W &w, const Act &a, int k0, int, int *is) {
        const int8_t *x = a.q + k0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int n = c >> 1, h = c & 1;
            const uint4 q = w.q[c];
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const int4 xv = lds128(x + 128 * n + 32 * s + 16 * h);
                // field s masked in place: the bytes are 4^s x code
                const uint32_t mk = 0x03030303u << (2 * s);
                int acc = 0;
                acc = dp4a_us(q.x & mk, (uint32_t)xv.x, acc);
                acc = dp4a_us(q.y & mk, (uint32_t)xv.y, acc);
                acc = dp4a_us(q.z & mk, (uint32_t)xv.z, acc);
                acc = dp4a_us(q.w & mk, (uint32_t)xv.w, acc);
                is[8 * n + 2 * s + h] = acc >> (2 * s);   // exact: a multiple of 4^s
            }
        }
    }
    __device__ static float combine(const W &w, const Act &a, int k0, int, const int *is) {
        const uint32_t sw[4] = {w.s.x, w.s.y, w.s.z, w.s.w};
        // block sums of the 16 sub-blocks as 8 words of int16 pairs
        const int8_t *bs = reinterpret_cast<const int8_t *>(a.bs + (k0 >> 4));
        const int4 b0 = lds128(bs), b1 = lds128(bs + 16);
        const uint32_t bw[8] = {(uint32_t)b0.x, (uint32_t)b0.y, (uint32_t)b0.z, (uint32_t)b0.w,
                                (uint32_t)b1.x, (uint32_t)b1.y, (uint32_t)b1.z, (uint32_t)b1.w};
        int P = 0, M = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            // scale byte j = 4q + t: low nibble scale, high nibble min
            const uint32_t sc = sw[q] & 0x0F0F0F0Fu, mn = (sw[q] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
            for (int t = 0; t < 4; ++t) P += (int)prmt(sc, 0, 0x4440u + t) * is[4 * q + t];
            M = dp2a_lo(bw[2 * q], mn, M);
            M = dp2a_hi(bw[2 * q + 1], mn, M);
        }
        const float d = h2f(w.dd), dmin = h2f(w.dd >> 16);
        const float dx = a.d[k0 >> a.lgB];
        return dx * (d * (float)P - dmin * (float)M);
    }
};

// ------------------------------------------------------------------ Q8_0
// record = 8 blocks (256 columns) per row: planes 2b, 2b+1 = the 32 codes of
// block b, plane 16 = the 8 f16 scales.
struct FQ80 {
    static constexpr int QK = 256;
    static constexpr int NSUB = 8;   // one isum per 32-block
    static constexpr int REC = 17 * 512;
    struct W { uint4 q[16]; uint4 d; };
    __host__ __device__ static int nrec(int cols) { return cols / 256; }
    __host__ __device__ static size_t rec_off(int, int r) { return (size_t)r * REC; }
    __host__ __device__ static size_t tile_bytes(int cols) { return (size_t)(cols / 256) * REC; }
    __device__ static void load(W &w, const uint8_t *rec, int, int lane) {
#pragma unroll
        for (int p = 0; p < 16; ++p) w.q[p] = ldg_stream(rec + p * 512 + lane * 16);
        w.d = ldg_stream(rec + 16 * 512 + lane * 16);
    }
    __device__ static void load_s(W &w, const uint8_t *rec, int, int lane) {
#pragma unroll
        for (int p = 0; p < 16; ++p) w.q[p] = lds_u4(rec + p * 512 + lane * 16);
        w.d = lds_u4(rec + 16 * 512 + lane * 16);
    }
    __host__ __device__ static uint32_t rec_bytes(int, int) { return REC; }
    __host__ __device__ static int rec_blocks(int, int) { return 8; }
    __device__ static void isums(const W &w, const Act &a, int k0, int, int *is) {
        const int8_t *x = a.q + k0;
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            const int4 x0 = lds128(x + 32 * b), x1 = lds128(x + 32 * b + 16);
            const uint4 q0 = w.q[2 * b], q1 = w.q[2 * b + 1];
            int acc = 0;
            acc = dp4a(q0.x, (uint32_t)x0.x, acc);
            acc = dp4a(q0.y, (uint32_t)x0.y, acc);
            acc = dp4a(q0.z, (uint32_t)x0.z, acc);
            acc = dp4a(q0.w, (uint32_t)x0.w, acc);
            acc = dp4a(q1.x, (uint32_t)x1.x, acc);
            acc = dp4a(q1.y, (uint32_t)x1.y, acc);
            acc = dp4a(q1.z, (uint32_t)x1.z, acc);
            acc = dp4a(q1.w, (uint32_t)x1.w, acc);
            is[b] = acc;
        }
    }
    __device__ static float combine(const W &w, const Act &a, int k0, int, const int *is) {
        const uint32_t dw[4] = {w.d.x, w.d.y, w.d.z, w.d.w};
        float acc = 0.f;
        if (a.lgB == 8) {
#pragma unroll
            for (int b = 0; b < 8; ++b) acc += h2f(dw[b >> 1] >> (16 * (b & 1))) * (float)is[b];
            return a.d[k0 >> 8] * acc;
        }
#pragma unroll
        for (int b = 0; b < 8; ++b)
            acc += h2f(dw[b >> 1] >> (16 * (b & 1))) * a.d[(k0 >> 5) + b] * (float)is[b];
        return acc;
    }
};

// ----------------------------------------------------------------- MXFP4
// record = nb <= 8 blocks per row: planes b = the 16 code bytes of block b,
// then a 256-byte plane with the 8 E8M0 scale bytes of each row.  Integer
// lattice v = 2 * E2M1 value; byte permutes look magnitudes up from a table
// and split positive from negative codes (bit 3 = sign).  The permute visits
// elements in the order (j, j+16, j+1, j+17) of each code word, so the
// activation codes are read in the same interleaved order.
struct FMX4 {
    static constexpr int QK = 256;    // 8 blocks per full record
    static constexpr int NSUB = 8;
    struct W { uint4 q[8]; uint2 e; };
    __host__ __device__ static int nrec(int cols) { return (cols / 32 + 7) / 8; }
    __host__ __device__ static int rec_blocks(int cols, int r) {
        int nb = cols / 32 - 8 * r;
        return nb > 8 ? 8 : nb;
    }
    __host__ __device__ static size_t rec_off(int cols, int r) {
        (void)cols;
        return (size_t)r * (8 * 512 + 256);
    }
    __host__ __device__ static size_t tile_bytes(int cols) {
        int nb = cols / 32;
        return (size_t)(nb / 8) * (8 * 512 + 256) + ((nb % 8) ? (size_t)(nb % 8) * 512 + 256 : 0);
    }
    __device__ static void load(W &w, const uint8_t *rec, int nb, int lane) {
#pragma unroll
        for (int b = 0; b < 8; ++b)
            if (b < nb) w.q[b] = ldg_stream(rec + b * 512 + lane * 16);
        w.e = ldg_stream64(rec + nb * 512 + lane * 8);
    }
    __device__ static void load_s(W &w, const uint8_t *rec, int nb, int lane) {
#pragma unroll
        for (int b = 0; b < 8; ++b)
            if (b < nb) w.q[b] = lds_u4(rec + b * 512 + lane * 16);
        w.e = lds_u2(rec + nb * 512 + lane * 8);
    }
    __host__ __device__ static uint32_t rec_bytes(int cols, int r) { return (uint32_t)rec_blocks(cols, r) * 512 + 256; }
    // magnitudes 0,1,2,3 | 4,6,8,12 of the doubled E2M1 lattice
    static constexpr uint32_t LUT0 = 0x03020100u, LUT1 = 0x0C080604u;
    // codes of one 32-block: is = sum v_i * x_i; x points at the block's codes
    __device__ static int block_dot(const uint4 &q, const int8_t *x) {
        // interleave activations to the permute order (j, j+16, j+1, j+17)
        const int4 xa = lds128(x), xb = lds128(x + 16);
        const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
        const uint32_t xaw[4] = {(uint32_t)xa.x, (uint32_t)xa.y, (uint32_t)xa.z, (uint32_t)xa.w};
        const uint32_t xbw[4] = {(uint32_t)xb.x, (uint32_t)xb.y, (uint32_t)xb.z, (uint32_t)xb.w};
        int pos = 0, neg = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t wq = qw[k], wn = wq ^ 0x88888888u;
            const uint32_t x0 = __byte_perm(xaw[k], xbw[k], 0x5140);
            const uint32_t x1 = __byte_perm(xaw[k], xbw[k], 0x7362);
            // positive codes: magnitude; negative codes: bit 3 set -> sign of a
            // table byte (all zero) -> 0.  Flipped codes give the converse.
            // prmt reads only the low four selector nibbles, so the low half
            // of a code word needs no mask.
            pos = dp4a(prmt(LUT0, LUT1, wq), x0, pos);
            pos = dp4a(prmt(LUT0, LUT1, wq >> 16), x1, pos);
            neg = dp4a(prmt(LUT0, LUT1, wn), x0, neg);
            neg = dp4a(prmt(LUT0, LUT1, wn >> 16), x1, neg);
        }
        return pos - neg;
    }
    __device__ static void isums(const W &w, const Act &a, int k0, int nb, int *is) {
#pragma unroll
        for (int b = 0; b < 8; ++b)
            if (b < nb) is[b] = block_dot(w.q[b], a.q + k0 + 32 * b);
    }
    __device__ static float scale(uint32_t e) {
        // 2^(e-128): e >= 2 is a normal float with biased exponent e-1
        return e >= 2u ? __uint_as_float((e - 1u) << 23) : ldexpf(1.f, (int)e - 128);
    }
    __device__ static float combine(const W &w, const Act &a, int k0, int nb, const int *is) {
        float acc = 0.f;
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            if (b < nb) {
                const uint32_t e = byte_of(b < 4 ? w.e.x : w.e.y, b & 3);
                acc += scale(e) * a.d[(k0 + 32 * b) >> a.lgB] * (float)is[b];
            }
        }
        return acc;
    }
};

// ------------------------------------------------------------------ Q6_K
// record = one 256-column block per row: planes 0..12 = the block's bytes
// [16p, 16p+16) (0..7: ql, 8..11: qh, 12: the 16 int8 scales), then a
// 128-byte plane with d (f16 and two zero bytes) per row.  Element
// i = 128n + 32s + l has its low nibble in ql[64n + 32(s%2) + l] (the high
// nibble for s >= 2) and its top two bits at bits 2s of qh[32n + l]; the
// stored 6-bit code u is the weight code + 32.  With 16-sub-blocks j = i/16,
// isum_j = dot(u, x) - 32 * bsum_j (the signed codes' exact dot).
struct FQ6K {
    static constexpr int QK = 256;
    static constexpr int NSUB = 16;
    static constexpr int REC = 13 * 512 + 128;
    struct W { uint4 ql[8]; uint4 qh[4]; uint4 sc; uint32_t d; };
    __host__ __device__ static int nrec(int cols) { return cols / 256; }
    __host__ __device__ static size_t rec_off(int, int r) { return (size_t)r * REC; }
    __host__ __device__ static size_t tile_bytes(int cols) { return (size_t)(cols / 256) * REC; }
    __host__ __device__ static uint32_t rec_bytes(int, int) { return REC; }
    __host__ __device__ static int rec_blocks(int, int) { return 8; }
    __device__ static void load(W &w, const uint8_t *rec, int, int lane) {
#pragma unroll
        for (int p = 0; p < 8; ++p) w.ql[p] = ldg_stream(rec + p * 512 + lane * 16);
#pragma unroll
        for (int p = 0; p < 4; ++p) w.qh[p] = ldg_stream(rec + (8 + p) * 512 + lane * 16);
        w.sc = ldg_stream(rec + 12 * 512 + lane * 16);
        w.d = ldg_stream32(rec + 13 * 512 + lane * 4);
    }
    __device__ static void load_s(W &w, const uint8_t *rec, int, int lane) {
#pragma unroll
        for (int p = 0; p < 8; ++p) w.ql[p] = lds_u4(rec + p * 512 + lane * 16);
#pragma unroll
        for (int p = 0; p < 4; ++p) w.qh[p] = lds_u4(rec + (8 + p) * 512 + lane * 16);
        w.sc = lds_u4(rec + 12 * 512 + lane * 16);
        w.d = lds_u1(rec + 13 * 512 + lane * 4);
    }
    __device__ static uint32_t wd(const uint4 &v, int i) { return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w)); }
    __device__ static void isums(const W &w, const Act &a, int k0, int, int *is) {
        const int8_t *x = a.q + k0;
        const int16_t *bs = a.bs + (k0 >> 4);
#pragma unroll
        for (int n = 0; n < 2; ++n) {
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const int4 xa = lds128(x + 128 * n + 32 * s), xb = lds128(x + 128 * n + 32 * s + 16);
                const uint32_t xw[8] = {(uint32_t)xa.x, (uint32_t)xa.y, (uint32_t)xa.z, (uint32_t)xa.w,
                                        (uint32_t)xb.x, (uint32_t)xb.y, (uint32_t)xb.z, (uint32_t)xb.w};
                int acc0 = 0, acc1 = 0;
#pragma unroll
                for (int wl = 0; wl < 8; ++wl) {
                    const uint32_t q = wd(w.ql[4 * n + 2 * (s & 1) + (wl >> 2)], wl & 3);
                    const uint32_t h = wd(w.qh[2 * n + (wl >> 2)], wl & 3);
                    const uint32_t lo = (s >= 2 ? (q >> 4) : q) & 0x0F0F0F0Fu;
                    const uint32_t u = lo | (((h >> (2 * s)) & 0x03030303u) << 4);
                    if (wl < 4) acc0 = dp4a(u, xw[wl], acc0);
                    else acc1 = dp4a(u, xw[wl], acc1);
                }
                const int j = 8 * n + 2 * s;
                is[j] = acc0 - 32 * (int)bs[j];
                is[j + 1] = acc1 - 32 * (int)bs[j + 1];
            }
        }
    }
    // d_x * d * sum_j sc_j is_j
    __device__ static float combine(const W &w, const Act &a, int k0, int, const int *is) {
        const uint32_t sw[4] = {w.sc.x, w.sc.y, w.sc.z, w.sc.w};
        int P = 0;
#pragma unroll
        for (int j = 0; j < 16; ++j) P += (int)(int8_t)byte_of(sw[j >> 2], j & 3) * is[j];
        const float d = h2f(w.d);
        const float dx = a.d[k0 >> a.lgB];
        return dx * (d * (float)P);
    }
};

// ------------------------------------------------------------------ Q3_K
// record = one 256-column block per row: planes 0..1 = hmask, 2..5 = qs,
// plane 6 = the 12 scale bytes, d (f16) and two zero bytes.  Element
// i = 128n + 32s + l takes two bits at bits 2s of qs[32n + l] and bit
// 4n + s of hmask[l]; u = low + 4 * bit is the weight code + 4.  With
// 16-sub-blocks j, isum_j = dot(u, x) - 4 * bsum_j.  Scale j: 6 bits, low
// nibble in byte j (j < 8) or the high nibble of byte j - 8, top two bits at
// bit 2(j/4) of byte 8 + j%4, offset by 32.
struct FQ3K {
    static constexpr int QK = 256;
    static constexpr int NSUB = 16;
    static constexpr int REC = 7 * 512;
    struct W { uint4 hm[2]; uint4 qs[4]; uint4 sd; };
    __host__ __device__ static int nrec(int cols) { return cols / 256; }
    __host__ __device__ static size_t rec_off(int, int r) { return (size_t)r * REC; }
    __host__ __device__ static size_t tile_bytes(int cols) { return (size_t)(cols / 256) * REC; }
    __host__ __device__ static uint32_t rec_bytes(int, int) { return REC; }
    __host__ __device__ static int rec_blocks(int, int) { return 8; }
    __device__ static void load(W &w, const uint8_t *rec, int, int lane) {
#pragma unroll
        for (int p = 0; p < 2; ++p) w.hm[p] = ldg_stream(rec + p * 512 + lane * 16);
#pragma unroll
        for (int p = 0; p < 4; ++p) w.qs[p] = ldg_stream(rec + (2 + p) * 512 + lane * 16);
        w.sd = ldg_stream(rec + 6 * 512 + lane * 16);
    }
    __device__ static void load_s(W &w, const uint8_t *rec, int, int lane) {
#pragma unroll
        for (int p = 0; p < 2; ++p) w.hm[p] = lds_u4(rec + p * 512 + lane * 16);
#pragma unroll
        for (int p = 0; p < 4; ++p) w.qs[p] = lds_u4(rec + (2 + p) * 512 + lane * 16);
        w.sd = lds_u4(rec + 6 * 512 + lane * 16);
    }
    __device__ static void isums(const W &w, const Act &a, int k0, int, int *is) {
        const int8_t *x = a.q + k0;
        const int16_t *bs = a.bs + (k0 >> 4);
#pragma unroll
        for (int n = 0; n < 2; ++n) {
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const int4 xa = lds128(x + 128 * n + 32 * s), xb = lds128(x + 128 * n + 32 * s + 16);
                const uint32_t xw[8] = {(uint32_t)xa.x, (uint32_t)xa.y, (uint32_t)xa.z, (uint32_t)xa.w,
                                        (uint32_t)xb.x, (uint32_t)xb.y, (uint32_t)xb.z, (uint32_t)xb.w};
                int acc0 = 0, acc1 = 0;
#pragma unroll
                for (int wl = 0; wl < 8; ++wl) {
                    const uint32_t q = FQ6K::wd(w.qs[2 * n + (wl >> 2)], wl & 3);
                    const uint32_t h = FQ6K::wd(w.hm[wl >> 2], wl & 3);
                    const uint32_t u = ((q >> (2 * s)) & 0x03030303u) | (((h >> (4 * n + s)) & 0x01010101u) << 2);
                    if (wl < 4) acc0 = dp4a(u, xw[wl], acc0);
                    else acc1 = dp4a(u, xw[wl], acc1);
                }
                const int j = 8 * n + 2 * s;
                is[j] = acc0 - 4 * (int)bs[j];
                is[j + 1] = acc1 - 4 * (int)bs[j + 1];
            }
        }
    }
    // d_x * d * sum_j (s_j - 32) is_j
    __device__ static float combine(const W &w, const Act &a, int k0, int, const int *is) {
        const uint32_t lo[2] = {w.sd.x, w.sd.y}, hi = w.sd.z;
        int P = 0;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const uint32_t b = byte_of(lo[(j & 7) >> 2], j & 3);
            const int low = (int)(j < 8 ? (b & 15u) : (b >> 4));
            const int high = (int)((byte_of(hi, j & 3) >> (2 * (j >> 2))) & 3u);
            P += ((low | (high << 4)) - 32) * is[j];
        }
        const float d = h2f(w.sd.w);
        const float dx = a.d[k0 >> a.lgB];
        return dx * (d * (float)P);
    }
};

// ---------------------------------------------------- shared-expert gate
// Per-token weight of the shared expert, sigma(w . x), w the f32 gate vector
// (the pulsar README names the tensor, gate_inp_shexp, among the f32 tensors
// it loads for qwen35moe; its plain reading is this scalar gate).  One warp:
// the logit in the router's fixed order - 1024-element segments, lane l
// accumulating float4 chunks l, l + 32, ... with fmaf in element order, an
// xor butterfly over 16, 8, 4, 2, 1, segments added in order - then
// 1 / (1 + exp(-l)).  w and x 16-byte aligned; every lane returns the weight.
__device__ __forceinline__ float shared_gate_weight(const float *w, const float *x, int H, int lane) {
    float l = 0.f;
    for (int s0 = 0; s0 < H; s0 += 1024) {
        const int seglen = min(1024, H - s0);
        float v = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int c = lane + 32 * j;
            if (4 * c < seglen) {
                const float4 wv = *reinterpret_cast<const float4 *>(w + s0 + 4 * c);
                const float4 xv = *reinterpret_cast<const float4 *>(x + s0 + 4 * c);
                v = __fmaf_rn(wv.x, xv.x, v);
                v = __fmaf_rn(wv.y, xv.y, v);
                v = __fmaf_rn(wv.z, xv.z, v);
                v = __fmaf_rn(wv.w, xv.w, v);
            }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
        l = s0 == 0 ? v : __fadd_rn(l, v);
    }
    return 1.f / (1.f + expf(-l));
}

// ------------------------------------------------------------ quantiser
// Activation quantisation rule (pulsar README, "MoE resolve": activations
// quantised to q8_0/q8_K before integer dots).  Per block of B = 256 (32 where
// the width is not a multiple of 256): amax = max|x|, d = amax/127,
// q = rint(x * (127/amax)) with IEEE division and round-half-to-even, d = 0
// and q = 0 for an all-zero block, and the sums of each 16 codes.

// lane l's 8 elements (8l..8l+7 of the 256-chunk at c0); false past the row
template <bool coherent>
__device__ __forceinline__ bool quant_load8(const float *x, int n, int c0, int lane, float v[8]) {
    const int e0 = c0 + 8 * lane;
    if (e0 < n) {
        float4 a, b;
        if (coherent) {
            a = __ldcg(reinterpret_cast<const float4 *>(x + e0));
            b = __ldcg(reinterpret_cast<const float4 *>(x + e0 + 4));
        } else {
            a = *reinterpret_cast<const float4 *>(x + e0);
            b = *reinterpret_cast<const float4 *>(x + e0 + 4);
        }
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        return true;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = 0.f;
    return false;
}

// quantise a warp's 256-chunk (values already loaded) into the q8 record
__device__ __forceinline__ void quant_store8(const float v[8], bool active, int n, int c0, uint8_t *rec, int lane) {
    const int B = act_block(n);
    const int e0 = c0 + 8 * lane;
    uint32_t am = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) am = max(am, __float_as_uint(fabsf(v[i])));
    if (B == 256) {
        am = __reduce_max_sync(0xFFFFFFFFu, am);
    } else {
        am = max(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
        am = max(am, __shfl_xor_sync(0xFFFFFFFFu, am, 2));
    }
    const float amax = __uint_as_float(am);
    float d = 0.f, iscale = 0.f;
    if (amax > 0.f) {
        d = __fdiv_rn(amax, 127.f);
        iscale = __fdiv_rn(127.f, amax);
    }
    int q[8], s = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        int t = amax > 0.f ? __float2int_rn(__fmul_rn(v[i], iscale)) : 0;
        t = max(-127, min(127, t));
        q[i] = t;
        s += t;
    }
    s += __shfl_xor_sync(0xFFFFFFFFu, s, 1);
    if (active) {
        uint2 packed;
        packed.x = (uint32_t)(q[0] & 255) | ((uint32_t)(q[1] & 255) << 8) | ((uint32_t)(q[2] & 255) << 16) |
                   ((uint32_t)(q[3] & 255) << 24);
        packed.y = (uint32_t)(q[4] & 255) | ((uint32_t)(q[5] & 255) << 8) | ((uint32_t)(q[6] & 255) << 16) |
                   ((uint32_t)(q[7] & 255) << 24);
        *reinterpret_cast<uint2 *>(rec + q8_q_off(n) + e0) = packed;
        if ((lane & 1) == 0) reinterpret_cast<int16_t *>(rec + q8_bs_off(n))[e0 >> 4] = (int16_t)s;
        if (B == 256) {
            if (lane == 0) reinterpret_cast<float *>(rec)[c0 >> 8] = d;
        } else if ((lane & 3) == 0) {
            reinterpret_cast<float *>(rec)[e0 >> 5] = d;
        }
    }
}

// One warp quantises 256 consecutive elements (lane l: elements 8l..8l+7) of
// one row and writes them into the row's q8 record.  `coherent` selects L2
// loads for data another block of the same grid has just written.
template <bool coherent>
__device__ __forceinline__ void quant_chunk256(const float *x, int n, int c0, uint8_t *rec, int lane) {
    float v[8];
    const bool active = quant_load8<coherent>(x, n, c0, lane, v);
    quant_store8(v, active, n, c0, rec, lane);
}

}  // namespace moe
