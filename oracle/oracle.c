/*
 * oracle.c - plain, slow CPU oracle for the quantized routed-expert MoE FFN.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may load this file:
 * only the tests, the package's smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code, header or table with the CUDA library.
 *
 * What it computes, step by step, with the passage each step follows:
 *
 *  - Activation quantisation (pulsar README, "MoE resolve": activations are
 *    quantised to q8_0/q8_K and dotted as integers; Q4_K/Q6_K matmuls run on
 *    q8_K activations, model table notes).  Per block of B = 256 elements
 *    (B = 32 where the width is not a multiple of 256, following the README's
 *    "multiple of 32 but not 256 -> q8_0" rule): amax = max|x|, d = amax/127,
 *    q = rint(x * (127/amax)) in fp32, and the sums of each 16 codes.  The
 *    codes are an integer decision, so this step is done in fp32, the
 *    precision the kernel uses.
 *  - Router GEMV (README intro: the router stays resident; "Ornith": gate_inp
 *    is read as f32): logits in fp32 in one fixed summation order (the order
 *    is part of this build's definition of the logit so that expert ids are
 *    reproducible bit for bit): the row is cut into segments of 1024
 *    elements; in a segment, lane l of 32 accumulates the float4 chunks
 *    l, l+32, ... with fmaf in element order; the 32 lane sums are combined
 *    by the xor butterfly over offsets 16, 8, 4, 2, 1; segment values are
 *    added in order, then the router bias.  A Q8_0 router uses segments of
 *    32 weight blocks, lane l taking block l: (d_w * d_x) * isum in fp32.
 *  - Top-k (model table: top-k of E, "softmax router", "sigmoid-gated
 *    router"): k largest logits, the lower index first on equal logits;
 *    softmax or sigmoid weights, renormalised over the chosen k, in fp64.
 *  - Expert FFN ("MoE resolve": ds4's exact math, integer dots on q8
 *    activations; per-block rescale): every weight block is decoded to its
 *    integer codes and scales, the integer sub-block dots are formed exactly,
 *    and the per-block scale combine is done in fp64:
 *      Q8_0 : d_w * d_x * isum32
 *      Q4_K : d_x * (d * sum_j sc_j isum_j - dmin * sum_j m_j bsum_j), 32-sub-blocks
 *      Q2_K : the same over 16-sub-blocks
 *      MXFP4: 2^(e-128) * d_x * sum v_i q_i, v = 2 * E2M1 value
 *      Q6_K : d_x * d * sum_j sc_j isum_j, signed 6-bit codes q - 32, int8
 *             scales, 16-sub-blocks (the model table's Q6_K matmuls on q8_K)
 *      Q3_K : d_x * d * sum_j (s_j - 32) isum_j, 3-bit codes in [-4, 3],
 *             6-bit scales, 16-sub-blocks (the q3_K expert tensors of the
 *             streaming-lane notes)
 *    g and u (+ biases) give h = silu(g) * u (fp64, rounded to fp32 where the
 *    method stores it), h is requantised with the activation rule above, the
 *    down projection (+ bias) gives o, and y = sum over slots in slot order
 *    of w * o, plus the shared expert with weight 1, added last.
 *
 * Where the pages leave a step open, the step states the reading it takes and
 * is marked READING below: the router's summation order, the symmetric
 * activation scale, and the layouts of the Q6_K and Q3_K blocks (the pages
 * name those two formats but print no field list).
 *
 * Parity unpinned: the byte layout of the GGUF-style blocks.  The pages print
 * no worked example of any block; the block decoders are pinned to hand-
 * derived closed forms on the stated fields (and to the generator's encoders),
 * which fixes this file's reading of the layouts but not its byte-for-byte
 * agreement with real GGUF files.
 */
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#include <math.h>

enum { OQ_F32 = 0, OQ_Q8_0 = 1, OQ_Q4_K = 2, OQ_Q2_K = 3, OQ_MXFP4 = 4, OQ_Q6_K = 5, OQ_Q3_K = 6 };

/* ------------------------------------------------------------ decoding */

/* IEEE binary16 -> binary32 (exact) */
float oracle_f16(uint16_t h) {
    int sign = (h >> 15) & 1, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 0) v = ldexp((double)m, -24);
    else if (e == 31) v = m ? NAN : INFINITY;
    else v = ldexp((double)(1024 + m), e - 25);
    return (float)(sign ? -v : v);
}

static uint16_t rd16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* Q4_K super-block: 6-bit scale and min of sub-block j (GGUF packing) */
static void q4k_scale_min(const uint8_t *s, int j, int *sc, int *m) {
    if (j < 4) {
        *sc = s[j] & 63;
        *m = s[j + 4] & 63;
    } else {
        *sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
        *m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
}

/* integer codes of one Q4_K super-block (values 0..15, element order) */
static void q4k_codes(const uint8_t *blk, int *q) {
    const uint8_t *qs = blk + 16;
    for (int g = 0; g < 4; ++g)
        for (int l = 0; l < 32; ++l) {
            q[64 * g + l] = qs[32 * g + l] & 15;
            q[64 * g + 32 + l] = qs[32 * g + l] >> 4;
        }
}

static void q2k_codes(const uint8_t *blk, int *q) {
    const uint8_t *qs = blk + 16;
    for (int n = 0; n < 2; ++n)
        for (int s = 0; s < 4; ++s)
            for (int l = 0; l < 32; ++l)
                q[128 * n + 32 * s + l] = (qs[32 * n + l] >> (2 * s)) & 3;
}

/* MXFP4 element j of a block as the integer lattice value v = 2 * E2M1(j) */
static int mxfp4_v(const uint8_t *blk, int j) {
    static const int mag[8] = {0, 1, 2, 3, 4, 6, 8, 12};
    int c = j < 16 ? (blk[1 + j] & 15) : (blk[1 + j - 16] >> 4);
    return (c & 8) ? -mag[c & 7] : mag[c & 7];
}

/* READING: Q6_K and Q3_K follow the public GGUF block layouts.
 * Q6_K super-block {ql[128], qh[64], i8 sc[16], f16 d}: signed code of
 * element i.  With i = 128n + 32s + l, the low nibble sits in byte
 * 64n + l + 32*(s odd) of ql (upper nibble when s >= 2) and the top two bits
 * in bits 2s, 2s+1 of qh[32n + l]; the stored 6-bit value is offset by 32. */
static int q6k_code(const uint8_t *blk, int i) {
    int n = i / 128, s = (i % 128) / 32, l = i % 32;
    int lo = blk[64 * n + 32 * (s % 2) + l];
    lo = (s >= 2) ? (lo >> 4) : (lo & 15);
    int hi = (blk[128 + 32 * n + l] >> (2 * s)) & 3;
    return (lo | (hi << 4)) - 32;
}

static int q6k_scale(const uint8_t *blk, int j) { return (int8_t)blk[192 + j]; }

/* Q3_K super-block {hmask[32], qs[64], sc[12], f16 d}: signed code of
 * element i = 128n + 32s + l is the 2-bit field at bits 2s, 2s+1 of
 * qs[32n + l], minus 4 unless bit 4n + s of hmask[l] is set. */
static int q3k_code(const uint8_t *blk, int i) {
    int n = i / 128, s = (i % 128) / 32, l = i % 32;
    int lo = (blk[32 + 32 * n + l] >> (2 * s)) & 3;
    int set = (blk[l] >> (4 * n + s)) & 1;
    return set ? lo : lo - 4;
}

/* Q3_K scale of sub-block j (0..15): 4 low bits from the nibbles of bytes
 * 0..7 (j < 8: low nibble of byte j; else high nibble of byte j - 8), 2 high
 * bits from byte 8 + j%4 at bit 2*(j/4); the 6-bit value is offset by 32. */
static int q3k_scale(const uint8_t *blk, int j) {
    const uint8_t *s = blk + 96;
    int low = (j < 8) ? (s[j] & 15) : (s[j - 8] >> 4);
    int high = (s[8 + j % 4] >> (2 * (j / 4))) & 3;
    return (low | (high << 4)) - 32;
}

int oracle_block_elems(int qt) {
    switch (qt) { case OQ_F32: return 1; case OQ_Q8_0: case OQ_MXFP4: return 32;
                  case OQ_Q4_K: case OQ_Q2_K: case OQ_Q6_K: case OQ_Q3_K: return 256; }
    return -1;
}
int oracle_block_bytes(int qt) {
    switch (qt) { case OQ_F32: return 4; case OQ_Q8_0: return 34; case OQ_Q4_K: return 144;
                  case OQ_Q2_K: return 84; case OQ_MXFP4: return 17; case OQ_Q6_K: return 210;
                  case OQ_Q3_K: return 110; }
    return -1;
}

/* sub-blocks per weight block, for the integer-dot listing */
int oracle_subblocks(int qt) {
    switch (qt) { case OQ_Q4_K: return 8; case OQ_Q2_K: case OQ_Q6_K: case OQ_Q3_K: return 16;
                  case OQ_Q8_0: return 1; case OQ_MXFP4: return 1; }
    return -1;
}

/* Dequantise one row of blocks to fp64 values (used by tests as a pin target). */
int oracle_dequant_row(int qt, const uint8_t *row, int cols, double *out) {
    int qk = oracle_block_elems(qt), bb = oracle_block_bytes(qt);
    if (qk <= 1 || cols % qk) return -1;
    for (int b = 0; b < cols / qk; ++b) {
        const uint8_t *blk = row + (size_t)b * bb;
        double *o = out + (size_t)b * qk;
        int q[256];
        if (qt == OQ_Q8_0) {
            double d = oracle_f16(rd16(blk));
            for (int i = 0; i < 32; ++i) o[i] = d * (double)(int8_t)blk[2 + i];
        } else if (qt == OQ_Q4_K) {
            double d = oracle_f16(rd16(blk)), dm = oracle_f16(rd16(blk + 2));
            q4k_codes(blk, q);
            for (int i = 0; i < 256; ++i) {
                int sc, m; q4k_scale_min(blk + 4, i / 32, &sc, &m);
                o[i] = d * sc * q[i] - dm * m;
            }
        } else if (qt == OQ_Q2_K) {
            double d = oracle_f16(rd16(blk + 80)), dm = oracle_f16(rd16(blk + 82));
            q2k_codes(blk, q);
            for (int i = 0; i < 256; ++i) {
                int sc = blk[i / 16] & 15, m = blk[i / 16] >> 4;
                o[i] = d * sc * q[i] - dm * m;
            }
        } else if (qt == OQ_MXFP4) {
            double s = ldexp(1.0, (int)blk[0] - 128);
            for (int i = 0; i < 32; ++i) o[i] = s * mxfp4_v(blk, i);
        } else if (qt == OQ_Q6_K) {
            double d = oracle_f16(rd16(blk + 208));
            for (int i = 0; i < 256; ++i) o[i] = d * q6k_scale(blk, i / 16) * q6k_code(blk, i);
        } else if (qt == OQ_Q3_K) {
            double d = oracle_f16(rd16(blk + 108));
            for (int i = 0; i < 256; ++i) o[i] = d * q3k_scale(blk, i / 16) * q3k_code(blk, i);
        }
    }
    return 0;
}

/* ---------------------------------------------------- activation quant */

/* One row of n values into blocks of B: d[n/B], q[n], bsum[n/16].  fp32. */
int oracle_quantize(const float *x, int n, int B, float *d, int8_t *q, int16_t *bsum) {
    if (B != 256 && B != 32) return -1;
    if (n % B) return -1;
    for (int b = 0; b < n / B; ++b) {
        const float *xb = x + (size_t)b * B;
        float amax = 0.f;
        for (int i = 0; i < B; ++i) { float a = fabsf(xb[i]); if (a > amax) amax = a; }
        if (amax == 0.f) {
            d[b] = 0.f;
            for (int i = 0; i < B; ++i) q[(size_t)b * B + i] = 0;
        } else {
            /* READING: symmetric scale amax/127, round half to even */
            float iscale = 127.f / amax;
            d[b] = amax / 127.f;
            for (int i = 0; i < B; ++i) {
                float p = xb[i] * iscale;
                int v = (int)rintf(p);
                if (v > 127) v = 127;
                if (v < -127) v = -127;
                q[(size_t)b * B + i] = (int8_t)v;
            }
        }
    }
    for (int j = 0; j < n / 16; ++j) {
        int s = 0;
        for (int i = 0; i < 16; ++i) s += q[16 * j + i];
        bsum[j] = (int16_t)s;
    }
    return 0;
}

/* ------------------------------------------------------------- router */

static float butterfly32(float v[32]) {
    for (int off = 16; off >= 1; off >>= 1) {
        float nv[32];
        for (int l = 0; l < 32; ++l) nv[l] = v[l] + v[l ^ off];
        memcpy(v, nv, sizeof nv);
    }
    return v[0];
}

/* fp32 router, canonical order (READING: the order stated in the header) */
int oracle_router_f32(const float *W, int E, int H, const float *x, int T,
                      const float *bias, float *logits) {
    if (H % 4) return -1;
    int nseg = (H + 1023) / 1024;
    for (int t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e) {
            const float *w = W + (size_t)e * H;
            const float *xt = x + (size_t)t * H;
            float acc = 0.f;
            for (int s = 0; s < nseg; ++s) {
                float v[32];
                for (int l = 0; l < 32; ++l) {
                    v[l] = 0.f;
                    for (int c = l; c < 256; c += 32) {
                        int base = s * 1024 + 4 * c;
                        if (base >= H) break;
                        for (int j = 0; j < 4; ++j) v[l] = fmaf(w[base + j], xt[base + j], v[l]);
                    }
                }
                float seg = butterfly32(v);
                acc = (s == 0) ? seg : acc + seg;
            }
            if (bias) acc = acc + bias[e];
            logits[(size_t)t * E + e] = acc;
        }
    return 0;
}

/* Q8_0 router on q8 activations (d per B-block, codes), canonical order */
int oracle_router_q8_0(const uint8_t *W, int E, int H, const float *xd, const int8_t *xq,
                       int B, int T, const float *bias, float *logits) {
    if (H % 32 || H % B) return -1;
    int nblk = H / 32, nseg = (nblk + 31) / 32, nbx = H / B;
    for (int t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e) {
            const uint8_t *row = W + (size_t)e * nblk * 34;
            float acc = 0.f;
            for (int s = 0; s < nseg; ++s) {
                float v[32];
                for (int l = 0; l < 32; ++l) {
                    int b = s * 32 + l;
                    v[l] = 0.f;
                    if (b >= nblk) continue;
                    const uint8_t *blk = row + (size_t)b * 34;
                    int isum = 0;
                    for (int i = 0; i < 32; ++i)
                        isum += (int)(int8_t)blk[2 + i] * (int)xq[(size_t)t * H + 32 * b + i];
                    float p = oracle_f16(rd16(blk)) * xd[(size_t)t * nbx + (32 * b) / B];
                    v[l] = p * (float)isum;
                }
                float seg = butterfly32(v);
                acc = (s == 0) ? seg : acc + seg;
            }
            if (bias) acc = acc + bias[e];
            logits[(size_t)t * E + e] = acc;
        }
    return 0;
}

/* fp64 router logits, plain dot (pin target for the canonical fp32 order) */
int oracle_router_f64(const float *W, int E, int H, const float *x, int T,
                      const float *bias, double *logits) {
    for (int t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int j = 0; j < H; ++j) acc += (double)W[(size_t)e * H + j] * (double)x[(size_t)t * H + j];
            if (bias) acc += bias[e];
            logits[(size_t)t * E + e] = acc;
        }
    return 0;
}

/* top-k with lowest-index tie-break, then gating weights (fp64) */
int oracle_topk(const float *logits, int T, int E, int k, int gating, int renorm,
                int32_t *ids, double *w) {
    if (k < 1 || k > E || E > 4096) return -1;
    for (int t = 0; t < T; ++t) {
        const float *l = logits + (size_t)t * E;
        unsigned char taken[4096];
        memset(taken, 0, (size_t)E);
        for (int s = 0; s < k; ++s) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || l[e] > l[best]) best = e;   /* strict: lower index wins ties */
            }
            taken[best] = 1;
            ids[(size_t)t * k + s] = best;
        }
        int32_t *id = ids + (size_t)t * k;
        double *wt = w + (size_t)t * k;
        if (gating == 0) {                        /* softmax */
            if (renorm) {
                double mx = l[id[0]], z = 0.0;
                for (int s = 0; s < k; ++s) z += exp((double)l[id[s]] - mx);
                for (int s = 0; s < k; ++s) wt[s] = exp((double)l[id[s]] - mx) / z;
            } else {
                double mx = l[id[0]], z = 0.0;
                for (int e = 0; e < E; ++e) z += exp((double)l[e] - mx);
                for (int s = 0; s < k; ++s) wt[s] = exp((double)l[id[s]] - mx) / z;
            }
        } else {                                  /* sigmoid */
            double z = 0.0, sg[4096];
            for (int s = 0; s < k; ++s) { sg[s] = 1.0 / (1.0 + exp(-(double)l[id[s]])); z += sg[s]; }
            for (int s = 0; s < k; ++s) wt[s] = renorm ? sg[s] / z : sg[s];
        }
    }
    return 0;
}

/* ---------------------------------------------------------- row dots */

/* Exact integer sub-block dots of one weight row with q8 codes xq[cols]:
 * Q4_K 8 per super-block, Q2_K 16, Q8_0 and MXFP4 one per 32-block. */
int oracle_row_isums(int qt, const uint8_t *row, int cols, const int8_t *xq, int32_t *isums) {
    int qk = oracle_block_elems(qt), bb = oracle_block_bytes(qt);
    if (qk <= 1 || cols % qk) return -1;
    int nsub = oracle_subblocks(qt), sublen = qk / nsub;
    for (int b = 0; b < cols / qk; ++b) {
        const uint8_t *blk = row + (size_t)b * bb;
        const int8_t *x = xq + (size_t)b * qk;
        int q[256];
        if (qt == OQ_Q4_K) q4k_codes(blk, q);
        else if (qt == OQ_Q2_K) q2k_codes(blk, q);
        else if (qt == OQ_Q6_K) for (int i = 0; i < 256; ++i) q[i] = q6k_code(blk, i);
        else if (qt == OQ_Q3_K) for (int i = 0; i < 256; ++i) q[i] = q3k_code(blk, i);
        else if (qt == OQ_Q8_0) for (int i = 0; i < 32; ++i) q[i] = (int8_t)blk[2 + i];
        else for (int i = 0; i < 32; ++i) q[i] = mxfp4_v(blk, i);
        for (int j = 0; j < nsub; ++j) {
            int s = 0;
            for (int i = 0; i < sublen; ++i) s += q[j * sublen + i] * (int)x[j * sublen + i];
            isums[(size_t)b * nsub + j] = s;
        }
    }
    return 0;
}

/* One weight row against one q8 activation row: the per-block scale combine
 * of the integer dots, summed over blocks in order, in fp64. */
double oracle_row_dot(int qt, const uint8_t *row, int cols, const float *xd, const int8_t *xq,
                      const int16_t *xbsum, int B) {
    int qk = oracle_block_elems(qt), bb = oracle_block_bytes(qt);
    int32_t is[16];
    double acc = 0.0;
    if (qk <= 1 || cols % qk || B % 32 || cols % B || (qk > B)) return NAN;  /* K-quants need 256-blocks */
    for (int b = 0; b < cols / qk; ++b) {
        const uint8_t *blk = row + (size_t)b * bb;
        oracle_row_isums(qt, blk, qk, xq + (size_t)b * qk, is);
        double dx = xd[((size_t)b * qk) / B];
        const int16_t *bs = xbsum + (size_t)b * qk / 16;
        double term;
        if (qt == OQ_Q8_0) {
            term = (double)oracle_f16(rd16(blk)) * dx * is[0];
        } else if (qt == OQ_MXFP4) {
            term = ldexp(1.0, (int)blk[0] - 128) * dx * is[0];
        } else if (qt == OQ_Q4_K) {
            long long P = 0, M = 0;
            for (int j = 0; j < 8; ++j) {
                int sc, m; q4k_scale_min(blk + 4, j, &sc, &m);
                P += (long long)sc * is[j];
                M += (long long)m * (bs[2 * j] + bs[2 * j + 1]);
            }
            term = dx * ((double)oracle_f16(rd16(blk)) * (double)P - (double)oracle_f16(rd16(blk + 2)) * (double)M);
        } else if (qt == OQ_Q6_K || qt == OQ_Q3_K) {
            /* no min term: the codes are signed */
            long long P = 0;
            for (int j = 0; j < 16; ++j)
                P += (long long)(qt == OQ_Q6_K ? q6k_scale(blk, j) : q3k_scale(blk, j)) * is[j];
            double d = oracle_f16(rd16(blk + (qt == OQ_Q6_K ? 208 : 108)));
            term = dx * (d * (double)P);
        } else {
            long long P = 0, M = 0;
            for (int j = 0; j < 16; ++j) {
                P += (long long)(blk[j] & 15) * is[j];
                M += (long long)(blk[j] >> 4) * bs[j];
            }
            term = dx * ((double)oracle_f16(rd16(blk + 80)) * (double)P - (double)oracle_f16(rd16(blk + 82)) * (double)M);
        }
        acc += term;
    }
    return acc;
}

/* ------------------------------------------------------------- ffn */

typedef struct {
    int qtype, H, I, E;
    const uint8_t *gate, *up, *down;     /* AoS blocks [E][rows][row_bytes] */
    const float *bg, *bu, *bd;           /* [E][I], [E][I], [E][H] or NULL */
    const uint8_t *owned;                /* [E] or NULL (all owned) */
} oracle_pool;

static int act_block(int n) { return n % 256 == 0 ? 256 : 32; }
static size_t row_bytes(int qt, int cols) {
    return (size_t)(cols / oracle_block_elems(qt)) * oracle_block_bytes(qt);
}

/* h (fp32) of one expert for one token: silu(g) * u */
static void expert_h(const oracle_pool *p, int e, const float *xd, const int8_t *xq,
                     const int16_t *xbs, float *h) {
    int H = p->H, I = p->I, BH = act_block(H);
    size_t rbh = row_bytes(p->qtype, H);
    for (int r = 0; r < I; ++r) {
        const uint8_t *gr = p->gate + ((size_t)e * I + r) * rbh;
        const uint8_t *ur = p->up + ((size_t)e * I + r) * rbh;
        double g = oracle_row_dot(p->qtype, gr, H, xd, xq, xbs, BH);
        double u = oracle_row_dot(p->qtype, ur, H, xd, xq, xbs, BH);
        if (p->bg) g += p->bg[(size_t)e * I + r];
        if (p->bu) u += p->bu[(size_t)e * I + r];
        h[r] = (float)(g / (1.0 + exp(-g)) * u);
    }
}

static void expert_o(const oracle_pool *p, int e, const float *hd, const int8_t *hq,
                     const int16_t *hbs, double *o) {
    int H = p->H, I = p->I, BI = act_block(I);
    size_t rbi = row_bytes(p->qtype, I);
    for (int r = 0; r < H; ++r) {
        const uint8_t *dr = p->down + ((size_t)e * H + r) * rbi;
        o[r] = oracle_row_dot(p->qtype, dr, I, hd, hq, hbs, BI);
        if (p->bd) o[r] += p->bd[(size_t)e * H + r];
    }
}

/*
 * y[t][:] = sum_{s in slot order} w[t][s] * o(ids[t][s]) + g[t] * o_shared,
 * the shared expert added last with weight g[t] = shared_scale[t] (the
 * sigmoid of its gate logit, READING below) or 1 when shared_scale is NULL.
 * READING: the pulsar README names a shared-expert gate tensor
 * (gate_inp_shexp, one of the f32 tensors it loads for qwen35moe) but does
 * not state its use; the plain reading taken here is a per-token scalar
 * sigma(w . x) with w the f32 vector and x the token's hidden state, that
 * scales the shared expert's output.
 * xd/xq/xbs: the q8 activations of the T tokens (H wide).  Optional outputs
 * h_out [T][k][I] (fp32 h) and hq_* (the requantised h) for component checks.
 * Returns the number of skipped out-of-range ids (slots with e < 0 or e >= E).
 */
int oracle_expert_ffn(const oracle_pool *pool, const oracle_pool *shared, int T, int k,
                      const float *xd, const int8_t *xq, const int16_t *xbs,
                      const int32_t *ids, const double *w, const double *shared_scale, double *y,
                      float *h_out, float *hq_d, int8_t *hq_q, int16_t *hq_bs) {
    int H = pool->H, I = pool->I, BH = act_block(H), BI = act_block(I);
    int bad = 0;
    float h[16384]; float hd[512]; int8_t hq[16384]; int16_t hbs[1024];
    double o[16384];
    if (I > 16384 || H > 16384) return -1;
    if (shared && (shared->I > 16384 || shared->H != H)) return -1;
    for (int t = 0; t < T; ++t) {
        const float *xdt = xd + (size_t)t * (H / BH);
        const int8_t *xqt = xq + (size_t)t * H;
        const int16_t *xbt = xbs + (size_t)t * (H / 16);
        double *yt = y + (size_t)t * H;
        for (int r = 0; r < H; ++r) yt[r] = 0.0;
        for (int s = 0; s < k; ++s) {
            int e = ids[(size_t)t * k + s];
            if (e < 0 || e >= pool->E) { ++bad; continue; }
            if (pool->owned && !pool->owned[e]) continue;
            expert_h(pool, e, xdt, xqt, xbt, h);
            oracle_quantize(h, I, BI, hd, hq, hbs);
            if (h_out) memcpy(h_out + ((size_t)t * k + s) * I, h, sizeof(float) * I);
            if (hq_d) memcpy(hq_d + ((size_t)t * k + s) * (I / BI), hd, sizeof(float) * (I / BI));
            if (hq_q) memcpy(hq_q + ((size_t)t * k + s) * I, hq, (size_t)I);
            if (hq_bs) memcpy(hq_bs + ((size_t)t * k + s) * (I / 16), hbs, sizeof(int16_t) * (I / 16));
            expert_o(pool, e, hd, hq, hbs, o);
            double ws = w[(size_t)t * k + s];
            for (int r = 0; r < H; ++r) yt[r] += ws * o[r];
        }
        if (shared) {
            int Is = shared->I, BS = act_block(Is);
            expert_h(shared, 0, xdt, xqt, xbt, h);
            oracle_quantize(h, Is, BS, hd, hq, hbs);
            expert_o(shared, 0, hd, hq, hbs, o);
            double g = shared_scale ? shared_scale[t] : 1.0;
            for (int r = 0; r < H; ++r) yt[r] += g * o[r];
        }
    }
    return bad;
}
