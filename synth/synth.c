/*
 * synth.c - seeded synthetic inputs for the quantized routed-expert MoE FFN.
 *
 * This module is input generation only.  It draws normal variates from
 * counter-keyed splitmix64 streams and encodes weight matrices into the
 * GGUF-style block layouts (Q8_0, Q4_K, Q2_K, MXFP4, Q6_K, Q3_K) that the CUDA
 * library and the CPU oracle consume.  It computes nothing of the MoE path
 * itself (no dots, no routing, no activation quantisation).
 *
 * Determinism: every value depends only on (seed, stream, row); thread count
 * does not matter.  A normal draw maps 32 random bits through an inverse-CDF
 * table (4097 points, linear interpolation; tails end near +-3.7 sigma) that
 * is built once from the CDF's power series by bisection in IEEE double
 * arithmetic (built with -ffp-contract=off), so x86-64 and aarch64 hosts
 * produce the same bytes.
 *
 * Weight encoders follow a deliberately simple, deterministic rule (they are
 * not the reference's imatrix quantiser):
 *   Q8_0   : d = max|w|/127 stored as f16, q = clamp(rint(w/d), -127, 127).
 *   Q4_K   : per 32-sub-block scale = (max - min0)/15 and min = -min0 with
 *            min0 = min(0, min w); d = max scale/63, dmin = max min/63 (f16);
 *            6-bit sc/m = rint(scale/d), rint(min/dmin);
 *            q = clamp(rint((w + dmin*m)/(d*sc)), 0, 15).
 *   Q2_K   : the same with 16-sub-blocks, 2-bit q, 4-bit sc/m, /3 and /15.
 *   MXFP4  : e = ceil(log2(max|w|/6)), stored e+127; each w/2^e rounded to the
 *            nearest E2M1 value, ties to the even code.
 *   Q6_K   : per 16-sub-block step = max|w|/31; d = max step/127 (f16);
 *            int8 sc = rint(step/d); q = clamp(rint(w/(d*sc)), -32, 31),
 *            stored as q + 32 (low nibble in ql, top 2 bits in qh).
 *   Q3_K   : per 16-sub-block step = max|w|/4; d = max step/31 (f16);
 *            6-bit s = rint(step/d) + 32 (scale s - 32);
 *            q = clamp(rint(w/(d*(s-32))), -4, 3), stored as 2 low bits of
 *            q + 4 in qs and a high-mask bit set when q >= 0.
 */
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#include <stdlib.h>
#include <math.h>
#include <pthread.h>

/* ---------------------------------------------------------------- rng */

static inline uint64_t sm64_step(uint64_t *s) {
    uint64_t z = (*s += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static uint64_t stream_key(uint64_t seed, uint64_t stream, uint64_t row) {
    uint64_t s = seed ^ 0x5DEECE66Dull;
    uint64_t a = sm64_step(&s);
    s = a ^ stream;
    uint64_t b = sm64_step(&s);
    s = b ^ (row * 0xD1B54A32D192ED03ull);
    return sm64_step(&s);
}

/* Standard normal CDF by its Taylor series (IEEE double, no libm):
 * Phi(x) = 1/2 + (1/sqrt(2 pi)) sum_n (-1)^n x^(2n+1) / (2^n n! (2n+1)).
 * Accurate to ~1e-12 for |x| <= 4, which is all the table below needs. */
static double det_phi(double x) {
    double term = x, sum = x, x2 = x * x;
    for (int n = 1; n < 200; ++n) {
        term *= -x2 / (2.0 * n);
        double add = term / (double)(2 * n + 1);
        sum += add;
        if (add < 1e-18 && add > -1e-18) break;
    }
    return 0.5 + 0.39894228040143267793994605993438 * sum;
}

/* Inverse-CDF table at u_j = (j + 0.5) / NTAB1, j = 0..NTAB; a normal draw
 * takes 12 bits of a uniform as the cell and 16 more as the position in it. */
#define NTAB 4096
#define NTAB1 (NTAB + 1)
static float g_tab[NTAB + 1];
static pthread_once_t g_tab_once = PTHREAD_ONCE_INIT;

static void build_table(void) {
    for (int j = 0; j <= NTAB; ++j) {
        double u = ((double)j + 0.5) / (double)NTAB1, lo = -6.0, hi = 6.0;
        for (int it = 0; it < 64; ++it) {
            double mid = 0.5 * (lo + hi);
            if (det_phi(mid) < u) lo = mid; else hi = mid;
        }
        g_tab[j] = (float)(0.5 * (lo + hi));
    }
}

static inline float normal_from_u32(uint32_t u) {
    uint32_t cell = u >> 20, pos = (u >> 4) & 0xFFFFu;
    float a = g_tab[cell], b = g_tab[cell + 1];
    return a + (b - a) * ((float)pos * (1.0f / 65536.0f));
}

/* n standard normals scaled by sigma from the (seed, stream, row) key */
static void normal_row(uint64_t seed, uint64_t stream, uint64_t row, float sigma,
                       float *out, int64_t n) {
    pthread_once(&g_tab_once, build_table);
    uint64_t s = stream_key(seed, stream, row);
    for (int64_t i = 0; i < n; i += 2) {
        uint64_t r = sm64_step(&s);
        out[i] = sigma * normal_from_u32((uint32_t)r);
        if (i + 1 < n) out[i + 1] = sigma * normal_from_u32((uint32_t)(r >> 32));
    }
}

/* ------------------------------------------------------------ f32->f16 */

static uint16_t f32_to_f16(float f) {
    uint32_t x; memcpy(&x, &f, 4);
    uint32_t sign = (x >> 16) & 0x8000u;
    uint32_t ax = x & 0x7FFFFFFFu;
    if (ax >= 0x7F800000u) return (uint16_t)(sign | 0x7C00u | (ax > 0x7F800000u ? 0x200u : 0));
    if (ax >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u);       /* rounds to inf */
    if (ax < 0x38800000u) {                                         /* f16 subnormal */
        if (ax < 0x33000000u) return (uint16_t)sign;                /* < 2^-25 -> 0 */
        uint32_t e = ax >> 23, mant = (ax & 0x7FFFFFu) | 0x800000u;
        uint32_t shift = 126 - e;                                   /* 14..24 */
        uint32_t h = mant >> shift;
        uint32_t rem = mant & ((1u << shift) - 1u), half = 1u << (shift - 1);
        if (rem > half || (rem == half && (h & 1u))) h++;
        return (uint16_t)(sign | h);
    }
    uint32_t h = ((ax >> 13) - (112u << 10));
    uint32_t rem = ax & 0x1FFFu;
    if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h++;
    return (uint16_t)(sign | h);
}

static float f16_value(uint16_t h) {       /* exact widening, used to encode */
    uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
    uint32_t e = (h >> 10) & 0x1Fu, m = h & 0x3FFu, x;
    if (e == 0) {
        float v = (float)m * 0x1p-24f;
        return sign ? -v : v;
    }
    if (e == 31) x = sign | 0x7F800000u | (m << 13);
    else x = sign | ((e + 112u) << 23) | (m << 13);
    float f; memcpy(&f, &x, 4); return f;
}

static inline int clampi(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }

/* -------------------------------------------------------------- encoders */

static void enc_q8_0(const float *w, int64_t cols, uint8_t *out) {
    for (int64_t b = 0; b < cols / 32; ++b) {
        const float *x = w + 32 * b;
        uint8_t *blk = out + 34 * b;
        float amax = 0.f;
        for (int i = 0; i < 32; ++i) { float a = fabsf(x[i]); if (a > amax) amax = a; }
        uint16_t dh = f32_to_f16(amax / 127.f);
        float d = f16_value(dh);
        memcpy(blk, &dh, 2);
        for (int i = 0; i < 32; ++i) {
            int q = d > 0.f ? (int)rintf(x[i] / d) : 0;
            blk[2 + i] = (uint8_t)(int8_t)clampi(q, -127, 127);
        }
    }
}

/* shared helper for the two K-quant encoders: nsub sub-blocks of len elements */
static void kquant_params(const float *x, int nsub, int len, int qmax, int smax,
                          uint16_t *dh, uint16_t *dmh, int *sc, int *mn) {
    float scale[16], minv[16], smx = 0.f, mmx = 0.f;
    for (int j = 0; j < nsub; ++j) {
        float lo = 0.f, hi = -INFINITY;
        for (int i = 0; i < len; ++i) {
            float v = x[j * len + i];
            if (v < lo) lo = v;
            if (v > hi) hi = v;
        }
        if (hi < 0.f) hi = 0.f;
        scale[j] = (hi - lo) / (float)qmax;
        minv[j] = -lo;
        if (scale[j] > smx) smx = scale[j];
        if (minv[j] > mmx) mmx = minv[j];
    }
    *dh = f32_to_f16(smx / (float)smax);
    *dmh = f32_to_f16(mmx / (float)smax);
    float d = f16_value(*dh), dm = f16_value(*dmh);
    for (int j = 0; j < nsub; ++j) {
        sc[j] = d > 0.f ? clampi((int)rintf(scale[j] / d), 0, smax) : 0;
        mn[j] = dm > 0.f ? clampi((int)rintf(minv[j] / dm), 0, smax) : 0;
    }
}

static void enc_q4_k(const float *w, int64_t cols, uint8_t *out) {
    for (int64_t b = 0; b < cols / 256; ++b) {
        const float *x = w + 256 * b;
        uint8_t *blk = out + 144 * b;
        uint16_t dh, dmh; int sc[8], mn[8];
        kquant_params(x, 8, 32, 15, 63, &dh, &dmh, sc, mn);
        float d = f16_value(dh), dm = f16_value(dmh);
        memcpy(blk, &dh, 2); memcpy(blk + 2, &dmh, 2);
        uint8_t *s = blk + 4;
        memset(s, 0, 12);
        for (int j = 0; j < 4; ++j) {
            s[j] = (uint8_t)(sc[j] & 63);
            s[j + 4] = (uint8_t)(mn[j] & 63);
        }
        for (int j = 4; j < 8; ++j) {
            s[j + 4] = (uint8_t)((sc[j] & 15) | ((mn[j] & 15) << 4));
            s[j - 4] |= (uint8_t)((sc[j] >> 4) << 6);
            s[j] |= (uint8_t)((mn[j] >> 4) << 6);
        }
        int q[256];
        for (int i = 0; i < 256; ++i) {
            int j = i / 32;
            float step = d * (float)sc[j];
            q[i] = step > 0.f ? clampi((int)rintf((x[i] + dm * (float)mn[j]) / step), 0, 15) : 0;
        }
        uint8_t *qs = blk + 16;
        for (int g = 0; g < 4; ++g)
            for (int l = 0; l < 32; ++l)
                qs[32 * g + l] = (uint8_t)(q[64 * g + l] | (q[64 * g + 32 + l] << 4));
    }
}

static void enc_q2_k(const float *w, int64_t cols, uint8_t *out) {
    for (int64_t b = 0; b < cols / 256; ++b) {
        const float *x = w + 256 * b;
        uint8_t *blk = out + 84 * b;
        uint16_t dh, dmh; int sc[16], mn[16];
        kquant_params(x, 16, 16, 3, 15, &dh, &dmh, sc, mn);
        float d = f16_value(dh), dm = f16_value(dmh);
        for (int j = 0; j < 16; ++j) blk[j] = (uint8_t)(sc[j] | (mn[j] << 4));
        int q[256];
        for (int i = 0; i < 256; ++i) {
            int j = i / 16;
            float step = d * (float)sc[j];
            q[i] = step > 0.f ? clampi((int)rintf((x[i] + dm * (float)mn[j]) / step), 0, 3) : 0;
        }
        uint8_t *qs = blk + 16;
        memset(qs, 0, 64);
        for (int n = 0; n < 2; ++n)
            for (int sft = 0; sft < 4; ++sft)
                for (int l = 0; l < 32; ++l)
                    qs[32 * n + l] |= (uint8_t)(q[128 * n + 32 * sft + l] << (2 * sft));
        memcpy(blk + 80, &dh, 2); memcpy(blk + 82, &dmh, 2);
    }
}

/* E2M1 magnitudes by code 0..7, and rounding to the nearest, ties to even code */
static const float E2M1[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};

static int e2m1_code(float v) {
    float a = fabsf(v);
    int best = 0;
    for (int c = 1; c < 8; ++c) {
        float dc = fabsf(a - E2M1[c]), db = fabsf(a - E2M1[best]);
        if (dc < db || (dc == db && (c & 1) == 0)) best = c;
    }
    return best | ((v < 0.f && best != 0) ? 8 : 0);
}

static void enc_mxfp4(const float *w, int64_t cols, uint8_t *out) {
    for (int64_t b = 0; b < cols / 32; ++b) {
        const float *x = w + 32 * b;
        uint8_t *blk = out + 17 * b;
        float amax = 0.f;
        for (int i = 0; i < 32; ++i) { float a = fabsf(x[i]); if (a > amax) amax = a; }
        int e;
        if (amax == 0.f) {
            e = -127;
        } else {
            int k; double m = frexp((double)amax / 6.0, &k);
            e = (m == 0.5) ? k - 1 : k;
            if (e < -127) e = -127;
            if (e > 127) e = 127;
        }
        blk[0] = (uint8_t)(e + 127);
        double inv = ldexp(1.0, -e);
        uint8_t code[32];
        for (int i = 0; i < 32; ++i) code[i] = (uint8_t)e2m1_code((float)((double)x[i] * inv));
        for (int j = 0; j < 16; ++j) blk[1 + j] = (uint8_t)(code[j] | (code[j + 16] << 4));
    }
}

/* Q6_K: {u8 ql[128]; u8 qh[64]; i8 sc[16]; f16 d} = 210 B per 256 weights.
 * Element 128n + 32s + l (half n, quarter s, lane l) keeps its low nibble in
 * ql[64n + 32(s&1) + l] (low nibble for s < 2, high for s >= 2) and its top
 * two bits at bits 2s..2s+1 of qh[32n + l]; sub-block j = i/16 uses sc[j]. */
static void enc_q6_k(const float *w, int64_t cols, uint8_t *out) {
    for (int64_t b = 0; b < cols / 256; ++b) {
        const float *x = w + 256 * b;
        uint8_t *blk = out + 210 * b;
        float step[16], smx = 0.f;
        for (int j = 0; j < 16; ++j) {
            float amax = 0.f;
            for (int i = 0; i < 16; ++i) { float a = fabsf(x[16 * j + i]); if (a > amax) amax = a; }
            step[j] = amax / 31.f;
            if (step[j] > smx) smx = step[j];
        }
        uint16_t dh = f32_to_f16(smx / 127.f);
        float d = f16_value(dh);
        int sc[16], q[256];
        for (int j = 0; j < 16; ++j) sc[j] = d > 0.f ? clampi((int)rintf(step[j] / d), 0, 127) : 0;
        for (int i = 0; i < 256; ++i) {
            float st = d * (float)sc[i / 16];
            q[i] = (st > 0.f ? clampi((int)rintf(x[i] / st), -32, 31) : 0) + 32;
        }
        uint8_t *ql = blk, *qh = blk + 128;
        memset(blk, 0, 192);
        for (int n = 0; n < 2; ++n)
            for (int s = 0; s < 4; ++s)
                for (int l = 0; l < 32; ++l) {
                    int v = q[128 * n + 32 * s + l];
                    ql[64 * n + 32 * (s & 1) + l] |= (uint8_t)((v & 15) << (s < 2 ? 0 : 4));
                    qh[32 * n + l] |= (uint8_t)((v >> 4) << (2 * s));
                }
        for (int j = 0; j < 16; ++j) blk[192 + j] = (uint8_t)(int8_t)sc[j];
        memcpy(blk + 208, &dh, 2);
    }
}

/* Q3_K: {u8 hmask[32]; u8 qs[64]; u8 sc[12]; f16 d} = 110 B per 256 weights.
 * Element 128n + 32s + l keeps 2 low bits at bits 2s..2s+1 of qs[32n + l] and
 * its high bit at bit 4n + s of hmask[l]; value q = low - (high ? 0 : 4).
 * The 6-bit scale s_j of sub-block j = i/16 keeps its low nibble in sc[j]
 * (j < 8) or the high nibble of sc[j - 8] (j >= 8), and its top two bits at
 * bits 2(j/4)..2(j/4)+1 of sc[8 + j%4]. */
static void enc_q3_k(const float *w, int64_t cols, uint8_t *out) {
    for (int64_t b = 0; b < cols / 256; ++b) {
        const float *x = w + 256 * b;
        uint8_t *blk = out + 110 * b;
        float step[16], smx = 0.f;
        for (int j = 0; j < 16; ++j) {
            float amax = 0.f;
            for (int i = 0; i < 16; ++i) { float a = fabsf(x[16 * j + i]); if (a > amax) amax = a; }
            step[j] = amax / 4.f;
            if (step[j] > smx) smx = step[j];
        }
        uint16_t dh = f32_to_f16(smx / 31.f);
        float d = f16_value(dh);
        int sc[16], q[256];
        for (int j = 0; j < 16; ++j) sc[j] = d > 0.f ? clampi((int)rintf(step[j] / d), 0, 31) : 0;
        for (int i = 0; i < 256; ++i) {
            float st = d * (float)sc[i / 16];
            q[i] = st > 0.f ? clampi((int)rintf(x[i] / st), -4, 3) : 0;
        }
        uint8_t *hm = blk, *qs = blk + 32, *s6 = blk + 96;
        memset(blk, 0, 108);
        for (int n = 0; n < 2; ++n)
            for (int s = 0; s < 4; ++s)
                for (int l = 0; l < 32; ++l) {
                    int v = q[128 * n + 32 * s + l];
                    qs[32 * n + l] |= (uint8_t)(((v + 4) & 3) << (2 * s));
                    if (v >= 0) hm[l] |= (uint8_t)(1 << (4 * n + s));
                }
        for (int j = 0; j < 16; ++j) {
            int v = sc[j] + 32;
            s6[j < 8 ? j : j - 8] |= (uint8_t)((v & 15) << (j < 8 ? 0 : 4));
            s6[8 + j % 4] |= (uint8_t)((v >> 4) << (2 * (j / 4)));
        }
        memcpy(blk + 108, &dh, 2);
    }
}

/* qtype codes: 0..4 are the library's public enum; Q6_K and Q3_K are
 * generated for the CPU oracle (the library does not accept them yet) */
enum { Q_F32 = 0, Q_Q8_0 = 1, Q_Q4_K = 2, Q_Q2_K = 3, Q_MXFP4 = 4, Q_Q6_K = 5, Q_Q3_K = 6 };

int64_t synth_row_bytes(int qtype, int64_t cols) {
    switch (qtype) {
        case Q_F32: return 4 * cols;
        case Q_Q8_0: return cols % 32 ? -1 : cols / 32 * 34;
        case Q_Q4_K: return cols % 256 ? -1 : cols / 256 * 144;
        case Q_Q2_K: return cols % 256 ? -1 : cols / 256 * 84;
        case Q_MXFP4: return cols % 32 ? -1 : cols / 32 * 17;
        case Q_Q6_K: return cols % 256 ? -1 : cols / 256 * 210;
        case Q_Q3_K: return cols % 256 ? -1 : cols / 256 * 110;
    }
    return -1;
}

/* encode rows of an fp32 matrix (row-major) into blocks */
int synth_encode(int qtype, const float *w, int64_t rows, int64_t cols, void *out) {
    int64_t rb = synth_row_bytes(qtype, cols);
    if (rb < 0) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        const float *x = w + r * cols;
        uint8_t *o = (uint8_t *)out + r * rb;
        switch (qtype) {
            case Q_F32: memcpy(o, x, 4 * cols); break;
            case Q_Q8_0: enc_q8_0(x, cols, o); break;
            case Q_Q4_K: enc_q4_k(x, cols, o); break;
            case Q_Q2_K: enc_q2_k(x, cols, o); break;
            case Q_MXFP4: enc_mxfp4(x, cols, o); break;
            case Q_Q6_K: enc_q6_k(x, cols, o); break;
            case Q_Q3_K: enc_q3_k(x, cols, o); break;
            default: return -1;
        }
    }
    return 0;
}

/* ------------------------------------------------------ threaded drivers */

typedef struct {
    int qtype; uint64_t seed, stream; float sigma;
    int64_t r0, r1, cols, row0; void *out;
} job_t;

static void *matrix_worker(void *p) {
    job_t *j = (job_t *)p;
    int64_t rb = synth_row_bytes(j->qtype, j->cols);
    float *row = (float *)malloc(sizeof(float) * (size_t)j->cols);
    if (!row) return (void *)1;
    for (int64_t r = j->r0; r < j->r1; ++r) {
        normal_row(j->seed, j->stream, (uint64_t)(r + j->row0), j->sigma, row, j->cols);
        synth_encode(j->qtype, row, 1, j->cols, (uint8_t *)j->out + r * rb);
    }
    free(row);
    return NULL;
}

/* rows x cols matrix of N(0, sigma^2) values encoded as qtype (F32: raw);
 * row r of the output is row row0 + r of the stream */
int synth_matrix(int qtype, uint64_t seed, uint64_t stream, float sigma,
                 int64_t rows, int64_t cols, void *out, int threads, int64_t row0) {
    if (synth_row_bytes(qtype, cols) < 0 || rows < 0) return -1;
    if (threads < 1) threads = 1;
    if (threads > 256) threads = 256;
    if ((int64_t)threads > rows) threads = rows > 0 ? (int)rows : 1;
    pthread_t th[256]; job_t jobs[256];
    int64_t per = (rows + threads - 1) / threads;
    int started = 0, rc = 0;
    for (int t = 0; t < threads; ++t) {
        jobs[t] = (job_t){qtype, seed, stream, sigma, t * per, (t + 1) * per < rows ? (t + 1) * per : rows, cols,
                          row0, out};
        if (jobs[t].r0 >= jobs[t].r1) continue;
        if (threads == 1) { if (matrix_worker(&jobs[t])) rc = -2; continue; }
        if (pthread_create(&th[started], NULL, matrix_worker, &jobs[t]) != 0) {
            if (matrix_worker(&jobs[t])) rc = -2;
            continue;
        }
        ++started;
    }
    for (int t = 0; t < started; ++t) { void *r; pthread_join(th[t], &r); if (r) rc = -2; }
    return rc;
}

/* n normals for one stream (row 0) */
int synth_normal(uint64_t seed, uint64_t stream, float sigma, float *out, int64_t n) {
    normal_row(seed, stream, 0, sigma, out, n);
    return 0;
}
