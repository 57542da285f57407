// moe_kernels.cu - activation quantiser, router GEMV + top-k, one-time weight
// packing and the integer-dot test hook.
#include "moe_common.cuh"
#include "moe_launch.h"

namespace moe {

// ------------------------------------------------------------ quantiser
//
// pulsar README, "MoE resolve": activations are quantised to q8_0/q8_K and
// dotted as integers (quant_chunk256 in moe_common.cuh holds the rule).
__global__ void __launch_bounds__(256) quantize_kernel(const float *__restrict__ x, int T, int n,
                                                       uint8_t *__restrict__ xq) {
    const int chunks = (n + 255) / 256;
    const int wid = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (wid >= T * chunks) return;
    const int t = wid / chunks, c = wid % chunks;
    quant_chunk256<false>(x + (size_t)t * n, n, 256 * c, xq + (size_t)t * q8_row_bytes(n), threadIdx.x & 31);
}

cudaError_t launch_quantize(const float *x, int T, int n, uint8_t *xq, cudaStream_t s) {
    const int warps = T * ((n + 255) / 256);
    if (warps == 0) return cudaSuccess;
    quantize_kernel<<<(warps + 7) / 8, 256, 0, s>>>(x, T, n, xq);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- router
//
// Router GEMV (README intro: the router stays resident; "Ornith": gate_inp is
// an f32 tensor) with the fixed summation order stated in moe.h, then top-k
// with lowest-index tie-break and softmax or sigmoid gating (README model
// table).  Grid: (segment, group of 8 experts); each warp owns one expert row
// and writes its segment value for every token.  The last block to finish
// (atomic ticket) adds the segments in order, selects the top k and writes
// ids, weights and logits; it then rearms the ticket.
constexpr int ROUTE_WARPS = 8;

__device__ __forceinline__ float butterfly_sum(float v) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
    return v;
}

__device__ void route_topk(const RouteArgs &a, float *smem) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float *lg = smem + warp * MOE_MAX_EXPERTS;
    for (int t = warp; t < a.T; t += ROUTE_WARPS) {
        for (int e = lane; e < a.E; e += 32) {
            const float *p = a.partial + ((size_t)t * a.E + e) * a.nseg;
            float l = __ldcg(p);
            for (int s = 1; s < a.nseg; ++s) l = __fadd_rn(l, __ldcg(p + s));
            if (a.bias) l = __fadd_rn(l, a.bias[e]);
            lg[e] = l;
            if (a.logits_out) a.logits_out[(size_t)t * a.E + e] = l;
        }
        __syncwarp();
        // k rounds of a (value desc, index asc) arg-max; chosen entries are
        // remembered in a per-lane bit set (lane owns e = lane + 32 j)
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
                const bool better = (oi != 0x7FFFFFFF) &&
                                    (bi == 0x7FFFFFFF || ov > bv || (ov == bv && oi < bi));
                if (better) { bv = ov; bi = oi; }
            }
            if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
            if (lane == s) mysel = bv;
            if (lane == 0) a.ids[(size_t)t * a.k + s] = bi;
        }
        // gating weights: lane s < k holds the s-th chosen logit
        const float l0 = __shfl_sync(0xFFFFFFFFu, mysel, 0);
        float w = 0.f, z;
        if (a.gating == MOE_GATE_SOFTMAX) {
            w = lane < a.k ? expf(mysel - l0) : 0.f;
            if (a.renorm) {
                z = butterfly_sum(w);
            } else {
                float acc = 0.f;
                for (int e = lane; e < a.E; e += 32) acc += expf(lg[e] - l0);
                z = butterfly_sum(acc);
            }
            w = w / z;
        } else {
            w = lane < a.k ? 1.f / (1.f + expf(-mysel)) : 0.f;
            if (a.renorm) w = w / butterfly_sum(w);
        }
        if (lane < a.k) a.weights[(size_t)t * a.k + lane] = w;
        __syncwarp();
    }
}

template <bool Q8>
__global__ void __launch_bounds__(256) route_kernel(RouteArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ unsigned s_last;
    const int seg = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.y * ROUTE_WARPS + warp;
    const int s0 = seg * 1024;
    const int seglen = min(1024, a.H - s0);

    if (!Q8) {
        float *xs = reinterpret_cast<float *>(smem_raw);          // [T][1024]
        for (int i = threadIdx.x; i < a.T * 256; i += blockDim.x) {
            const int t = i >> 8, c = i & 255;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (4 * c < seglen) v = *reinterpret_cast<const float4 *>(a.hidden + (size_t)t * a.H + s0 + 4 * c);
            reinterpret_cast<float4 *>(xs)[i] = v;
        }
        __syncthreads();
        if (e < a.E) {
            const float *wr = reinterpret_cast<const float *>(a.w) + (size_t)e * a.H + s0;
            float4 wv[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int c = lane + 32 * j;
                if (4 * c < seglen) {
                    const uint4 u = ldg_stream(wr + 4 * c);
                    wv[j] = make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z),
                                        __uint_as_float(u.w));
                }
            }
            for (int t = 0; t < a.T; ++t) {
                const float4 *xt = reinterpret_cast<const float4 *>(xs + t * 1024);
                float v = 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int c = lane + 32 * j;
                    if (4 * c < seglen) {
                        const float4 xv = xt[c];
                        v = __fmaf_rn(wv[j].x, xv.x, v);
                        v = __fmaf_rn(wv[j].y, xv.y, v);
                        v = __fmaf_rn(wv[j].z, xv.z, v);
                        v = __fmaf_rn(wv[j].w, xv.w, v);
                    }
                }
                v = butterfly_sum(v);
                if (lane == 0) a.partial[((size_t)t * a.E + e) * a.nseg + seg] = v;
            }
        }
    } else {
        // Q8_0 router: segment = 32 blocks; lane l takes block l of the segment
        const int nblk = a.H / 32;
        const int nb = min(32, nblk - seg * 32);
        int8_t *xs = reinterpret_cast<int8_t *>(smem_raw);                    // [T][1024]
        float *xd = reinterpret_cast<float *>(smem_raw + a.T * 1024);        // [T][4]
        uint8_t *wbuf = smem_raw + a.T * 1024 + a.T * 16 + warp * 1088;      // per-warp row segment
        const size_t rb = q8_row_bytes(a.H);
        for (int i = threadIdx.x; i < a.T * 64; i += blockDim.x) {
            const int t = i >> 6, c = i & 63;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (16 * c < 32 * nb) v = *reinterpret_cast<const uint4 *>(a.xq + (size_t)t * rb + q8_q_off(a.H) + s0 + 16 * c);
            reinterpret_cast<uint4 *>(xs)[i] = v;
        }
        for (int i = threadIdx.x; i < a.T * 4; i += blockDim.x) {
            const int t = i >> 2, b = i & 3;
            float v = 0.f;
            if (256 * b < 32 * nb) v = reinterpret_cast<const float *>(a.xq + (size_t)t * rb)[(s0 >> 8) + b];
            xd[i] = v;
        }
        if (e < a.E) {
            const uint8_t *wr = reinterpret_cast<const uint8_t *>(a.w) + (size_t)e * nblk * 34 + (size_t)seg * 32 * 34;
            const int chunks = nb * 34 / 16;   // nb is a multiple of 8 (H % 256 == 0)
            for (int c = lane; c < chunks; c += 32)
                reinterpret_cast<uint4 *>(wbuf)[c] = ldg_stream(wr + 16 * c);
        }
        __syncthreads();
        if (e < a.E) {
            const bool has = lane < nb;
            uint32_t qw[8];
            float dw = 0.f;
            if (has) {
                const uint16_t *h = reinterpret_cast<const uint16_t *>(wbuf + 34 * lane);
                dw = h2f(h[0]);
#pragma unroll
                for (int m = 0; m < 8; ++m) qw[m] = (uint32_t)h[1 + 2 * m] | ((uint32_t)h[2 + 2 * m] << 16);
            }
            for (int t = 0; t < a.T; ++t) {
                float v = 0.f;
                if (has) {
                    const int8_t *xb = xs + t * 1024 + 32 * lane;
                    const int4 x0 = lds128(xb), x1 = lds128(xb + 16);
                    int acc = 0;
                    acc = dp4a(qw[0], (uint32_t)x0.x, acc);
                    acc = dp4a(qw[1], (uint32_t)x0.y, acc);
                    acc = dp4a(qw[2], (uint32_t)x0.z, acc);
                    acc = dp4a(qw[3], (uint32_t)x0.w, acc);
                    acc = dp4a(qw[4], (uint32_t)x1.x, acc);
                    acc = dp4a(qw[5], (uint32_t)x1.y, acc);
                    acc = dp4a(qw[6], (uint32_t)x1.z, acc);
                    acc = dp4a(qw[7], (uint32_t)x1.w, acc);
                    const float dx = xd[t * 4 + (lane >> 3)];
                    v = __fmul_rn(__fmul_rn(dw, dx), (float)acc);
                }
                v = butterfly_sum(v);
                if (lane == 0) a.partial[((size_t)t * a.E + e) * a.nseg + seg] = v;
            }
        }
    }

    // last block: combine segments, top-k, gating
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned total = gridDim.x * gridDim.y;
        s_last = (atomicAdd(a.counter, 1u) == total - 1u);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    route_topk(a, reinterpret_cast<float *>(smem_raw));
    __syncthreads();
    if (threadIdx.x == 0) *a.counter = 0u;
}

cudaError_t launch_route(const RouteArgs &a, int rtype, cudaStream_t s) {
    dim3 grid(a.nseg, (a.E + ROUTE_WARPS - 1) / ROUTE_WARPS);
    size_t stage = rtype == MOE_Q8_0 ? (size_t)a.T * 1024 + a.T * 16 + ROUTE_WARPS * 1088
                                     : (size_t)a.T * 4096;
    size_t topk = (size_t)ROUTE_WARPS * MOE_MAX_EXPERTS * 4;
    size_t smem = stage > topk ? stage : topk;
    cudaError_t err;
    if (rtype == MOE_Q8_0) {
        err = ensure_smem<route_kernel<true>>(smem);
        if (err != cudaSuccess) return err;
        route_kernel<true><<<grid, 256, smem, s>>>(a);
    } else {
        err = ensure_smem<route_kernel<false>>(smem);
        if (err != cudaSuccess) return err;
        route_kernel<false><<<grid, 256, smem, s>>>(a);
    }
    return cudaGetLastError();
}

// ------------------------------------------------------ shared-expert gate
__global__ void __launch_bounds__(32) shared_gate_kernel(const float *__restrict__ hidden, int H,
                                                         const float *__restrict__ w, float *__restrict__ scale) {
    const int t = blockIdx.x;
    const float s = shared_gate_weight(w, hidden + (size_t)t * H, H, threadIdx.x);
    if (threadIdx.x == 0) scale[t] = s;
}

cudaError_t launch_shared_gate(const float *hidden, int T, int H, const float *w, float *scale, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    shared_gate_kernel<<<T, 32, 0, s>>>(hidden, H, w, scale);
    return cudaGetLastError();
}

// ------------------------------------------------- expert-parallel partials
// y[i] = sum over ranks r = 0, 1, ... of parts[r][i], added in rank order
// (README "MoE resolve": tier cards compute their slots and the partial
// outputs are summed; a fixed order keeps the sum reproducible).
__global__ void __launch_bounds__(256) sum_partials_kernel(const float4 *__restrict__ parts, int R, size_t n4,
                                                           float4 *__restrict__ y) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
        float4 s = parts[i];
        for (int r = 1; r < R; ++r) {
            const float4 v = parts[(size_t)r * n4 + i];
            s.x = __fadd_rn(s.x, v.x);
            s.y = __fadd_rn(s.y, v.y);
            s.z = __fadd_rn(s.z, v.z);
            s.w = __fadd_rn(s.w, v.w);
        }
        y[i] = s;
    }
}

cudaError_t launch_sum_partials(const float *parts, int R, size_t n, float *y, cudaStream_t s) {
    const size_t n4 = n / 4;
    if (n4 == 0) return cudaSuccess;
    size_t blocks = (n4 + 255) / 256;
    const size_t cap = (size_t)num_sms() * 8;
    if (blocks > cap) blocks = cap;
    sum_partials_kernel<<<(unsigned)blocks, 256, 0, s>>>(reinterpret_cast<const float4 *>(parts), R, n4,
                                                         reinterpret_cast<float4 *>(y));
    return cudaGetLastError();
}

// ----------------------------------------------------------------- packing
// One thread per (row, record): copies that row's bytes of the record from
// the GGUF block row into the record's planes (layout stated in moe.h).
__global__ void pack_kernel(const uint8_t *__restrict__ src, int qtype, int rows, int cols,
                            uint8_t *__restrict__ dst) {
    const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    int nrec;
    size_t tile, row_bytes;
    switch (qtype) {
        case MOE_Q4_K: nrec = FQ4K::nrec(cols); tile = FQ4K::tile_bytes(cols); row_bytes = (size_t)cols / 256 * 144; break;
        case MOE_Q2_K: nrec = FQ2K::nrec(cols); tile = FQ2K::tile_bytes(cols); row_bytes = (size_t)cols / 256 * 84; break;
        case MOE_Q8_0: nrec = FQ80::nrec(cols); tile = FQ80::tile_bytes(cols); row_bytes = (size_t)cols / 32 * 34; break;
        case MOE_Q6_K: nrec = FQ6K::nrec(cols); tile = FQ6K::tile_bytes(cols); row_bytes = (size_t)cols / 256 * 210; break;
        case MOE_Q3_K: nrec = FQ3K::nrec(cols); tile = FQ3K::tile_bytes(cols); row_bytes = (size_t)cols / 256 * 110; break;
        default: nrec = FMX4::nrec(cols); tile = FMX4::tile_bytes(cols); row_bytes = (size_t)cols / 32 * 17; break;
    }
    if (tid >= (long long)rows * nrec) return;
    const int row = (int)(tid / nrec), r = (int)(tid % nrec);
    const int lane = row & 31;
    const uint8_t *s = src + (size_t)row * row_bytes;
    uint8_t *base = dst + (size_t)(row >> 5) * tile;
    if (qtype == MOE_Q4_K) {
        const uint8_t *b = s + (size_t)r * 144;
        uint8_t *o = base + FQ4K::rec_off(cols, r);
        for (int p = 0; p < 9; ++p)
            for (int i = 0; i < 16; ++i) o[p * 512 + lane * 16 + i] = b[16 * p + i];
    } else if (qtype == MOE_Q2_K) {
        const uint8_t *b = s + (size_t)r * 84;
        uint8_t *o = base + FQ2K::rec_off(cols, r);
        for (int p = 0; p < 5; ++p)
            for (int i = 0; i < 16; ++i) o[p * 512 + lane * 16 + i] = b[16 * p + i];
        for (int i = 0; i < 4; ++i) o[5 * 512 + lane * 4 + i] = b[80 + i];
    } else if (qtype == MOE_Q6_K) {
        const uint8_t *b = s + (size_t)r * 210;
        uint8_t *o = base + FQ6K::rec_off(cols, r);
        for (int p = 0; p < 13; ++p)
            for (int i = 0; i < 16; ++i) o[p * 512 + lane * 16 + i] = b[16 * p + i];
        for (int i = 0; i < 4; ++i) o[13 * 512 + lane * 4 + i] = i < 2 ? b[208 + i] : 0;
    } else if (qtype == MOE_Q3_K) {
        const uint8_t *b = s + (size_t)r * 110;
        uint8_t *o = base + FQ3K::rec_off(cols, r);
        for (int p = 0; p < 7; ++p)
            for (int i = 0; i < 16; ++i) o[p * 512 + lane * 16 + i] = (16 * p + i < 110) ? b[16 * p + i] : 0;
    } else if (qtype == MOE_Q8_0) {
        uint8_t *o = base + FQ80::rec_off(cols, r);
        for (int bb = 0; bb < 8; ++bb) {
            const uint8_t *b = s + (size_t)(8 * r + bb) * 34;
            for (int i = 0; i < 32; ++i) o[(2 * bb + (i >> 4)) * 512 + lane * 16 + (i & 15)] = b[2 + i];
            o[16 * 512 + lane * 16 + 2 * bb] = b[0];
            o[16 * 512 + lane * 16 + 2 * bb + 1] = b[1];
        }
    } else {
        const int nb = FMX4::rec_blocks(cols, r);
        uint8_t *o = base + FMX4::rec_off(cols, r);
        for (int bb = 0; bb < 8; ++bb) {
            if (bb < nb) {
                const uint8_t *b = s + (size_t)(8 * r + bb) * 17;
                for (int i = 0; i < 16; ++i) o[bb * 512 + lane * 16 + i] = b[1 + i];
                o[nb * 512 + lane * 8 + bb] = b[0];
            } else {
                o[nb * 512 + lane * 8 + bb] = 0;
            }
        }
    }
}

cudaError_t launch_pack(const uint8_t *src, int qtype, int rows, int cols, uint8_t *dst, cudaStream_t s) {
    int nrec = qtype == MOE_MXFP4 ? FMX4::nrec(cols) : cols / 256;
    long long n = (long long)rows * nrec;
    if (n == 0) return cudaSuccess;
    pack_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(src, qtype, rows, cols, dst);
    return cudaGetLastError();
}

// ------------------------------------------------------------ row-dot hook
// One warp walks the records of the row's tile; the lane owning the row
// writes its exact sub-block dots (the same decode and dot code the FFN runs).
template <class F>
__device__ void row_dots_fixed(const uint8_t *packed, int cols, int row, const Act &x, int32_t *out) {
    const int lane = threadIdx.x & 31;
    const uint8_t *tile = packed + (size_t)(row >> 5) * F::tile_bytes(cols);
    for (int r = 0; r < F::nrec(cols); ++r) {
        typename F::W w;
        F::load(w, tile + F::rec_off(cols, r), 0, lane);
        int is[F::NSUB];
        F::isums(w, x, r * F::QK, 8, is);
        if (lane == (row & 31))
            for (int j = 0; j < F::NSUB; ++j) out[r * F::NSUB + j] = is[j];
    }
}

__global__ void row_dots_kernel(const uint8_t *packed, int qtype, int cols, int row, const uint8_t *xq,
                                int32_t *out) {
    const Act x = act_view(xq, cols);
    const int lane = threadIdx.x & 31;
    if (qtype == MOE_Q4_K) row_dots_fixed<FQ4K>(packed, cols, row, x, out);
    else if (qtype == MOE_Q2_K) row_dots_fixed<FQ2K>(packed, cols, row, x, out);
    else if (qtype == MOE_Q8_0) row_dots_fixed<FQ80>(packed, cols, row, x, out);
    else if (qtype == MOE_Q6_K) row_dots_fixed<FQ6K>(packed, cols, row, x, out);
    else if (qtype == MOE_Q3_K) row_dots_fixed<FQ3K>(packed, cols, row, x, out);
    else {
        const uint8_t *tile = packed + (size_t)(row >> 5) * FMX4::tile_bytes(cols);
        for (int r = 0; r < FMX4::nrec(cols); ++r) {
            const int nb = FMX4::rec_blocks(cols, r);
            FMX4::W w;
            FMX4::load(w, tile + FMX4::rec_off(cols, r), nb, lane);
            int is[8];
            FMX4::isums(w, x, r * 256, nb, is);
            if (lane == (row & 31))
                for (int j = 0; j < nb; ++j) out[r * 8 + j] = is[j];
        }
    }
}

cudaError_t launch_row_dots(const uint8_t *packed, int qtype, int cols, int row, const uint8_t *xq,
                            int32_t *out, cudaStream_t s) {
    row_dots_kernel<<<1, 32, 0, s>>>(packed, qtype, cols, row, xq, out);
    return cudaGetLastError();
}

int smem_optin() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 48 * 1024;
    if (cached[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess || v <= 0)
            v = 48 * 1024;
        cached[dev] = v;
    }
    return cached[dev];
}

int num_sms() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (cached[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
        cached[dev] = v;
    }
    return cached[dev];
}

}  // namespace moe
