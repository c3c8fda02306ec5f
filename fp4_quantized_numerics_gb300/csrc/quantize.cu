// quantize.cu -- fused RHT + block quantization, tensor amax, dequantization
// and quality statistics for sm_103a.
//
// Method ([ZC] zhichai.net post "Shrinkage Bias: The Hidden Geometric Trap in
// FP4 Training ... and the UFP4 Fix", Key points "The cause", "The RHT
// paradox", "The fix -- UFP4"; [AN] autonainews.com "UFP4 Eliminates Shrinkage
// Bias ...", "The UFP4 Recipe"): 16-element blocks along K are optionally
// rotated by the sign-randomised 16-point Hadamard transform, scaled by an
// E4M3 block scale under an FP32 tensor scale, and rounded onto the E2M1 or
// E1M2 grid, to nearest-even or stochastically.  The exact arithmetic is the
// contract in include/ufp4.h.
//
// Design (memory-bound, ~2.56 B/elem of algorithmic traffic for BF16 input):
//  * Row-wise: one thread owns 8 consecutive elements (one 16-byte load), a
//    lane pair owns one 16-block, so each warp load instruction reads 512
//    contiguous bytes.  The 16-point transform is three in-register butterfly
//    stages plus one stage across the lane pair (shuffle).  Codes leave as one
//    32-bit store per thread (128 contiguous bytes per warp).
//  * Column-wise (the quantization of X^T): a warp owns 16 rows x 128 columns;
//    each lane loads 16 rows x 4 columns (8-byte loads, 256 contiguous bytes
//    per warp instruction) and runs four full 16-point transforms in registers.
//  * The 1/4 of the orthonormal RHT is folded into the per-code multiplier
//    table (exact power-of-two scaling).
//  * The tensor amax needs every element before the first code: a first pass
//    writes one partial maximum per CTA into the caller's workspace; the
//    quantization pass reduces those partials in its prologue (no atomics, no
//    memset, deterministic).
#include "common.cuh"
#include "internal.h"

#include <algorithm>
#include <cfloat>
#include <type_traits>

namespace ufp4 {

namespace {

constexpr int kThreads = 256;

struct Args {
    const void *x;
    int64_t rows, cols, ld;     // input as stored
    int64_t out_rows, k, kpad;  // result: out_rows x k, padded to kpad
    int64_t nkt;                // kpad / 64
    uint64_t rht_seed, sr_seed, sr_counter, elem_base;
    const float *amax_in;
    const float *partials;
    float *partials_out;
    int n_partials;
    uint32_t *status;
    uint8_t *codes, *scales;
    float *tensor_scale;
    double *stats_out;
};

// ------------------------------------------------------------------ loads
// 8 consecutive elements as fp32, sign-flipped by the 8-bit mask `sflip`
// (bit j set: negate element j).
__device__ __forceinline__ void load8(const __nv_bfloat16 *p, uint32_t sflip, float v[8]) {
    uint4 w = *reinterpret_cast<const uint4 *>(p);
    uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        u[i] ^= (((sflip >> (2 * i)) & 1u) << 15) | (((sflip >> (2 * i + 1)) & 1u) << 31);
        v[2 * i] = bf16lo(u[i]);
        v[2 * i + 1] = bf16hi(u[i]);
    }
}
__device__ __forceinline__ void load8(const float *p, uint32_t sflip, float v[8]) {
    const float4 a = *reinterpret_cast<const float4 *>(p);
    const float4 b = *reinterpret_cast<const float4 *>(p + 4);
    const float t[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(__float_as_uint(t[i]) ^ (((sflip >> i) & 1u) << 31));
}

// 4 consecutive columns of one row as fp32 (no sign flip: column-wise signs
// depend on the row, applied by the caller).
__device__ __forceinline__ void load4(const __nv_bfloat16 *p, float v[4]) {
    const uint2 w = *reinterpret_cast<const uint2 *>(p);
    v[0] = bf16lo(w.x); v[1] = bf16hi(w.x); v[2] = bf16lo(w.y); v[3] = bf16hi(w.y);
}
__device__ __forceinline__ void load4(const float *p, float v[4]) {
    const float4 a = *reinterpret_cast<const float4 *>(p);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
}

// Row-wise unit values: the lane pair (2i, 2i+1) holds one 16-block, lane
// parity h holds elements 8h..8h+7.  With RHT the result is 4*y (the caller
// applies the exact factor 1/4).  Every lane of the warp must call this.
template <class In, bool RHT>
__device__ __forceinline__ void unit_values(const In *x, int64_t ld, int64_t r, int64_t c8,
                                            bool load, uint32_t sflip, float hsign, float v[8]) {
    if (load) {
        load8(x + r * ld + c8 * 8, RHT ? sflip : 0u, v);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = 0.0f;
    }
    if (RHT) {
        fwht8(v);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float o = __shfl_xor_sync(0xffffffffu, v[i], 1);
            v[i] = fmaf(hsign, v[i], o);   // h=0: o + v ; h=1: o - v  (one rounding)
        }
    }
}

// Position of a thread's unit in a row-major grid of units, advanced by a
// fixed stride without divisions.
struct Pos {
    int64_t r, c;
};
__device__ __forceinline__ void advance(Pos &p, int64_t dr, int64_t dc, int64_t upr) {
    p.r += dr;
    p.c += dc;
    if (p.c >= upr) { p.c -= upr; p.r += 1; }
}

// Tensor scale from the partial maxima (or amax_in); also fills the per-code
// multiplier table k[e] = min(S_enc / E4M3(e), FLT_MAX) * kfold.
__device__ __forceinline__ void tensor_scale_prologue(const Args &a, float qmax, float kfold,
                                                      float *s_k, float *s_red, float &S_enc) {
    float m = 0.0f;
    if (a.amax_in) {
        m = *a.amax_in;
    } else {
        for (int i = threadIdx.x; i < a.n_partials; i += blockDim.x) m = max_nan(m, a.partials[i]);
#pragma unroll
        for (int o = 16; o; o >>= 1) m = max_nan(m, __shfl_xor_sync(0xffffffffu, m, o));
        if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = m;
        __syncthreads();
        m = s_red[0];
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w) m = max_nan(m, s_red[w]);
    }
    const float A_t = m;
    float se = 1.0f, sd = 1.0f;
    if (A_t > 0.0f) {
        const float num = 448.0f * qmax;
        se = __fdiv_rn(num, A_t);
        if (se > kFltMax) se = kFltMax;
        sd = __fdiv_rn(A_t, num);
    }
    S_enc = se;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        if (a.tensor_scale) *a.tensor_scale = sd;
        if (a.status) *a.status = (isfinite(A_t) ? 0u : 1u);
    }
    for (int c = threadIdx.x; c < 256; c += blockDim.x) {
        const float d = e4m3_to_f32((uint32_t)c);
        float kk = 0.0f;
        if (d > 0.0f) {
            kk = __fdiv_rn(se, d);
            if (kk > kFltMax) kk = kFltMax;
        } else if (!(d == 0.0f)) {
            kk = d;   // NaN code: only reachable from non-finite input
        }
        s_k[c] = kk * kfold;
    }
    __syncthreads();
}

// Block scale code of a block whose magnitude maximum is amax.
__device__ __forceinline__ uint32_t block_scale(float amax, float qmax, float S_enc) {
    return e4m3_from_f32(__fmul_rn(__fdiv_rn(amax, qmax), S_enc));
}

// Codes of 8 values q (already multiplied by k) as 8 nibbles, element j in
// bits 4j..4j+3.  `i0` is the logical output index of element 0 (multiple of
// 8) for stochastic rounding.
template <int GRID, int ROUND>
__device__ __forceinline__ uint32_t codes8(const float q[8], const Args &a, uint64_t i0) {
    uint32_t w = 0;
    if (ROUND == kRTNE) {
        if (GRID == kE2M1) {
#pragma unroll
            for (int j = 0; j < 4; ++j) w |= e2m1x2_rn(q[2 * j], q[2 * j + 1]) << (8 * j);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) w |= e1m2_rn(q[j]) << (4 * j);
        }
    } else {
        const uint2 key = make_uint2((uint32_t)a.sr_seed, (uint32_t)(a.sr_seed >> 32));
        const uint64_t c0 = i0 >> 2;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const uint64_t c = c0 + t;
            const uint4 r = philox4x32_10(
                make_uint4((uint32_t)c, (uint32_t)(c >> 32), (uint32_t)a.sr_counter,
                           (uint32_t)(a.sr_counter >> 32)), key);
            w |= sr_code<GRID>(q[4 * t + 0], r.x) << (16 * t + 0);
            w |= sr_code<GRID>(q[4 * t + 1], r.y) << (16 * t + 4);
            w |= sr_code<GRID>(q[4 * t + 2], r.z) << (16 * t + 8);
            w |= sr_code<GRID>(q[4 * t + 3], r.w) << (16 * t + 12);
        }
    }
    return w;
}

// Zero the scale entries of the padding rows out_rows..rpad-1.
__device__ __forceinline__ void zero_pad_rows(const Args &a) {
    const int64_t rpad = rpad_of(a.out_rows);
    const int64_t nb = a.kpad / 16;
    const int64_t n = (rpad - a.out_rows) * nb;
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < n;
         t += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = a.out_rows + t / nb, b = t % nb;
        a.scales[scale_offset(r, b, a.nkt)] = 0;
    }
}

// ======================================================= row-wise kernels
template <class In, bool RHT>
__global__ void __launch_bounds__(kThreads) k_amax_rowwise(Args a) {
    __shared__ float s_red[kThreads / 32];
    const uint32_t lane = threadIdx.x & 31;
    const uint32_t h = lane & 1;
    const uint32_t sflip = RHT ? ((rht_sign_mask(a.rht_seed) >> (8 * h)) & 0xFFu) : 0u;
    const float hsign = h ? -1.0f : 1.0f;
    const int64_t upr = a.k / 8;  // only real elements
    const int64_t total = a.out_rows * upr;
    const int64_t T = (int64_t)gridDim.x * blockDim.x;
    const int64_t tid = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    Pos p{tid / upr, tid % upr};
    const int64_t dr = T / upr, dc = T % upr;
    const int64_t iters = (total + T - 1) / T;
    float m = 0.0f;
    for (int64_t it = 0; it < iters; ++it) {
        const bool valid = p.r < a.out_rows;
        float v[8];
        unit_values<In, RHT>(static_cast<const In *>(a.x), a.ld, p.r, p.c, valid, sflip, hsign, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) m = max_nan(m, fabsf(v[i]));
        advance(p, dr, dc, upr);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) m = max_nan(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) s_red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kThreads / 32; ++w) m = max_nan(m, s_red[w]);
        a.partials_out[blockIdx.x] = RHT ? m * 0.25f : m;
    }
}

template <class In, int GRID, int ROUND, bool RHT>
__global__ void __launch_bounds__(kThreads) k_quant_rowwise(Args a) {
    __shared__ float s_k[256];
    __shared__ float s_red[kThreads / 32];
    const float qmax = GRID == kE2M1 ? 6.0f : 3.5f;
    float S_enc;
    tensor_scale_prologue(a, qmax, RHT ? 0.25f : 1.0f, s_k, s_red, S_enc);

    const uint32_t lane = threadIdx.x & 31;
    const uint32_t h = lane & 1;
    const uint32_t sflip = RHT ? ((rht_sign_mask(a.rht_seed) >> (8 * h)) & 0xFFu) : 0u;
    const float hsign = h ? -1.0f : 1.0f;
    const int64_t upr = a.kpad / 8;   // units per row, padding included
    const int64_t kvalid8 = a.k / 8;
    const int64_t total = a.out_rows * upr;
    const int64_t T = (int64_t)gridDim.x * blockDim.x;
    const int64_t tid = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    Pos p{tid / upr, tid % upr};
    const int64_t dr = T / upr, dc = T % upr;
    const int64_t iters = (total + T - 1) / T;
    const In *x = static_cast<const In *>(a.x);
    const int64_t cstride = a.kpad / 2;
    for (int64_t it = 0; it < iters; ++it) {
        const bool valid = p.r < a.out_rows;
        float v[8];
        unit_values<In, RHT>(x, a.ld, p.r, p.c, valid && p.c < kvalid8, sflip, hsign, v);
        float m = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        if (RHT) m *= 0.25f;
        const uint32_t e = block_scale(m, qmax, S_enc);
        const float kk = s_k[e];
        float q[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = __fmul_rn(v[i], kk);
        uint32_t w = codes8<GRID, ROUND>(q, a, a.elem_base + (uint64_t)(p.r * a.k + p.c * 8));
        if (e == 0) w = 0;
        if (valid) {
            *reinterpret_cast<uint32_t *>(a.codes + p.r * cstride + p.c * 4) = w;
            if (h == 0) a.scales[scale_offset(p.r, p.c >> 1, a.nkt)] = (uint8_t)e;
        }
        advance(p, dr, dc, upr);
    }
    zero_pad_rows(a);
}

// ==================================================== column-wise kernels
// Tile: 128 output rows (input columns) x 128 output k (input rows); warp w
// owns 16-block kb = tile_k * 8 + w, lane l owns input columns 4l..4l+3.
template <class In, bool RHT>
__device__ __forceinline__ void col_block(const In *x, int64_t ld, int64_t r0, int64_t c,
                                          uint32_t smask, float v[4][16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        float t[4];
        load4(x + (r0 + i) * ld + c, t);
        const float s = (RHT && ((smask >> i) & 1u)) ? -1.0f : 1.0f;
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j][i] = RHT ? t[j] * s : t[j];
    }
    if (RHT) {
#pragma unroll
        for (int j = 0; j < 4; ++j) fwht16(v[j]);
    }
}

template <class In, bool RHT>
__global__ void __launch_bounds__(kThreads) k_amax_colwise(Args a) {
    __shared__ float s_red[kThreads / 32];
    const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t smask = RHT ? rht_sign_mask(a.rht_seed) : 0u;
    const int64_t C = a.cols, R = a.rows;
    const int64_t ntc = (C + 127) / 128, ntk = (R + 127) / 128;
    float m = 0.0f;
    for (int64_t t = blockIdx.x; t < ntc * ntk; t += gridDim.x) {
        const int64_t tk = t % ntk, tc = t / ntk;
        const int64_t r0 = (tk * 8 + warp) * 16;
        const int64_t c = tc * 128 + lane * 4;
        if (r0 >= R || c >= C) continue;
        float v[4][16];
        col_block<In, RHT>(static_cast<const In *>(a.x), a.ld, r0, c, smask, v);
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int i = 0; i < 16; ++i) m = max_nan(m, fabsf(v[j][i]));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) m = max_nan(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) s_red[warp] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kThreads / 32; ++w) m = max_nan(m, s_red[w]);
        a.partials_out[blockIdx.x] = RHT ? m * 0.25f : m;
    }
}

template <int GRID, int ROUND>
__device__ __forceinline__ uint2 codes16(const float q[16], const Args &a, uint64_t i0) {
    float lo[8], hi[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) { lo[i] = q[i]; hi[i] = q[8 + i]; }
    return make_uint2(codes8<GRID, ROUND>(lo, a, i0), codes8<GRID, ROUND>(hi, a, i0 + 8));
}

template <class In, int GRID, int ROUND, bool RHT>
__global__ void __launch_bounds__(kThreads) k_quant_colwise(Args a) {
    __shared__ float s_k[256];
    __shared__ float s_red[kThreads / 32];
    const float qmax = GRID == kE2M1 ? 6.0f : 3.5f;
    float S_enc;
    tensor_scale_prologue(a, qmax, RHT ? 0.25f : 1.0f, s_k, s_red, S_enc);

    const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t smask = RHT ? rht_sign_mask(a.rht_seed) : 0u;
    const int64_t C = a.cols, R = a.rows;           // input; output is C x R
    const int64_t nbk = a.kpad / 16;                 // output blocks per row (with pad)
    const int64_t ntc = (C + 127) / 128, ntk = (nbk + 7) / 8;
    const int64_t cstride = a.kpad / 2;
    for (int64_t t = blockIdx.x; t < ntc * ntk; t += gridDim.x) {
        const int64_t tk = t % ntk, tc = t / ntk;
        const int64_t kb = tk * 8 + warp;
        const int64_t r0 = kb * 16;
        const int64_t c = tc * 128 + lane * 4;
        if (kb >= nbk || c >= C) continue;
        if (r0 >= R) {   // padding blocks along k
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                *reinterpret_cast<uint2 *>(a.codes + (c + j) * cstride + r0 / 2) = make_uint2(0, 0);
                a.scales[scale_offset(c + j, kb, a.nkt)] = 0;
            }
            continue;
        }
        float v[4][16];
        col_block<In, RHT>(static_cast<const In *>(a.x), a.ld, r0, c, smask, v);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float m = 0.0f;
#pragma unroll
            for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(v[j][i]));
            if (RHT) m *= 0.25f;
            const uint32_t e = block_scale(m, qmax, S_enc);
            const float kk = s_k[e];
            float q[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) q[i] = __fmul_rn(v[j][i], kk);
            uint2 w = codes16<GRID, ROUND>(q, a, a.elem_base + (uint64_t)((c + j) * R + r0));
            if (e == 0) w = make_uint2(0, 0);
            *reinterpret_cast<uint2 *>(a.codes + (c + j) * cstride + r0 / 2) = w;
            a.scales[scale_offset(c + j, kb, a.nkt)] = (uint8_t)e;
        }
    }
    zero_pad_rows(a);
}

// ============================================================= statistics
// Per element: deq = fl32(fl32(v e) S_dec), A = y (rotated input);
// sums of deq*A, A*A, (A-deq)^2, (v - a) over a != 0, count.
struct Acc {
    double aq = 0, aa = 0, e2 = 0, bias = 0, cnt = 0;
};

__device__ __forceinline__ void acc_block8(Acc &acc, const float y[8], uint32_t w, float e,
                                           float S_dec, int grid, float qmax) {
    float aq = 0, aa = 0, e2 = 0, bias = 0, cnt = 0;
    const float unit = __fmul_rn(e, S_dec);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t c = (w >> (4 * j)) & 0xFu;
        const float v = grid_value(grid, c);
        const float sv = (c & 8u) ? -v : v;
        const float dq = __fmul_rn(__fmul_rn(sv, e), S_dec);
        aq += dq * y[j];
        aa += y[j] * y[j];
        e2 += (y[j] - dq) * (y[j] - dq);
        if (e > 0.0f) {
            const float g = fminf(fabsf(y[j]) / unit, qmax);
            if (g != 0.0f) { bias += v - g; cnt += 1.0f; }
        }
    }
    acc.aq += aq; acc.aa += aa; acc.e2 += e2; acc.bias += bias; acc.cnt += cnt;
}

__device__ void stats_reduce(Acc acc, double *out) {
    __shared__ double s[kThreads / 32][5];
    double v[5] = {acc.aq, acc.aa, acc.e2, acc.bias, acc.cnt};
#pragma unroll
    for (int i = 0; i < 5; ++i)
#pragma unroll
        for (int o = 16; o; o >>= 1) v[i] += __shfl_xor_sync(0xffffffffu, v[i], o);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0)
        for (int i = 0; i < 5; ++i) s[warp][i] = v[i];
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int i = 0; i < 5; ++i) {
            double t = 0;
            for (int w = 0; w < kThreads / 32; ++w) t += s[w][i];
            out[blockIdx.x * 8 + i] = t;
        }
    }
}

template <class In, bool RHT>
__global__ void __launch_bounds__(kThreads) k_stats_rowwise(Args a, int grid) {
    const float qmax = grid_qmax(grid);
    const float S_dec = *a.tensor_scale;
    const uint32_t lane = threadIdx.x & 31, h = lane & 1;
    const uint32_t sflip = RHT ? ((rht_sign_mask(a.rht_seed) >> (8 * h)) & 0xFFu) : 0u;
    const float hsign = h ? -1.0f : 1.0f;
    const int64_t upr = a.k / 8;
    const int64_t total = a.out_rows * upr;
    const int64_t T = (int64_t)gridDim.x * blockDim.x;
    const int64_t tid = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    Pos p{tid / upr, tid % upr};
    const int64_t dr = T / upr, dc = T % upr;
    const int64_t iters = (total + T - 1) / T;
    Acc acc;
    for (int64_t it = 0; it < iters; ++it) {
        const bool valid = p.r < a.out_rows;
        float v[8];
        unit_values<In, RHT>(static_cast<const In *>(a.x), a.ld, p.r, p.c, valid, sflip, hsign, v);
        if (valid) {
            if (RHT)
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] *= 0.25f;
            const uint32_t w = *reinterpret_cast<const uint32_t *>(a.codes + p.r * (a.kpad / 2) + p.c * 4);
            const float e = e4m3_to_f32(a.scales[scale_offset(p.r, p.c >> 1, a.nkt)]);
            acc_block8(acc, v, w, e, S_dec, grid, qmax);
        }
        advance(p, dr, dc, upr);
    }
    stats_reduce(acc, a.stats_out);
}

template <class In, bool RHT>
__global__ void __launch_bounds__(kThreads) k_stats_colwise(Args a, int grid) {
    const float qmax = grid_qmax(grid);
    const float S_dec = *a.tensor_scale;
    const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t smask = RHT ? rht_sign_mask(a.rht_seed) : 0u;
    const int64_t C = a.cols, R = a.rows;
    const int64_t ntc = (C + 127) / 128, ntk = (R + 127) / 128;
    const int64_t cstride = a.kpad / 2;
    Acc acc;
    for (int64_t t = blockIdx.x; t < ntc * ntk; t += gridDim.x) {
        const int64_t tk = t % ntk, tc = t / ntk;
        const int64_t kb = tk * 8 + warp;
        const int64_t r0 = kb * 16;
        const int64_t c = tc * 128 + lane * 4;
        if (r0 >= R || c >= C) continue;
        float v[4][16];
        col_block<In, RHT>(static_cast<const In *>(a.x), a.ld, r0, c, smask, v);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (RHT)
#pragma unroll
                for (int i = 0; i < 16; ++i) v[j][i] *= 0.25f;
            const uint2 w = *reinterpret_cast<const uint2 *>(a.codes + (c + j) * cstride + r0 / 2);
            const float e = e4m3_to_f32(a.scales[scale_offset(c + j, kb, a.nkt)]);
            acc_block8(acc, &v[j][0], w.x, e, S_dec, grid, qmax);
            acc_block8(acc, &v[j][8], w.y, e, S_dec, grid, qmax);
        }
    }
    stats_reduce(acc, a.stats_out);
}

// ========================================================== dequantization
template <bool INV>
__global__ void __launch_bounds__(kThreads) k_dequant(const uint8_t *codes, const uint8_t *scales,
                                                      const float *ts, int64_t rows, int64_t k,
                                                      int grid, uint64_t rht_seed, float *out,
                                                      int64_t ld) {
    const float S_dec = *ts;
    const uint32_t lane = threadIdx.x & 31, h = lane & 1;
    const uint32_t smask = INV ? ((rht_sign_mask(rht_seed) >> (8 * h)) & 0xFFu) : 0u;
    const float hsign = h ? -1.0f : 1.0f;
    const int64_t kpad = kpad_of(k), nkt = kpad / 64;
    const int64_t upr = k / 8;
    const int64_t total = rows * upr;
    const int64_t T = (int64_t)gridDim.x * blockDim.x;
    const int64_t tid = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    Pos p{tid / upr, tid % upr};
    const int64_t dr = T / upr, dc = T % upr;
    const int64_t iters = (total + T - 1) / T;
    for (int64_t it = 0; it < iters; ++it) {
        const bool valid = p.r < rows;
        float v[8];
        if (valid) {
            const uint32_t w = *reinterpret_cast<const uint32_t *>(codes + p.r * (kpad / 2) + p.c * 4);
            const float e = e4m3_to_f32(scales[scale_offset(p.r, p.c >> 1, nkt)]);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t c = (w >> (4 * j)) & 0xFu;
                const float g = grid_value(grid, c);
                v[j] = __fmul_rn(__fmul_rn((c & 8u) ? -g : g, e), S_dec);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = 0.0f;
        }
        if (INV) {
            fwht8(v);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float o = __shfl_xor_sync(0xffffffffu, v[i], 1);
                v[i] = fmaf(hsign, v[i], o);
                v[i] *= ((smask >> i) & 1u) ? -0.25f : 0.25f;
            }
        }
        if (valid) {
            float *o = out + p.r * ld + p.c * 8;
            *reinterpret_cast<float4 *>(o) = make_float4(v[0], v[1], v[2], v[3]);
            *reinterpret_cast<float4 *>(o + 4) = make_float4(v[4], v[5], v[6], v[7]);
        }
        advance(p, dr, dc, upr);
    }
}

// ================================================================ dispatch
template <class In>
cudaError_t quantize_typed(const QuantLaunch &q, Args &a, void *ws, cudaStream_t s) {
    const int sms = num_sms();
    const bool col = q.colwise != 0;
    // pass 1: tensor amax
    if (!q.amax_in) {
        int64_t work;
        if (!col) work = (a.out_rows * (a.k / 8) + kThreads - 1) / kThreads;
        else work = ((a.cols + 127) / 128) * ((a.rows + 127) / 128);
        int g = (int)std::min<int64_t>(std::max<int64_t>(work, 1), (int64_t)sms * 8);
        if (g > kMaxPartials) g = kMaxPartials;
        a.partials_out = reinterpret_cast<float *>(static_cast<char *>(ws) + kWsPartials);
        a.partials = a.partials_out;
        a.n_partials = g;
        if (!col) {
            if (q.rht) k_amax_rowwise<In, true><<<g, kThreads, 0, s>>>(a);
            else k_amax_rowwise<In, false><<<g, kThreads, 0, s>>>(a);
        } else {
            if (q.rht) k_amax_colwise<In, true><<<g, kThreads, 0, s>>>(a);
            else k_amax_colwise<In, false><<<g, kThreads, 0, s>>>(a);
        }
        cudaError_t err = cudaGetLastError();
        if (err != cudaSuccess) return err;
    }
    // pass 2: quantize
    int64_t work;
    if (!col) work = (a.out_rows * (a.kpad / 8) + kThreads - 1) / kThreads;
    else work = ((a.cols + 127) / 128) * ((a.kpad / 16 + 7) / 8);
    const int g = (int)std::min<int64_t>(std::max<int64_t>(work, 1), (int64_t)sms * 8);
#define UFP4_Q(COLW, GRID, ROUND, RHT)                                        \
    if (col == COLW && q.grid == GRID && q.round == ROUND && (q.rht != 0) == RHT) { \
        if (COLW) k_quant_colwise<In, GRID, ROUND, RHT><<<g, kThreads, 0, s>>>(a); \
        else k_quant_rowwise<In, GRID, ROUND, RHT><<<g, kThreads, 0, s>>>(a);     \
        return cudaGetLastError();                                              \
    }
    UFP4_Q(false, kE2M1, kRTNE, false) UFP4_Q(false, kE2M1, kRTNE, true)
    UFP4_Q(false, kE2M1, kSR, false)   UFP4_Q(false, kE2M1, kSR, true)
    UFP4_Q(false, kE1M2, kRTNE, false) UFP4_Q(false, kE1M2, kRTNE, true)
    UFP4_Q(false, kE1M2, kSR, false)   UFP4_Q(false, kE1M2, kSR, true)
    UFP4_Q(true, kE2M1, kRTNE, false)  UFP4_Q(true, kE2M1, kRTNE, true)
    UFP4_Q(true, kE2M1, kSR, false)    UFP4_Q(true, kE2M1, kSR, true)
    UFP4_Q(true, kE1M2, kRTNE, false)  UFP4_Q(true, kE1M2, kRTNE, true)
    UFP4_Q(true, kE1M2, kSR, false)    UFP4_Q(true, kE1M2, kSR, true)
#undef UFP4_Q
    return cudaErrorInvalidValue;
}

Args make_args(const QuantLaunch &q, void *ws) {
    Args a{};
    a.x = q.x;
    a.rows = q.rows; a.cols = q.cols; a.ld = q.ld;
    a.out_rows = q.out_rows; a.k = q.k; a.kpad = kpad_of(q.k); a.nkt = a.kpad / 64;
    a.rht_seed = q.rht_seed; a.sr_seed = q.sr_seed; a.sr_counter = q.sr_counter;
    a.elem_base = q.elem_base;
    a.amax_in = q.amax_in;
    a.status = ws ? reinterpret_cast<uint32_t *>(static_cast<char *>(ws) + kWsStatus) : nullptr;
    a.codes = q.codes; a.scales = q.scales; a.tensor_scale = q.tensor_scale;
    return a;
}

}  // namespace

int num_sms() {
    static int cached[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    if (!cached[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = n > 0 ? n : 1;
    }
    return cached[dev];
}

cudaError_t launch_quantize(const QuantLaunch &q, void *ws, cudaStream_t s) {
    Args a = make_args(q, ws);
    if (q.dtype == 0) return quantize_typed<__nv_bfloat16>(q, a, ws, s);
    return quantize_typed<float>(q, a, ws, s);
}

cudaError_t launch_dequantize(const uint8_t *codes, const uint8_t *scales, const float *ts,
                              int64_t rows, int64_t k, int grid, int inverse_rht,
                              uint64_t rht_seed, float *out, int64_t ld_out, cudaStream_t s) {
    const int64_t work = (rows * (k / 8) + kThreads - 1) / kThreads;
    const int g = (int)std::min<int64_t>(std::max<int64_t>(work, 1), (int64_t)num_sms() * 8);
    if (inverse_rht) k_dequant<true><<<g, kThreads, 0, s>>>(codes, scales, ts, rows, k, grid, rht_seed, out, ld_out);
    else k_dequant<false><<<g, kThreads, 0, s>>>(codes, scales, ts, rows, k, grid, rht_seed, out, ld_out);
    return cudaGetLastError();
}

cudaError_t launch_stats(const QuantLaunch &q, void *ws, int *n_ctas, cudaStream_t s) {
    Args a = make_args(q, ws);
    a.stats_out = reinterpret_cast<double *>(static_cast<char *>(ws) + kWsStats);
    const bool col = q.colwise != 0;
    int64_t work;
    if (!col) work = (a.out_rows * (a.k / 8) + kThreads - 1) / kThreads;
    else work = ((a.cols + 127) / 128) * ((a.rows + 127) / 128);
    const int g = (int)std::min<int64_t>(std::max<int64_t>(work, 1),
                                         std::min<int64_t>((int64_t)num_sms() * 4, kMaxStatsCtas));
    *n_ctas = g;
    const bool bf = q.dtype == 0;
#define UFP4_S(COLW, BF, RHT)                                                              \
    if (col == COLW && bf == BF && (q.rht != 0) == RHT) {                                  \
        if (COLW) k_stats_colwise<std::conditional_t<BF, __nv_bfloat16, float>, RHT>       \
            <<<g, kThreads, 0, s>>>(a, q.grid);                                            \
        else k_stats_rowwise<std::conditional_t<BF, __nv_bfloat16, float>, RHT>            \
            <<<g, kThreads, 0, s>>>(a, q.grid);                                            \
        return cudaGetLastError();                                                         \
    }
    UFP4_S(false, true, false) UFP4_S(false, true, true) UFP4_S(false, false, false)
    UFP4_S(false, false, true) UFP4_S(true, true, false) UFP4_S(true, true, true)
    UFP4_S(true, false, false) UFP4_S(true, false, true)
#undef UFP4_S
    return cudaErrorInvalidValue;
}

}  // namespace ufp4
