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
#include "ptx.cuh"

#include <cuda.h>

#include <algorithm>
#include <cfloat>
#include <mutex>
#include <type_traits>
#include <vector>

namespace ufp4 {

// Raised by a bounded wait of the staged quantization kernels that gave up.
__device__ uint32_t g_quant_timeout;

namespace {

constexpr int kThreads = 256;

struct Args {
    const void *x;
    int64_t rows, cols, ld;     // input as stored
    int64_t out_rows, k, kpad;  // result: out_rows x k, padded to kpad
    int64_t nkt;                // kpad / 64
    uint64_t rht_seed, sr_seed, sr_counter, elem_base;
    // Philox4x32-10 round keys of sr_seed (round r: srk[2r], srk[2r + 1]),
    // set by set_sr_keys on the host, so that a round reads its key from the
    // kernel's parameters instead of advancing it
    uint32_t srk[20];
    const float *amax_in;
    const float *partials;
    float *partials_out;
    int n_partials;
    uint32_t *status;
    uint8_t *codes, *scales;
    uint8_t *eplane;            // E1M2 correction plane beside the codes, or null
    float *tensor_scale;
    double *stats_out;
    // uniform grids (E1M2 kernels): qmax and the largest magnitude index,
    // 3.5 / 7 for E1M2, 2 / 4 for clamped E2M1
    float uqmax;
    uint32_t utop;
};

// A test-only build (-DUFP4_PROBE, tests/probe) records the values each
// quantization path hands to its block scale -- the rotated y when the
// transform is on -- so that tests can compare them element by element; in
// the library these hooks are empty.
#ifdef UFP4_PROBE
#include "probe_hooks.inc"
#else
#define UFP4_PROBE_ROW8(a, r, b, lo, hi, rht) ((void)0)
#define UFP4_PROBE_ROW16(a, r, b, v, rht) ((void)0)
#define UFP4_PROBE_COL16(a, c, kb, v, rht) ((void)0)
#endif

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
                                                      float *s_k, float *s_red, float &S_enc,
                                                      bool e1m2_fold = false, bool *folded = nullptr,
                                                      float *amax_out = nullptr) {
    float m = 0.0f;
    if (a.amax_in) {
        m = *a.amax_in;
    } else {
        for (int i = threadIdx.x; i < a.n_partials; i += blockDim.x) m = max_nan(m, __ldcg(a.partials + i));
#pragma unroll
        for (int o = 16; o; o >>= 1) m = max_nan(m, __shfl_xor_sync(0xffffffffu, m, o));
        if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = m;
        __syncthreads();
        m = s_red[0];
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w) m = max_nan(m, s_red[w]);
    }
    const float A_t = m;
    if (amax_out) *amax_out = A_t;
    float se = 1.0f, sd = 1.0f;
    if (A_t > 0.0f) {
        const float num = 448.0f * qmax;
        se = __fdiv_rn(num, A_t);
        if (se > kFltMax) se = kFltMax;
        sd = __fdiv_rn(A_t, num);
    }
    S_enc = se;
    // E1M2 codes come from x = q * 2^-8 (see e1m2x8); folding 2^-8 into the
    // table is exact while every k = S_enc / e >= S_enc / 448 stays >= 2^-118,
    // i.e. S_enc >= 2^-109 (A_t below ~1e36).
    const bool fold = e1m2_fold && se >= 1.5407439555097887e-33f;
    if (folded) *folded = fold;
    if (fold) kfold *= 0.00390625f;
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

// Block scale code of a block whose magnitude maximum is amax:
// E4M3(fl32(fl32(amax / qmax) * S_enc)).  The division uses Markstein's
// correction of the reciprocal product (P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990): q = RN(a * RN(1/b)), r = RN(a - b q) (exact with FMA),
// RN(q + r RN(1/b)) -- the correctly rounded quotient.  An exhaustive GPU
// comparison over every finite fp32 a showed it equal to IEEE division for
// b = 6 and b = 3.5 whenever a >= 2^-123; below that (results near the
// subnormal range) the IEEE division is used.
__device__ __forceinline__ float div_qmax(float a, float qmax) {
    if (qmax == 2.0f) return a * 0.5f;                        // exact
    if (!(a >= 9.4039548e-38f)) return __fdiv_rn(a, qmax);   // 2^-123, NaN, 0
    const float rcp = qmax == 6.0f ? 0.16666667163372040f : 0.28571429848670960f;
    const float q = __fmul_rn(a, rcp);
    const float r = __fmaf_rn(-qmax, q, a);
    return __fmaf_rn(r, rcp, q);
}

__device__ __forceinline__ uint32_t block_scale(float amax, float qmax, float S_enc) {
    return e4m3_from_f32(__fmul_rn(div_qmax(amax, qmax), S_enc));
}

// k = min(S_enc / E4M3(e), FLT_MAX) (x 1/4 for RHT), the per-code multiplier
// of the table, computed in place (grouped tensors: one S_enc per segment).
__device__ __forceinline__ float inline_k(uint32_t e, float S_enc, bool rht) {
    const float d = e4m3_to_f32(e);
    float kk = 0.0f;
    if (d > 0.0f) {
        kk = __fdiv_rn(S_enc, d);
        if (kk > kFltMax) kk = kFltMax;
    } else if (!(d == 0.0f)) {
        kk = d;
    }
    return rht ? kk * 0.25f : kk;
}

// Packed fp32 pairs (f32x2): two values per register pair and instruction.
__device__ __forceinline__ uint64_t pk2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void upk2(uint64_t r, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
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
            for (int j = 0; j < 8; ++j) w |= e1m2_rn(q[j], (float)a.utop) << (4 * j);
        }
    } else {
        // one Philox4x32-10 call per 8 codes: code j takes half (j % 2) of
        // word j / 2 (i0 is a multiple of 8, so the call's counter is i0 / 8)
        const uint64_t c = i0 >> 3;
        const uint4 r = philox4x32_10_keys(
            make_uint4((uint32_t)c, (uint32_t)(c >> 32), (uint32_t)a.sr_counter, (uint32_t)(a.sr_counter >> 32)),
            a.srk);
        const uint32_t rr[4] = {r.x, r.y, r.z, r.w};
        float qs[8];
        if (GRID == kE1M2) {
            // the decision's 2^17 scaling, two values per packed multiply
            const uint64_t S17 = pk2(131072.0f, 131072.0f);
#pragma unroll
            for (int j = 0; j < 8; j += 2) upk2(mul2(pk2(q[j], q[j + 1]), S17), qs[j], qs[j + 1]);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t h = (j & 1) ? rr[j >> 1] >> 16 : rr[j >> 1] & 0xFFFFu;
            const uint32_t code = GRID == kE1M2 ? sr_code_e1m2_scaled(qs[j], h, a.utop)
                                                : sr_code<GRID>(q[j], h, a.utop);
            w |= code << (4 * j);
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
// One thread owns one 16-block: a single 32-byte load (BF16) per block, so a
// warp's load covers 1 KB of contiguous row.  The 16 values are held as 8
// packed pairs P_j = (v_j, v_{j+8}); the butterflies on index bits 0..2 act
// on both halves at once with add/sub.rn.f32x2, the bit-3 stage pairs the
// halves.  Blocks are enumerated row-major over (row, block-in-row) with a
// fast 32-bit divider; each thread keeps two blocks in flight.

// max(a, b, c) in one instruction (PTX three-input max; NaN as fmaxf).
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// RHT sign flips, precomputed once per thread as XOR masks on the loaded
// words: row-wise BF16 word i holds elements (2i, 2i+1) -> bits 15 / 31;
// row-wise FP32 word e -> bit 31; column-wise BF16 row i holds two columns
// -> 0x80008000; column-wise FP32 row i -> bit 31 of both words.
struct Signs {
    uint32_t m[16];
};
template <class In> __device__ __forceinline__ Signs row_signs(uint32_t smask);
template <> __device__ __forceinline__ Signs row_signs<__nv_bfloat16>(uint32_t smask) {
    // word i holds elements 2i (low half) and 2i + 1 (high half): m[i] is the
    // fp32 sign bit of element 2i, m[8 + i] that of element 2i + 1
    Signs s;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        s.m[i] = ((smask >> (2 * i)) & 1u) << 31;
        s.m[8 + i] = ((smask >> (2 * i + 1)) & 1u) << 31;
    }
    return s;
}
template <> __device__ __forceinline__ Signs row_signs<float>(uint32_t smask) {
    Signs s;
#pragma unroll
    for (int i = 0; i < 16; ++i) s.m[i] = ((smask >> i) & 1u) << 31;
    return s;
}
template <class In> __device__ __forceinline__ Signs col_signs(uint32_t smask);
template <> __device__ __forceinline__ Signs col_signs<__nv_bfloat16>(uint32_t smask) {
    // row i of a column unit: both columns take the fp32 sign bit m[i]
    Signs s;
#pragma unroll
    for (int i = 0; i < 16; ++i) s.m[i] = ((smask >> i) & 1u) << 31;
    return s;
}
template <> __device__ __forceinline__ Signs col_signs<float>(uint32_t smask) {
    Signs s;
#pragma unroll
    for (int i = 0; i < 16; ++i) s.m[i] = ((smask >> i) & 1u) << 31;
    return s;
}

// BF16 halves of a 32-bit word as fp32 bit patterns, with the fp32 sign bit
// `sb` (0 or 1 << 31) flipped in: the low half as w * 2^16 + sb (one
// multiply-add: the product's low 16 bits are zero, so adding bit 31 flips
// it), the high half as (w & 0xFFFF0000) ^ sb (one three-input logic op).
__device__ __forceinline__ uint32_t bf16lo_s(uint32_t w, uint32_t sb) {
    uint32_t r;
    asm("mad.lo.u32 %0, %1, 65536, %2;" : "=r"(r) : "r"(w), "r"(sb));
    return r;
}
__device__ __forceinline__ uint32_t bf16hi_s(uint32_t w, uint32_t sb) { return (w & 0xFFFF0000u) ^ sb; }

// Raw 16 elements of one block.
template <class In> struct Raw;
template <> struct Raw<__nv_bfloat16> {
    uint32_t w[8];
    // 16-byte loads: a row of a strided input is only 16-byte aligned
    __device__ __forceinline__ void load(const __nv_bfloat16 *p) {
        asm volatile("ld.global.nc.v4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "l"(p));
        asm volatile("ld.global.nc.v4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7]) : "l"(p + 8));
    }
    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = 0u;
    }
    __device__ __forceinline__ void load_shared(uint32_t sa) {
        asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "r"(sa));
        asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7]) : "r"(sa + 16));
    }
    // element e as fp32, with the row-wise sign applied
    __device__ __forceinline__ float get(int e, const Signs &sg) const {
        return __uint_as_float((e & 1) ? bf16hi_s(w[e >> 1], sg.m[8 + (e >> 1)]) : bf16lo_s(w[e >> 1], sg.m[e >> 1]));
    }
    __device__ __forceinline__ float get(int e) const {
        const uint32_t u = w[e >> 1];
        return __uint_as_float((e & 1) ? (u & 0xFFFF0000u) : (u << 16));
    }
};
template <> struct Raw<float> {
    uint32_t w[16];
    // 16-byte loads: a row of a strided input is only 16-byte aligned
    __device__ __forceinline__ void load(const float *p) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
            asm volatile("ld.global.nc.v4.b32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(w[4 * q]), "=r"(w[4 * q + 1]), "=r"(w[4 * q + 2]), "=r"(w[4 * q + 3])
                         : "l"(p + 4 * q));
    }
    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = 0u;
    }
    __device__ __forceinline__ void load_shared(uint32_t sa) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
            asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(w[4 * q]), "=r"(w[4 * q + 1]), "=r"(w[4 * q + 2]), "=r"(w[4 * q + 3])
                         : "r"(sa + 16 * q));
    }
    __device__ __forceinline__ float get(int e, const Signs &sg) const { return __uint_as_float(w[e] ^ sg.m[e]); }
    __device__ __forceinline__ float get(int e) const { return __uint_as_float(w[e]); }
};

template <class In>
__device__ __forceinline__ void block_values_rht(const Raw<In> &raw, const Signs &sg, float lo[8], float hi[8]) {
    uint64_t P[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) P[j] = pk2(raw.get(j, sg), raw.get(j + 8, sg));
#pragma unroll
    for (int s = 1; s < 8; s <<= 1) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if ((j & s) == 0) {
                const uint64_t a = P[j], b = P[j + s];
                P[j] = add2(a, b);
                P[j + s] = sub2(a, b);
            }
        }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float a, b;
        upk2(P[j], a, b);
        lo[j] = a + b;
        hi[j] = a - b;
    }
}

// Values of one block after the optional transform: lo[j] = v_j, hi[j] =
// v_{j+8}; with RHT they are 4 y (H16 diag(d) x, unnormalised).
template <class In, bool RHT>
__device__ __forceinline__ void block_values(const Raw<In> &raw, const Signs &sg, float lo[8], float hi[8]) {
    if (!RHT) {
#pragma unroll
        for (int j = 0; j < 8; ++j) { lo[j] = raw.get(j); hi[j] = raw.get(j + 8); }
    } else {
        block_values_rht(raw, sg, lo, hi);
    }
}

struct FastDiv {
    uint32_t m, s;
};
FastDiv make_fastdiv(uint32_t d) {
    uint32_t s = 0;
    while ((1ull << s) < d) ++s;
    const uint64_t m = ((1ull << 32) * ((1ull << s) - d)) / d + 1;
    return FastDiv{(uint32_t)m, s};
}
__device__ __forceinline__ uint32_t fdiv(uint32_t n, FastDiv f) {
    return (uint32_t)(((uint64_t)__umulhi(n, f.m) + n) >> f.s);
}

// E2M1 RTNE of 8 values, element j in bits 4j..4j+3 (satfinite clamps at 6).
__device__ __forceinline__ uint32_t e2m1x8(const float v[8]) {
    uint32_t w;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(w)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return w;
}

// E1M2 RTNE of 8 values x = q * 2^-8 (q in grid units), already clamped to
// |x| <= 7 * 2^-9.  On [0, 15 * 2^-9] E4M3 is a uniform grid of step 2^-9
// (subnormals, then the first normal binade), so the saturating E4M3 RNE of
// x is sign << 7 | m with m = rint(2|q|), ties to even: exactly the E1M2 code.
// The bytes are regrouped as sign << 3 | m nibbles, element j at bits 4j.
__device__ __forceinline__ uint32_t e1m2x8(const float x[8]) {
    uint32_t ev, od;
    asm("{\n\t.reg .b16 h0, h1, h2, h3;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 h0, %3, %2;\n\t"    // bytes (x0, x2)
        "cvt.rn.satfinite.e4m3x2.f32 h1, %5, %4;\n\t"    // bytes (x4, x6)
        "cvt.rn.satfinite.e4m3x2.f32 h2, %7, %6;\n\t"    // bytes (x1, x3)
        "cvt.rn.satfinite.e4m3x2.f32 h3, %9, %8;\n\t"    // bytes (x5, x7)
        "mov.b32 %0, {h0, h1};\n\t"
        "mov.b32 %1, {h2, h3};\n\t}"
        : "=r"(ev), "=r"(od)
        : "f"(x[0]), "f"(x[2]), "f"(x[4]), "f"(x[6]), "f"(x[1]), "f"(x[3]), "f"(x[5]), "f"(x[7]));
    // ev bytes: x0, x2, x4, x6 ; od bytes: x1, x3, x5, x7
    const uint32_t ne = (ev | (ev >> 4)) & 0x0F0F0F0Fu;
    const uint32_t no = (od | (od >> 4)) & 0x0F0F0F0Fu;
    return ne | (no << 4);
}

// Two blocks per thread per step, software-pipelined: the loads of step i+1
// are issued before the arithmetic of step i, so every thread always has
// 64 bytes (BF16) in flight.
template <class In>
struct RowFetch {
    Raw<In> raw[2];
    uint32_t r[2], b[2];
    bool ok[2];
    __device__ __forceinline__ void fetch(const In *x, int64_t ld, uint32_t u0, uint32_t T, uint32_t total,
                                          FastDiv bdiv, uint32_t bpr, uint32_t kvb) {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const uint32_t u = u0 + t * T;
            ok[t] = u < total;
            r[t] = fdiv(u, bdiv);
            b[t] = u - r[t] * bpr;
            if (ok[t] && b[t] < kvb) raw[t].load(x + (int64_t)r[t] * ld + b[t] * 16);
            else raw[t].zero();
        }
    }
};

template <class In, bool RHT>
__global__ void __launch_bounds__(kThreads) k_amax_rowwise(Args a, FastDiv bdiv, uint32_t bpr,
                                                           uint32_t total) {
    __shared__ float s_red[kThreads / 32];
    const uint32_t smask = RHT ? rht_sign_mask(a.rht_seed) : 0u;
    const Signs sg = row_signs<In>(smask);
    const uint32_t T = gridDim.x * blockDim.x;
    const In *x = static_cast<const In *>(a.x);
    float m = 0.0f;
    uint32_t u0 = blockIdx.x * blockDim.x + threadIdx.x;
    RowFetch<In> cur;
    cur.fetch(x, a.ld, u0, T, total, bdiv, bpr, bpr);
    for (; u0 < total; u0 += 2 * T) {
        RowFetch<In> nxt;
        nxt.fetch(x, a.ld, u0 + 2 * T, T, total, bdiv, bpr, bpr);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            float lo[8], hi[8];
            block_values<In, RHT>(cur.raw[t], sg, lo, hi);
#pragma unroll
            for (int j = 0; j < 8; ++j) m = max3_nan(m, fabsf(lo[j]), fabsf(hi[j]));
        }
        cur = nxt;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) m = max_nan(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kThreads / 32; ++w) m = max_nan(m, s_red[w]);
        a.partials_out[blockIdx.x] = RHT ? m * 0.25f : m;
    }
}

__device__ __forceinline__ uint32_t scale_offset32(uint32_t r, uint32_t b, uint32_t nkt) {
    return (((r >> 7) * nkt + (b >> 2)) << 9) + ((r & 31) << 4) + (((r >> 5) & 3) << 2) + (b & 3);
}

// Rounding of one block's 16 values q (grid units, already multiplied by
// the table's k) into two 32-bit words of nibbles.  `folded`: for E1M2 the
// table already holds k * 2^-8.  `e` is the block's scale code: when the E4M3
// rounding of the scale was an ordinary round-to-nearest of a normal value
// (8 <= e < 0x7E) it moved the scale by at most 1/16 relative, so
// |q| <= qmax * 16/15 < 3.75 and the E4M3 step of e1m2x8 cannot carry past
// m = 7; subnormal scales (e < 8) and saturated ones (e = 448, e.g. a caller
// amax below the true maximum) take the explicit clamp.
template <int GRID, int ROUND>
__device__ __forceinline__ uint2 round_block(float ql[8], float qh[8], uint32_t e, bool folded, const Args &a,
                                             uint64_t i0) {
    if (ROUND == kRTNE && GRID == kE2M1) return make_uint2(e2m1x8(ql), e2m1x8(qh));
    if (ROUND == kRTNE) {
        if (!folded) {
            const uint64_t S8 = pk2(0.00390625f, 0.00390625f);
#pragma unroll
            for (int j = 0; j < 8; ++j) upk2(mul2(pk2(ql[j], qh[j]), S8), ql[j], qh[j]);
        }
        if (e < 8u || e >= 0x7Eu) {
            const float c = (float)a.utop * 0.001953125f;   // top index * 2^-9
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                ql[j] = fminf(fmaxf(ql[j], -c), c);
                qh[j] = fminf(fmaxf(qh[j], -c), c);
            }
        }
        return make_uint2(e1m2x8(ql), e1m2x8(qh));
    }
    return make_uint2(codes8<GRID, ROUND>(ql, a, i0), codes8<GRID, ROUND>(qh, a, i0 + 8));
}

// Packed codes at byte offset `off` of the code buffer, and their E1M2
// correction plane at the same offset of the plane when the tensor has one.
__device__ __forceinline__ void put_codes(const Args &a, size_t off, uint2 w) {
    *reinterpret_cast<uint2 *>(a.codes + off) = w;
    if (a.eplane) *reinterpret_cast<uint2 *>(a.eplane + off) = make_uint2(e1m2_eplane(w.x), e1m2_eplane(w.y));
}
__device__ __forceinline__ void put_codes(const Args &a, size_t off, uint4 w) {
    *reinterpret_cast<uint4 *>(a.codes + off) = w;
    if (a.eplane)
        *reinterpret_cast<uint4 *>(a.eplane + off) =
            make_uint4(e1m2_eplane(w.x), e1m2_eplane(w.y), e1m2_eplane(w.z), e1m2_eplane(w.w));
}

__device__ __forceinline__ void store_block(const Args &a, uint32_t r, uint32_t b, uint2 w, uint32_t e,
                                            uint32_t cstride, uint32_t nkt) {
    if (e == 0) w = make_uint2(0u, 0u);
    put_codes(a, (size_t)r * cstride + b * 8, w);
    a.scales[scale_offset32(r, b, nkt)] = (uint8_t)e;
}

// Quantize one row-wise 16-block (row r, block b) from its raw elements.
template <class In, int GRID, int ROUND, bool RHT>
__device__ __forceinline__ void quant_block_row(const Args &a, const Raw<In> &raw, uint32_t r, uint32_t b,
                                                const Signs &sg, float S_enc, const float *s_k,
                                                uint32_t cstride, uint32_t nkt, bool folded) {
    const float qmax = GRID == kE2M1 ? 6.0f : a.uqmax;
    float lo[8], hi[8];
    block_values<In, RHT>(raw, sg, lo, hi);
    UFP4_PROBE_ROW8(a, r, b, lo, hi, RHT);
    float m = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) m = max3f(m, fabsf(lo[j]), fabsf(hi[j]));
    if (RHT) m *= 0.25f;
    const uint32_t e = block_scale(m, qmax, S_enc);
    const float kk = s_k ? s_k[e] : inline_k(e, S_enc, RHT);
    const uint64_t K2 = pk2(kk, kk);
    float ql[8], qh[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) upk2(mul2(pk2(lo[j], hi[j]), K2), ql[j], qh[j]);
    const uint64_t i0 = a.elem_base + (uint64_t)r * (uint64_t)a.k + (uint64_t)b * 16u;
    store_block(a, r, b, round_block<GRID, ROUND>(ql, qh, e, folded, a, i0), e, cstride, nkt);
}

// Per element: deq = fl32(fl32(v e) S_dec), A = y (rotated input);
// sums of deq*A, A*A, (A-deq)^2, (v - a) over a != 0, count.
// Each thread keeps the five sums in fp32 with Kahan's compensation (W. Kahan,
// "Further remarks on reducing truncation errors", CACM 8(1), 1965): the
// error stays at a few fp32 ulps of the sum however many blocks a thread
// adds, and the GB300's fp64 rate (a small fraction of fp32) is spent only
// on the final cross-thread reduction.
struct Acc {
    float s[5] = {0, 0, 0, 0, 0};   // <deq, A>, <A, A>, ||A - deq||^2, bias sum, bias count
    float c[5] = {0, 0, 0, 0, 0};   // compensations (the negated lost low parts)
};
__device__ __forceinline__ void kahan_add(float &s, float &c, float x) {
    const float y = __fsub_rn(x, c);
    const float t = __fadd_rn(s, y);
    c = __fsub_rn(__fsub_rn(t, s), y);
    s = t;
}

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
    kahan_add(acc.s[0], acc.c[0], aq);
    kahan_add(acc.s[1], acc.c[1], aa);
    kahan_add(acc.s[2], acc.c[2], e2);
    kahan_add(acc.s[3], acc.c[3], bias);
    kahan_add(acc.s[4], acc.c[4], cnt);
}

__device__ void stats_reduce(Acc acc, double *out) {
    __shared__ double s[kThreads / 32][5];
    double v[5];
#pragma unroll
    for (int i = 0; i < 5; ++i) v[i] = (double)acc.s[i] - (double)acc.c[i];
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

// quant_block_row, and the block's terms of the quality statistics (the
// sums of ufp4_stats over the result actually stored) added to acc.
template <class In, int GRID, int ROUND, bool RHT>
__device__ __forceinline__ void quant_block_row_stats(const Args &a, const Raw<In> &raw, uint32_t r, uint32_t b,
                                                      const Signs &sg, float S_enc, float S_dec, const float *s_k,
                                                      uint32_t cstride, uint32_t nkt, bool folded, Acc &acc) {
    const float qmax = GRID == kE2M1 ? 6.0f : a.uqmax;
    float lo[8], hi[8];
    block_values<In, RHT>(raw, sg, lo, hi);
    float m = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) m = max3f(m, fabsf(lo[j]), fabsf(hi[j]));
    if (RHT) m *= 0.25f;
    const uint32_t e = block_scale(m, qmax, S_enc);
    const float kk = s_k ? s_k[e] : inline_k(e, S_enc, RHT);
    const uint64_t K2 = pk2(kk, kk);
    float ql[8], qh[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) upk2(mul2(pk2(lo[j], hi[j]), K2), ql[j], qh[j]);
    const uint64_t i0 = a.elem_base + (uint64_t)r * (uint64_t)a.k + (uint64_t)b * 16u;
    uint2 w = round_block<GRID, ROUND>(ql, qh, e, folded, a, i0);
    if (e == 0) w = make_uint2(0u, 0u);
    store_block(a, r, b, w, e, cstride, nkt);
    if (RHT) {
#pragma unroll
        for (int j = 0; j < 8; ++j) { lo[j] *= 0.25f; hi[j] *= 0.25f; }
    }
    const float ev = e4m3_to_f32(e);
    acc_block8(acc, lo, w.x, ev, S_dec, GRID, qmax);
    acc_block8(acc, hi, w.y, ev, S_dec, GRID, qmax);
}

// Two row-wise blocks (A, B) held as packed pairs P_j = (A_j, B_j), so all
// four butterfly stages and the scaling run on f32x2.
template <int GRID, int ROUND, bool RHT>
__device__ __forceinline__ void quant_pair_row(const Args &a, const Raw<__nv_bfloat16> &ra,
                                               const Raw<__nv_bfloat16> &rb, uint32_t r0, uint32_t b0,
                                               uint32_t r1, uint32_t b1, bool has_b, const Signs &sg,
                                               float S_enc, const float *s_k, uint32_t cstride,
                                               uint32_t nkt, bool folded) {
    const float qmax = GRID == kE2M1 ? 6.0f : a.uqmax;
    uint64_t P[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) P[j] = RHT ? pk2(ra.get(j, sg), rb.get(j, sg)) : pk2(ra.get(j), rb.get(j));
    if (RHT) {
#pragma unroll
        for (int st = 1; st < 16; st <<= 1) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                if ((j & st) == 0) {
                    const uint64_t x = P[j], y = P[j + st];
                    P[j] = add2(x, y);
                    P[j + st] = sub2(x, y);
                }
            }
        }
    }
    float va[16], vb[16];
    float ma = 0.0f, mb = 0.0f;
#pragma unroll
    for (int j = 0; j < 16; ++j) upk2(P[j], va[j], vb[j]);
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
        ma = max3f(ma, fabsf(va[j]), fabsf(va[j + 1]));
        mb = max3f(mb, fabsf(vb[j]), fabsf(vb[j + 1]));
    }
    UFP4_PROBE_ROW16(a, r0, b0, va, RHT);
    if (has_b) UFP4_PROBE_ROW16(a, r1, b1, vb, RHT);
    if (RHT) { ma *= 0.25f; mb *= 0.25f; }
    const uint32_t ea = block_scale(ma, qmax, S_enc), eb = block_scale(mb, qmax, S_enc);
    const uint64_t K2 = pk2(s_k[ea], s_k[eb]);
#pragma unroll
    for (int j = 0; j < 16; ++j) upk2(mul2(P[j], K2), va[j], vb[j]);
    const uint64_t ia = a.elem_base + (uint64_t)r0 * (uint64_t)a.k + (uint64_t)b0 * 16u;
    const uint64_t ib = a.elem_base + (uint64_t)r1 * (uint64_t)a.k + (uint64_t)b1 * 16u;
    store_block(a, r0, b0, round_block<GRID, ROUND>(va, va + 8, ea, folded, a, ia), ea, cstride, nkt);
    if (has_b) store_block(a, r1, b1, round_block<GRID, ROUND>(vb, vb + 8, eb, folded, a, ib), eb, cstride, nkt);
}

template <class In, int GRID, int ROUND, bool RHT>
__global__ void __launch_bounds__(kThreads) k_quant_rowwise(Args a, FastDiv bdiv, uint32_t bpr,
                                                            uint32_t total) {
    __shared__ float s_k[256];
    __shared__ float s_red[kThreads / 32];
    const float qmax = GRID == kE2M1 ? 6.0f : a.uqmax;
    float S_enc;
    bool folded = false;
    tensor_scale_prologue(a, qmax, RHT ? 0.25f : 1.0f, s_k, s_red, S_enc, GRID == kE1M2 && ROUND == kRTNE,
                          &folded);

    const uint32_t smask = RHT ? rht_sign_mask(a.rht_seed) : 0u;
    const Signs sg = row_signs<In>(smask);
    const uint32_t T = gridDim.x * blockDim.x;
    const uint32_t kvb = (uint32_t)(a.k / 16);      // real blocks per row
    const uint32_t nkt = (uint32_t)a.nkt;
    const In *x = static_cast<const In *>(a.x);
    const uint32_t cstride = (uint32_t)(a.kpad / 2);
    uint32_t u0 = blockIdx.x * blockDim.x + threadIdx.x;
    RowFetch<In> cur;
    cur.fetch(x, a.ld, u0, T, total, bdiv, bpr, kvb);
    for (; u0 < total; u0 += 2 * T) {
        RowFetch<In> nxt;
        nxt.fetch(x, a.ld, u0 + 2 * T, T, total, bdiv, bpr, kvb);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            if (!cur.ok[t]) continue;
            quant_block_row<In, GRID, ROUND, RHT>(a, cur.raw[t], cur.r[t], cur.b[t], sg, S_enc, s_k,
                                                  cstride, nkt, folded);
        }
        cur = nxt;
    }
    zero_pad_rows(a);
}

// Grid of exactly the CTAs that fit on the device at once (persistent).
template <class K>
int resident_grid(K kernel, int64_t work_ctas, size_t smem = 0) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    const int64_t g = std::min<int64_t>(std::max<int64_t>(work_ctas, 1), (int64_t)per_sm * num_sms());
    return (int)std::min<int64_t>(g, kMaxPartials);
}

// ==================================================== column-wise kernels
// The quantization of X^T: 16-blocks run down the columns.  A thread owns a
// unit of 16 rows x 2 adjacent columns (two blocks, one per column); a warp's
// 32 units are 64 adjacent columns, so each row load of the warp reads 128
// contiguous bytes (BF16).  The two columns are held as packed pairs
// P_i = (col0[i], col1[i]), so all four butterfly stages run on f32x2.
// Units are enumerated (row-block, column-pair) with the column pair fastest;
// the next unit's 16 loads are issued before the current unit's arithmetic.
template <class In> struct ColRaw;
template <> struct ColRaw<__nv_bfloat16> {
    uint32_t w[16];   // row i: (col0, col1) as bf16 pair
    __device__ __forceinline__ void load(const __nv_bfloat16 *p, int64_t ld) {
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = __ldg(reinterpret_cast<const unsigned int *>(p + i * ld));
    }
    __device__ __forceinline__ void load_rows(const __nv_bfloat16 *p, int64_t ld, int nvalid) {
#pragma unroll
        for (int i = 0; i < 16; ++i)
            w[i] = i < nvalid ? __ldg(reinterpret_cast<const unsigned int *>(p + i * ld)) : 0u;
    }
    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = 0u;
    }
    __device__ __forceinline__ void load_shared(uint32_t sa, uint32_t pitch) {
#pragma unroll
        for (int i = 0; i < 16; ++i) asm volatile("ld.shared.b32 %0, [%1];" : "=r"(w[i]) : "r"(sa + i * pitch));
    }
    // rows nvalid..15 read as zeros (the rows of a tile past its segment's end)
    __device__ __forceinline__ void load_shared_rows(uint32_t sa, uint32_t pitch, int nvalid) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            w[i] = 0u;
            if (i < nvalid) asm volatile("ld.shared.b32 %0, [%1];" : "=r"(w[i]) : "r"(sa + i * pitch));
        }
    }
    __device__ __forceinline__ uint64_t pair(int i, const Signs &sg) const {
        return pk2(__uint_as_float(bf16lo_s(w[i], sg.m[i])), __uint_as_float(bf16hi_s(w[i], sg.m[i])));
    }
    __device__ __forceinline__ uint64_t pair(int i) const {
        const uint32_t u = w[i];
        return pk2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
    }
};
template <> struct ColRaw<float> {
    uint2 w[16];
    __device__ __forceinline__ void load(const float *p, int64_t ld) {
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = __ldg(reinterpret_cast<const uint2 *>(p + i * ld));
    }
    __device__ __forceinline__ void load_rows(const float *p, int64_t ld, int nvalid) {
#pragma unroll
        for (int i = 0; i < 16; ++i)
            w[i] = i < nvalid ? __ldg(reinterpret_cast<const uint2 *>(p + i * ld)) : make_uint2(0u, 0u);
    }
    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = make_uint2(0u, 0u);
    }
    __device__ __forceinline__ void load_shared(uint32_t sa, uint32_t pitch) {
#pragma unroll
        for (int i = 0; i < 16; ++i)
            asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(w[i].x), "=r"(w[i].y) : "r"(sa + i * pitch));
    }
    __device__ __forceinline__ uint64_t pair(int i, const Signs &sg) const {
        return pk2(__uint_as_float(w[i].x ^ sg.m[i]), __uint_as_float(w[i].y ^ sg.m[i]));
    }
    __device__ __forceinline__ uint64_t pair(int i) const {
        return pk2(__uint_as_float(w[i].x), __uint_as_float(w[i].y));
    }
};

// Column values after the optional transform: P[i] = (c0[i], c1[i]); with
// RHT they are 4 y (unnormalised).
template <class In, bool RHT>
__device__ __forceinline__ void col_values(const ColRaw<In> &raw, const Signs &sg, uint64_t P[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) P[i] = RHT ? raw.pair(i, sg) : raw.pair(i);
    if (RHT) {
#pragma unroll
        for (int s = 1; s < 16; s <<= 1) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                if ((i & s) == 0) {
                    const uint64_t a = P[i], b = P[i + s];
                    P[i] = add2(a, b);
                    P[i + s] = sub2(a, b);
                }
            }
        }
    }
}

template <class In>
struct ColFetch {
    ColRaw<In> raw;
    uint32_t kb, cp;
    bool ok, real;
    __device__ __forceinline__ void fetch(const In *x, int64_t ld, uint32_t u, uint32_t total, FastDiv cdiv,
                                          uint32_t ncp, uint32_t nkb_real) {
        ok = u < total;
        kb = fdiv(u, cdiv);
        cp = u - kb * ncp;
        real = ok && kb < nkb_real;
        if (real) raw.load(x + (int64_t)kb * 16 * ld + cp * 2, ld);
        else raw.zero();
    }
};

template <class In, bool RHT>
__global__ void __launch_bounds__(kThreads) k_amax_colwise(Args a, FastDiv cdiv, uint32_t ncp,
                                                           uint32_t total) {
    __shared__ float s_red[kThreads / 32];
    const uint32_t smask = RHT ? rht_sign_mask(a.rht_seed) : 0u;
    const Signs sg = col_signs<In>(smask);
    const uint32_t T = gridDim.x * blockDim.x;
    const uint32_t nkb = (uint32_t)(a.rows / 16);
    const In *x = static_cast<const In *>(a.x);
    float m = 0.0f;
    uint32_t u = blockIdx.x * blockDim.x + threadIdx.x;
    ColFetch<In> cur;
    cur.fetch(x, a.ld, u, total, cdiv, ncp, nkb);
    for (; u < total; u += T) {
        ColFetch<In> nxt;
        nxt.fetch(x, a.ld, u + T, total, cdiv, ncp, nkb);
        uint64_t P[16];
        col_values<In, RHT>(cur.raw, sg, P);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float c0, c1;
            upk2(P[i], c0, c1);
            m = max3_nan(m, fabsf(c0), fabsf(c1));
        }
        cur = nxt;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) m = max_nan(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kThreads / 32; ++w) m = max_nan(m, s_red[w]);
        a.partials_out[blockIdx.x] = RHT ? m * 0.25f : m;
    }
}

// Quantize one column-wise unit: 16 rows x columns (c, c+1) starting at
// row-block kb (two output blocks: rows c and c+1 of the result, block kb).
// `real` = false for the padding blocks past the last row (zeros written).
template <class In, int GRID, int ROUND, bool RHT>
__device__ __forceinline__ void col_unit_words(const Args &a, const ColRaw<In> &raw, uint32_t kb, uint32_t c,
                                               bool real, const Signs &sg, float S_enc, const float *s_k,
                                               bool folded, uint2 &w0, uint2 &w1, uint32_t &e0_out,
                                               uint32_t &e1_out) {
    const float qmax = GRID == kE2M1 ? 6.0f : a.uqmax;
    uint64_t P[16];
    col_values<In, RHT>(raw, sg, P);
    float v0[16], v1[16];
    float m0 = 0.0f, m1 = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) upk2(P[i], v0[i], v1[i]);
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
        m0 = max3f(m0, fabsf(v0[i]), fabsf(v0[i + 1]));
        m1 = max3f(m1, fabsf(v1[i]), fabsf(v1[i + 1]));
    }
    if (real) {
        UFP4_PROBE_COL16(a, c, kb, v0, RHT);
        UFP4_PROBE_COL16(a, c + 1, kb, v1, RHT);
    }
    if (RHT) { m0 *= 0.25f; m1 *= 0.25f; }
    uint32_t e0 = block_scale(m0, qmax, S_enc), e1 = block_scale(m1, qmax, S_enc);
    if (!real) { e0 = 0u; e1 = 0u; }
    const uint64_t K2 = s_k ? pk2(s_k[e0], s_k[e1]) : pk2(inline_k(e0, S_enc, RHT), inline_k(e1, S_enc, RHT));
#pragma unroll
    for (int i = 0; i < 16; ++i) upk2(mul2(P[i], K2), v0[i], v1[i]);
    const uint64_t R = (uint64_t)a.rows;
    const uint64_t i0 = a.elem_base + (uint64_t)c * R + (uint64_t)kb * 16u;
    w0 = round_block<GRID, ROUND>(v0, v0 + 8, e0, folded, a, i0);
    w1 = round_block<GRID, ROUND>(v1, v1 + 8, e1, folded, a, i0 + R);
    if (e0 == 0) w0 = make_uint2(0u, 0u);
    if (e1 == 0) w1 = make_uint2(0u, 0u);
    e0_out = e0;
    e1_out = e1;
}

template <class In, int GRID, int ROUND, bool RHT>
__device__ __forceinline__ void quant_unit_col(const Args &a, const ColRaw<In> &raw, uint32_t kb, uint32_t c,
                                               bool real, const Signs &sg, float S_enc, const float *s_k,
                                               uint32_t cstride, uint32_t nkt, bool folded) {
    uint2 w0, w1;
    uint32_t e0, e1;
    col_unit_words<In, GRID, ROUND, RHT>(a, raw, kb, c, real, sg, S_enc, s_k, folded, w0, w1, e0, e1);
    store_block(a, c, kb, w0, e0, cstride, nkt);
    store_block(a, c + 1, kb, w1, e1, cstride, nkt);
}

template <class In, int GRID, int ROUND, bool RHT>
__global__ void __launch_bounds__(kThreads) k_quant_colwise(Args a, FastDiv cdiv, uint32_t ncp,
                                                            uint32_t total) {
    __shared__ float s_k[256];
    __shared__ float s_red[kThreads / 32];
    const float qmax = GRID == kE2M1 ? 6.0f : a.uqmax;
    float S_enc;
    bool folded = false;
    tensor_scale_prologue(a, qmax, RHT ? 0.25f : 1.0f, s_k, s_red, S_enc, GRID == kE1M2 && ROUND == kRTNE,
                          &folded);

    const uint32_t smask = RHT ? rht_sign_mask(a.rht_seed) : 0u;
    const Signs sg = col_signs<In>(smask);
    const uint32_t T = gridDim.x * blockDim.x;
    const uint32_t nkb = (uint32_t)(a.rows / 16);   // real blocks along k
    const uint32_t nkt = (uint32_t)a.nkt;
    const In *x = static_cast<const In *>(a.x);
    const uint32_t cstride = (uint32_t)(a.kpad / 2);
    uint32_t u = blockIdx.x * blockDim.x + threadIdx.x;
    ColFetch<In> cur;
    cur.fetch(x, a.ld, u, total, cdiv, ncp, nkb);
    for (; u < total; u += T) {
        ColFetch<In> nxt;
        nxt.fetch(x, a.ld, u + T, total, cdiv, ncp, nkb);
        if (cur.ok)
            quant_unit_col<In, GRID, ROUND, RHT>(a, cur.raw, cur.kb, cur.cp * 2, cur.real, sg, S_enc, s_k,
                                                 cstride, nkt, folded);
        cur = nxt;
    }
    zero_pad_rows(a);
}

// ================================================ TMA-staged (bulk copy) path
// For inputs whose bytes can be streamed in 16-byte-aligned pieces (row-wise:
// the whole tensor is contiguous; column-wise: every row segment of a chunk
// is a multiple of 16 bytes), one thread per CTA streams 16 KB chunks into a
// shared-memory ring with cp.async.bulk (mbarrier completion), so each CTA
// keeps its loads in flight independent of the register budget, and all 256
// threads compute from shared memory.  Quantization passes are issue-bound:
// a 3-deep ring (48 KB) and at least 3 resident CTAs per SM (registers <= 80;
// measured 17-25 % faster than 2 CTAs); the amax passes stream with little
// arithmetic and keep a 4-deep ring (64 KB in flight per CTA).
template <bool AMAX> constexpr int ring_depth() { return AMAX ? 4 : 3; }
constexpr int kStagedMinCtas = 3;
constexpr uint32_t kChunk = 16384;
template <bool AMAX> constexpr uint32_t ring_smem() { return ring_depth<AMAX>() * kChunk + 64; }
constexpr long long kRingWait = 4000000000LL;

struct RingCtl {
    uint32_t buf;    // shared address of stage 0
    uint32_t bars;   // shared address of the ring's mbarriers
    volatile int *abort;   // raised by a thread whose own wait gave up
};

template <int kRing>
__device__ __forceinline__ RingCtl ring_init(uint8_t *dsm) {
    static_assert(kRing * 8 + 4 <= 64, "the ring's barriers and abort flag fit its 64 bytes");
    RingCtl r;
    r.buf = ptx::smem_u32(dsm);
    r.bars = ptx::smem_u32(dsm + kRing * kChunk);
    r.abort = reinterpret_cast<volatile int *>(dsm + kRing * kChunk + 60);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kRing; ++s) ptx::mbar_init(r.bars + 8u * s, 1);
        *r.abort = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    return r;
}

// Each thread's own wait for chunk j's stage, without a CTA barrier: a thread
// that gives up raises the abort flag, which every thread reads after the
// barrier that ends the iteration.
template <int kRing>
__device__ __forceinline__ bool ring_wait_own(const RingCtl &r, uint32_t j) {
    const bool ok = ptx::mbar_wait_bounded(r.bars + 8u * (j % kRing), (j / kRing) & 1u, kRingWait);
    if (!ok) *r.abort = 1;
    return ok;
}

// Waits for chunk j's stage; false (for every thread) if any thread gave up.
template <int kRing>
__device__ __forceinline__ bool ring_wait(const RingCtl &r, uint32_t j) {
    const bool ok = ptx::mbar_wait_bounded(r.bars + 8u * (j % kRing), (j / kRing) & 1u, kRingWait);
    return __syncthreads_and(ok) != 0;
}

// After an early exit: the issuing thread waits (bounded) for every copy it
// started and that nobody consumed, so none lands in freed shared memory.
template <int kRing>
__device__ __forceinline__ void ring_drain(const RingCtl &r, uint32_t consumed, uint32_t issued) {
    if (threadIdx.x != 0) return;
    for (uint32_t j = consumed; j < issued; ++j)
        if (!ptx::mbar_wait_bounded(r.bars + 8u * (j % kRing), (j / kRing) & 1u, kRingWait)) break;
}

// Row-wise chunks: chunk i = bytes [i * kChunk, ...) of the contiguous input.
template <class In, int kRing>
__device__ __forceinline__ void row_issue(const RingCtl &r, const Args &a, uint32_t j, uint32_t nchunks,
                                          uint64_t total_bytes, uint32_t &issued) {
    const uint32_t i = blockIdx.x + j * gridDim.x;
    if (i >= nchunks) return;
    const uint64_t off = (uint64_t)i * kChunk;
    const uint64_t rem = total_bytes - off;
    const uint32_t bytes = rem < kChunk ? (uint32_t)rem : kChunk;
    const uint32_t bar = r.bars + 8u * (j % kRing);
    ptx::mbar_arrive_expect_tx(bar, bytes);
    ptx::bulk_load(r.buf + (j % kRing) * kChunk, static_cast<const uint8_t *>(a.x) + off, bytes, bar);
    issued = j + 1;
}

// STATS (quantization pass only): also accumulate the quality statistics of
// the result -- the sums of ufp4_stats -- and write one set of partial sums
// per CTA to a.stats_out, so that quantization and statistics take one read.
template <class In, int GRID, int ROUND, bool RHT, bool AMAX, bool STATS = false>
__global__ void __launch_bounds__(kThreads, kStagedMinCtas) k_row_staged(Args a, FastDiv bdiv, uint32_t kvb,
                                                         uint32_t nchunks, uint64_t total_bytes) {
    constexpr int kRing = ring_depth<AMAX>();
    extern __shared__ __align__(128) uint8_t dsm[];
    __shared__ float s_k[256];
    __shared__ float s_red[kThreads / 32];
    // start streaming before the tensor-scale prologue so its latency overlaps
    const RingCtl ring = ring_init<kRing>(dsm);
    uint32_t issued = 0, j = 0;
    if (threadIdx.x == 0)
        for (uint32_t t = 0; t < kRing; ++t) row_issue<In, kRing>(ring, a, t, nchunks, total_bytes, issued);
    float S_enc = 1.0f, S_dec = 1.0f;
    bool folded = false;
    if (!AMAX) {
        const float qmax = GRID == kE2M1 ? 6.0f : a.uqmax;
        float A_t = 0.0f;
        tensor_scale_prologue(a, qmax, RHT ? 0.25f : 1.0f, s_k, s_red, S_enc, GRID == kE1M2 && ROUND == kRTNE,
                              &folded, &A_t);
        if (STATS && A_t > 0.0f) S_dec = __fdiv_rn(A_t, 448.0f * qmax);   // as the prologue stores it
    }
    Acc acc;
    const uint32_t smask = RHT ? rht_sign_mask(a.rht_seed) : 0u;
    const Signs sg = row_signs<In>(smask);
    const uint32_t total_blocks = (uint32_t)(total_bytes / (16 * sizeof(In)));
    constexpr uint32_t BPC = kChunk / (16 * sizeof(In));
    const uint32_t nloc = nchunks > blockIdx.x ? (nchunks - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    const uint32_t cstride = (uint32_t)(a.kpad / 2), nkt = (uint32_t)a.nkt;
    float m = 0.0f;
    bool ok = true;
    for (; j < nloc; ++j) {
        if (!ring_wait<kRing>(ring, j)) { ok = false; break; }
        const uint32_t i = blockIdx.x + j * gridDim.x;
        const uint32_t st = ring.buf + (j % kRing) * kChunk;
        if (sizeof(In) == 2 && AMAX) {
            // BF16 maxima: 512 blocks per chunk, thread t owns blocks t and t + 256 as a packed pair
            // (quantization takes one block at a time below: measured 12 % faster with the
            // transform on a 512 MB operand than the packed pair, which holds twice the registers)
            const uint32_t k0 = threadIdx.x, k1 = threadIdx.x + kThreads;
            const uint32_t g0 = i * BPC + k0, g1 = i * BPC + k1;
            if (g0 < total_blocks) {
                const bool has1 = g1 < total_blocks;
                Raw<__nv_bfloat16> r0, r1;
                r0.load_shared(st + k0 * 32);
                if (has1) r1.load_shared(st + k1 * 32); else r1.zero();
                uint64_t P[16];
#pragma unroll
                for (int q = 0; q < 16; ++q) P[q] = RHT ? pk2(r0.get(q, sg), r1.get(q, sg)) : pk2(r0.get(q), r1.get(q));
                if (RHT) {
#pragma unroll
                    for (int sg = 1; sg < 16; sg <<= 1) {
#pragma unroll
                        for (int q = 0; q < 16; ++q) {
                            if ((q & sg) == 0) {
                                const uint64_t xx = P[q], yy = P[q + sg];
                                P[q] = add2(xx, yy);
                                P[q + sg] = sub2(xx, yy);
                            }
                        }
                    }
                }
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    float u0, u1;
                    upk2(P[q], u0, u1);
                    m = max3_nan(m, fabsf(u0), fabsf(u1));
                }
            }
        } else {
            // a thread's blocks of the chunk unrolled, so that their independent
            // arithmetic interleaves (2 % faster with the transform)
#pragma unroll
            for (uint32_t kk = 0; kk < (BPC + kThreads - 1) / kThreads; ++kk) {
                const uint32_t k = threadIdx.x + kk * kThreads;
                const uint32_t gb = i * BPC + k;
                if (k >= BPC || gb >= total_blocks) continue;
                Raw<In> raw;
                raw.load_shared(st + k * 16 * sizeof(In));
                if (AMAX) {
                    float lo[8], hi[8];
                    block_values<In, RHT>(raw, sg, lo, hi);
#pragma unroll
                    for (int q = 0; q < 8; ++q) m = max3_nan(m, fabsf(lo[q]), fabsf(hi[q]));
                } else {
                    const uint32_t r = fdiv(gb, bdiv);
                    if (STATS)
                        quant_block_row_stats<In, GRID, ROUND, RHT>(a, raw, r, gb - r * kvb, sg, S_enc, S_dec, s_k,
                                                                    cstride, nkt, folded, acc);
                    else
                        quant_block_row<In, GRID, ROUND, RHT>(a, raw, r, gb - r * kvb, sg, S_enc, s_k, cstride,
                                                              nkt, folded);
                }
            }
        }
        __syncthreads();
        if (threadIdx.x == 0) row_issue<In, kRing>(ring, a, j + kRing, nchunks, total_bytes, issued);
    }
    if (!ok) {
        if (threadIdx.x == 0) atomicOr(&g_quant_timeout, 1u);
        ring_drain<kRing>(ring, j, issued);
    }
    if (AMAX) {
#pragma unroll
        for (int o = 16; o; o >>= 1) m = max_nan(m, __shfl_xor_sync(0xffffffffu, m, o));
        if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = m;
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int w = 1; w < kThreads / 32; ++w) m = max_nan(m, s_red[w]);
            a.partials_out[blockIdx.x] = RHT ? m * 0.25f : m;
        }
    } else {
        // padding blocks k/16 .. kpad/16 - 1 of every row, and padding rows
        const uint32_t nbp = (uint32_t)(a.kpad / 16) - kvb;
        const uint32_t npad = (uint32_t)a.out_rows * nbp;
        for (uint32_t t = blockIdx.x * blockDim.x + threadIdx.x; t < npad; t += gridDim.x * blockDim.x) {
            const uint32_t r = t / nbp, b = kvb + (t - r * nbp);
            put_codes(a, (size_t)r * cstride + b * 8, make_uint2(0u, 0u));
            a.scales[scale_offset32(r, b, nkt)] = 0;
        }
        zero_pad_rows(a);
        if (STATS) stats_reduce(acc, a.stats_out);
    }
}

// Column-wise chunks: chunk i = (row block kb, column chunk cc) = 16 rows x
// CW columns, CW = kChunk / (16 * sizeof(In)); column chunk fastest.
template <class In, int kRing>
__device__ __forceinline__ void col_issue(const RingCtl &r, const Args &a, uint32_t j, uint32_t nchunks,
                                          uint32_t ncc, uint32_t &issued) {
    constexpr uint32_t CW = kChunk / (16 * sizeof(In));
    const uint32_t i = blockIdx.x + j * gridDim.x;
    if (i >= nchunks) return;
    const uint32_t kb = i / ncc, cc = i - kb * ncc;
    const uint32_t c0 = cc * CW;
    const int64_t left = a.cols - (int64_t)c0;
    const uint32_t ncols = left < (int64_t)CW ? (uint32_t)left : CW;
    const uint32_t rowbytes = ncols * sizeof(In);
    const uint32_t bar = r.bars + 8u * (j % kRing);
    const uint32_t st = r.buf + (j % kRing) * kChunk;
    ptx::mbar_arrive_expect_tx(bar, 16 * rowbytes);
    const In *src = static_cast<const In *>(a.x) + (int64_t)kb * 16 * a.ld + c0;
    for (int q = 0; q < 16; ++q)
        ptx::bulk_load(st + q * (CW * sizeof(In)), src + (int64_t)q * a.ld, rowbytes, bar);
    issued = j + 1;
}

template <class In, int GRID, int ROUND, bool RHT, bool AMAX>
__global__ void __launch_bounds__(kThreads, kStagedMinCtas) k_col_staged(Args a, uint32_t ncc, uint32_t nchunks) {
    constexpr int kRing = ring_depth<AMAX>();
    extern __shared__ __align__(128) uint8_t dsm[];
    __shared__ float s_k[256];
    __shared__ float s_red[kThreads / 32];
    constexpr uint32_t CW = kChunk / (16 * sizeof(In));
    const RingCtl ring = ring_init<kRing>(dsm);
    uint32_t issued = 0, j = 0;
    if (threadIdx.x == 0)
        for (uint32_t t = 0; t < kRing; ++t) col_issue<In, kRing>(ring, a, t, nchunks, ncc, issued);
    float S_enc = 1.0f;
    bool folded = false;
    if (!AMAX)
        tensor_scale_prologue(a, GRID == kE2M1 ? 6.0f : a.uqmax, RHT ? 0.25f : 1.0f, s_k, s_red, S_enc,
                              GRID == kE1M2 && ROUND == kRTNE, &folded);
    const uint32_t smask = RHT ? rht_sign_mask(a.rht_seed) : 0u;
    const Signs sg = col_signs<In>(smask);
    const uint32_t nloc = nchunks > blockIdx.x ? (nchunks - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    const uint32_t cstride = (uint32_t)(a.kpad / 2), nkt = (uint32_t)a.nkt;
    float m = 0.0f;
    bool ok = true;
    for (; j < nloc; ++j) {
        if (!ring_wait<kRing>(ring, j)) { ok = false; break; }
        const uint32_t i = blockIdx.x + j * gridDim.x;
        const uint32_t kb = i / ncc, cc = i - kb * ncc;
        const uint32_t c = cc * CW + 2 * threadIdx.x;
        if (2 * threadIdx.x < CW && c < (uint32_t)a.cols) {
            ColRaw<In> raw;
            raw.load_shared(ring.buf + (j % kRing) * kChunk + 2 * threadIdx.x * sizeof(In), CW * sizeof(In));
            if (AMAX) {
                uint64_t P[16];
                col_values<In, RHT>(raw, sg, P);
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    float c0, c1;
                    upk2(P[q], c0, c1);
                    m = max3_nan(m, fabsf(c0), fabsf(c1));
                }
            } else {
                quant_unit_col<In, GRID, ROUND, RHT>(a, raw, kb, c, true, sg, S_enc, s_k, cstride, nkt, folded);
            }
        }
        __syncthreads();
        if (threadIdx.x == 0) col_issue<In, kRing>(ring, a, j + kRing, nchunks, ncc, issued);
    }
    if (!ok) {
        if (threadIdx.x == 0) atomicOr(&g_quant_timeout, 1u);
        ring_drain<kRing>(ring, j, issued);
    }
    if (AMAX) {
#pragma unroll
        for (int o = 16; o; o >>= 1) m = max_nan(m, __shfl_xor_sync(0xffffffffu, m, o));
        if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = m;
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int w = 1; w < kThreads / 32; ++w) m = max_nan(m, s_red[w]);
            a.partials_out[blockIdx.x] = RHT ? m * 0.25f : m;
        }
    } else {
        // padding blocks past the last input row, for every output row
        const uint32_t kvb = (uint32_t)(a.rows / 16), nbp = (uint32_t)(a.kpad / 16) - kvb;
        const uint32_t npad = (uint32_t)a.out_rows * nbp;
        for (uint32_t t = blockIdx.x * blockDim.x + threadIdx.x; t < npad; t += gridDim.x * blockDim.x) {
            const uint32_t r = t / nbp, b = kvb + (t - r * nbp);
            put_codes(a, (size_t)r * cstride + b * 8, make_uint2(0u, 0u));
            a.scales[scale_offset32(r, b, nkt)] = 0;
        }
        zero_pad_rows(a);
    }
}

// ========================================= tensor-core amax (BF16, transform)
// With the transform on, the tensor amax is max |y| over y = (1/4) H16
// diag(d) x of every 16-block: a product with the constant 16 x 16 matrix
// H16 diag(d), whose entries +-1 are exact in BF16, and only the maximum is
// needed, not where each y lands.  So the blocks go through the tensor cores
// as the rows of A in mma.sync m16n8k16 BF16 products with fp32 accumulation
// (the products are exact; the tensor cores round the 16-term sums, within
// about 1e-7 relative of the fp64 transform), A loaded by ldmatrix from
// 16-row chunks staged in shared memory at a row pitch padded by 16 bytes, so
// that the eight rows one ldmatrix phase reads fall in different banks.
// ROW: the row-wise blocks (16 consecutive elements of a row, A row m = chunk
// row m of one block column); COL: the column-wise blocks (16 consecutive
// rows of a column, A row m = column m of a 16-column group, loaded
// transposed); both from one read for the dual pass.  Every BF16 amax with
// the transform runs here (when rows are 16-byte pieces), so the single- and
// dual-orientation quantizations of a tensor agree bit for bit.
constexpr uint32_t kMmaCW = 512;                  // columns per chunk (1 KB of BF16)
constexpr uint32_t kMmaPitch = kMmaCW * 2 + 16;   // padded row pitch in shared memory
constexpr uint32_t kMmaStage = 16 * kMmaPitch;    // 16,640 bytes
constexpr int kMmaRing = 3;   // 3 x 16.6 KB: 4 CTAs per SM
constexpr uint32_t kMmaSmem = kMmaRing * kMmaStage + 64;

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
// D = A B for A 16 x 16 (row-major fragment a), B 16 x 8 (fragment b0, b1).
__device__ __forceinline__ void mma_bf16(const uint32_t (&a)[4], uint32_t b0, uint32_t b1, float (&d)[4]) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%10,%10,%10,%10};"
                 : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}

template <bool ROW, bool COL>
__global__ void __launch_bounds__(kThreads, kStagedMinCtas) k_amax_mma(Args ar, Args ac, uint32_t ncc,
                                                                      uint32_t nchunks) {
    extern __shared__ __align__(128) uint8_t dsm[];
    __shared__ float s_red[kThreads / 32], s_red2[kThreads / 32];
    const Args &a = ROW ? ar : ac;   // the input as stored (both describe the same x)
    const uint32_t buf = ptx::smem_u32(dsm);
    const uint32_t bars = buf + kMmaRing * kMmaStage;
    volatile int *abort = reinterpret_cast<volatile int *>(dsm + kMmaRing * kMmaStage + 60);
    if (threadIdx.x == 0) {
        for (int t = 0; t < kMmaRing; ++t) ptx::mbar_init(bars + 8u * t, 1);
        *abort = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    const uint32_t rows = (uint32_t)a.rows, cols = (uint32_t)a.cols;
    uint32_t issued = 0, j = 0;
    // Chunk jj's 16 row copies are issued by the eight warps' lane 0, two rows
    // each; thread 0 also posts the chunk's byte count (the barrier's phase
    // needs that single arrival, so copies may land before or after it).
    auto issue = [&](uint32_t jj) {
        const uint32_t i = blockIdx.x + jj * gridDim.x;
        if (i >= nchunks) return;
        const uint32_t kb = i / ncc, cc = i - kb * ncc;
        const uint32_t c0 = cc * kMmaCW, r0 = kb * 16;
        const uint32_t ncols = min(kMmaCW, cols - c0), nrows = min(16u, rows - r0);
        const uint32_t bar = bars + 8u * (jj % kMmaRing);
        const uint32_t st = buf + (jj % kMmaRing) * kMmaStage;
        if (threadIdx.x == 0) ptx::mbar_arrive_expect_tx(bar, nrows * ncols * 2);
        const __nv_bfloat16 *src = static_cast<const __nv_bfloat16 *>(a.x) + (int64_t)r0 * a.ld + c0;
        for (uint32_t q = 2 * (threadIdx.x >> 5); q < min(nrows, 2 * (threadIdx.x >> 5) + 2); ++q)
            ptx::bulk_load(st + q * kMmaPitch, src + (int64_t)q * a.ld, ncols * 2, bar);
        issued = jj + 1;
    };
    if ((threadIdx.x & 31) == 0)
        for (uint32_t t = 0; t < kMmaRing; ++t) issue(t);
    // B fragments of H16 diag(d): B[k][n] = (-1)^popcount(n & k) d_k as BF16 +-1;
    // lane l holds k = 2 (l % 4) + {0, 1} (and + 8), n = l / 4 (and + 8)
    const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t smask = rht_sign_mask(a.rht_seed);
    auto bv = [&](uint32_t n, uint32_t k) -> uint32_t {
        return ((__popc(n & k) ^ (smask >> k)) & 1u) ? 0xBF80u : 0x3F80u;
    };
    const uint32_t k0 = 2 * (lane & 3), n0 = lane >> 2;
    const uint32_t bl0 = bv(n0, k0) | (bv(n0, k0 + 1) << 16), bl1 = bv(n0, k0 + 8) | (bv(n0, k0 + 9) << 16);
    const uint32_t bh0 = bv(n0 + 8, k0) | (bv(n0 + 8, k0 + 1) << 16);
    const uint32_t bh1 = bv(n0 + 8, k0 + 8) | (bv(n0 + 8, k0 + 9) << 16);
    float mr = 0.0f, mc = 0.0f;
    // running max of |D| over the A rows that hold data (rows m = lane / 4 and lane / 4 + 8)
    auto acc = [&](float &m, const float (&d)[4], const float (&e)[4], bool lo_ok, bool hi_ok) {
        if (lo_ok) m = max3_nan(max3_nan(m, fabsf(d[0]), fabsf(d[1])), fabsf(e[0]), fabsf(e[1]));
        if (hi_ok) m = max3_nan(max3_nan(m, fabsf(d[2]), fabsf(d[3])), fabsf(e[2]), fabsf(e[3]));
    };
    auto process = [&](uint32_t jj) {
        const uint32_t i = blockIdx.x + jj * gridDim.x;
        const uint32_t kb = i / ncc, cc = i - kb * ncc;
        const uint32_t c0 = cc * kMmaCW, r0 = kb * 16;
        const uint32_t ncols = min(kMmaCW, cols - c0), nrows = min(16u, rows - r0);
        const uint32_t st = buf + (jj % kMmaRing) * kMmaStage;
        if (ROW) {
            // groups = block columns b (16 rows of the chunk each); partial last rows masked
            const bool lo_ok = n0 < nrows, hi_ok = n0 + 8 < nrows;
            const uint32_t lrow = lane & 15, lhalf = (lane >> 4) * 16;
#pragma unroll
            for (uint32_t t = 0; t < kMmaCW / 16 / 8; ++t) {
                const uint32_t b = warp + 8 * t;
                if (b * 16 >= ncols) break;
                uint32_t af[4];
                ldsm_x4(st + lrow * kMmaPitch + b * 32 + lhalf, af);
                float d[4], e[4];
                mma_bf16(af, bl0, bl1, d);
                mma_bf16(af, bh0, bh1, e);
                acc(mr, d, e, lo_ok, hi_ok);
            }
        }
        if (COL) {
            // groups = 16 columns (16 rows each, loaded transposed); partial last group masked
            const uint32_t lrow = (lane & 7) + ((lane >> 4) << 3), lcol = ((lane >> 3) & 1) * 8;
#pragma unroll
            for (uint32_t t = 0; t < kMmaCW / 16 / 8; ++t) {
                const uint32_t g = warp + 8 * t;
                if (g * 16 >= ncols) break;
                uint32_t af[4];
                ldsm_x4_t(st + lrow * kMmaPitch + (g * 16 + lcol) * 2, af);
                float d[4], e[4];
                mma_bf16(af, bl0, bl1, d);
                mma_bf16(af, bh0, bh1, e);
                acc(mc, d, e, g * 16 + n0 < ncols, g * 16 + n0 + 8 < ncols);
            }
        }
    };
    bool ok = true;
    // one chunk per iteration, refilled as soon as every warp has read it
    // (measured 3 % faster than two chunks per barrier with a 4-deep ring)
    for (; j < nchunks && blockIdx.x + j * gridDim.x < nchunks; ++j) {
        const bool mine = ptx::mbar_wait_bounded(bars + 8u * (j % kMmaRing), (j / kMmaRing) & 1u, kRingWait);
        if (!mine) *abort = 1;
        else process(j);
        __syncthreads();
        if (*abort) { ok = false; break; }
        if ((threadIdx.x & 31) == 0) issue(j + kMmaRing);
    }
    if (!ok) {
        // every copy issued and not consumed lands before the CTA exits
        if (threadIdx.x == 0) atomicOr(&g_quant_timeout, 1u);
        if ((threadIdx.x & 31) == 0)
            for (uint32_t h = j; h < issued; ++h)
                if (!ptx::mbar_wait_bounded(bars + 8u * (h % kMmaRing), (h / kMmaRing) & 1u, kRingWait)) break;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        mr = max_nan(mr, __shfl_xor_sync(0xffffffffu, mr, o));
        mc = max_nan(mc, __shfl_xor_sync(0xffffffffu, mc, o));
    }
    if (lane == 0) { s_red[warp] = mr; s_red2[warp] = mc; }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kThreads / 32; ++w) { mr = max_nan(mr, s_red[w]); mc = max_nan(mc, s_red2[w]); }
        if (ROW) ar.partials_out[blockIdx.x] = mr * 0.25f;
        if (COL) ac.partials_out[blockIdx.x] = mc * 0.25f;
    }
}

// ================================================ dual orientation (X and X^T)
// A training step quantizes every operand both ways (X row-wise for one GEMM,
// X^T for another).  One read serves both: the column-wise ring of 16 rows x
// CW columns is staged as above, and each chunk is quantized as CW/2 column
// pairs (one unit per thread, output X^T) and as 16 x CW/16 row-wise blocks
// (two per thread for BF16, packed pairs; output X).  The two results keep
// their own tensor scale, SR counter and element numbering.  With AMAX the
// kernel only writes one partial maximum per CTA for each orientation (the
// row-wise and the column-wise transforms see different blocks).
template <class In, int GRID, int ROUND, bool RHT, bool AMAX>
__global__ void __launch_bounds__(kThreads, kStagedMinCtas) k_dual_staged(Args ar, Args ac, uint32_t ncc, uint32_t nchunks) {
    constexpr int kRing = ring_depth<AMAX>();
    extern __shared__ __align__(128) uint8_t dsm[];
    __shared__ float s_kr[256], s_kc[256];
    __shared__ float s_red[kThreads / 32];
    constexpr uint32_t CW = kChunk / (16 * sizeof(In));
    constexpr uint32_t BPR = CW / 16;   // row-wise blocks per chunk row
    const RingCtl ring = ring_init<kRing>(dsm);
    uint32_t issued = 0, j = 0;
    if (threadIdx.x == 0)
        for (uint32_t t = 0; t < kRing; ++t) col_issue<In, kRing>(ring, ar, t, nchunks, ncc, issued);
    const float qmax = GRID == kE2M1 ? 6.0f : ar.uqmax;
    float Sr = 1.0f, Sc = 1.0f;
    bool fr = false, fc = false;
    if (!AMAX) {
        float amr = 0.0f, amc = 0.0f;
        tensor_scale_prologue(ar, qmax, RHT ? 0.25f : 1.0f, s_kr, s_red, Sr, GRID == kE1M2 && ROUND == kRTNE, &fr,
                              &amr);
        tensor_scale_prologue(ac, qmax, RHT ? 0.25f : 1.0f, s_kc, s_red, Sc, GRID == kE1M2 && ROUND == kRTNE, &fc,
                              &amc);
        if (blockIdx.x == 0 && threadIdx.x == 0 && ar.status && !isfinite(amc)) *ar.status = 1u;
    }
    const uint32_t smask = RHT ? rht_sign_mask(ar.rht_seed) : 0u;
    const Signs sgr = row_signs<In>(smask), sgc = col_signs<In>(smask);
    const uint32_t nloc = nchunks > blockIdx.x ? (nchunks - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    const uint32_t csr = (uint32_t)(ar.kpad / 2), nktr = (uint32_t)ar.nkt;
    const uint32_t csc = (uint32_t)(ac.kpad / 2), nktc = (uint32_t)ac.nkt;
    const uint32_t cols = (uint32_t)ar.cols;
    float mr = 0.0f, mc = 0.0f;
    bool ok = true;
    auto process = [&](uint32_t jj) {
        const uint32_t i = blockIdx.x + jj * gridDim.x;
        const uint32_t kb = i / ncc, cc = i - kb * ncc;
        const uint32_t c0 = cc * CW;
        const uint32_t st = ring.buf + (jj % kRing) * kChunk;
        // column-wise unit: columns (c, c + 1), rows kb*16 .. +15
        const uint32_t c = c0 + 2 * threadIdx.x;
        if (2 * threadIdx.x < CW && c < cols) {
            ColRaw<In> raw;
            raw.load_shared(st + 2 * threadIdx.x * sizeof(In), CW * sizeof(In));
            if (AMAX) {
                uint64_t P[16];
                col_values<In, RHT>(raw, sgc, P);
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    float v0, v1;
                    upk2(P[q], v0, v1);
                    mc = max3_nan(mc, fabsf(v0), fabsf(v1));
                }
            } else {
                quant_unit_col<In, GRID, ROUND, RHT>(ac, raw, kb, c, true, sgc, Sc, s_kc, csc, nktc, fc);
            }
        }
        // row-wise blocks of the chunk: (row q, block bc) for k = q * BPR + bc
        if (sizeof(In) == 2) {
            // BF16: 512 blocks, thread t owns k = t and t + 256 (rows q and
            // q + 8, the same block column) as a packed pair
            const uint32_t q0 = threadIdx.x / BPR, bc = threadIdx.x % BPR;
            if (c0 + bc * 16 < cols) {
                Raw<__nv_bfloat16> r0, r1;
                r0.load_shared(st + q0 * (CW * 2) + bc * 32);
                r1.load_shared(st + (q0 + 8) * (CW * 2) + bc * 32);
                if (AMAX) {
                    uint64_t P[16];
#pragma unroll
                    for (int q = 0; q < 16; ++q) P[q] = RHT ? pk2(r0.get(q, sgr), r1.get(q, sgr)) : pk2(r0.get(q), r1.get(q));
                    if (RHT) {
#pragma unroll
                        for (int sgs = 1; sgs < 16; sgs <<= 1) {
#pragma unroll
                            for (int q = 0; q < 16; ++q) {
                                if ((q & sgs) == 0) {
                                    const uint64_t xx = P[q], yy = P[q + sgs];
                                    P[q] = add2(xx, yy);
                                    P[q + sgs] = sub2(xx, yy);
                                }
                            }
                        }
                    }
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        float u0, u1;
                        upk2(P[q], u0, u1);
                        mr = max3_nan(mr, fabsf(u0), fabsf(u1));
                    }
                } else {
                    const uint32_t b = cc * BPR + bc, r = kb * 16 + q0;
                    quant_pair_row<GRID, ROUND, RHT>(ar, r0, r1, r, b, r + 8, b, true, sgr, Sr, s_kr, csr, nktr, fr);
                }
            }
        } else {
            for (uint32_t k = threadIdx.x; k < 16 * BPR; k += kThreads) {
                const uint32_t q0 = k / BPR, bc = k % BPR;
                if (c0 + bc * 16 >= cols) continue;
                Raw<In> raw;
                raw.load_shared(st + q0 * (CW * sizeof(In)) + bc * 16 * sizeof(In));
                if (AMAX) {
                    float lo[8], hi[8];
                    block_values<In, RHT>(raw, sgr, lo, hi);
#pragma unroll
                    for (int q = 0; q < 8; ++q) mr = max3_nan(mr, fabsf(lo[q]), fabsf(hi[q]));
                } else {
                    quant_block_row<In, GRID, ROUND, RHT>(ar, raw, kb * 16 + q0, cc * BPR + bc, sgr, Sr, s_kr, csr,
                                                          nktr, fr);
                }
            }
        }
    };
    // One CTA barrier per iteration (each thread waits for its chunks itself);
    // the amax pass, light on arithmetic, takes two chunks per iteration.
    while (j < nloc) {
        const uint32_t nj = (AMAX && j + 1 < nloc) ? 2u : 1u;
        bool mine = true;
        for (uint32_t t = 0; t < nj && mine; ++t) mine = ring_wait_own<kRing>(ring, j + t);
        if (mine)
            for (uint32_t t = 0; t < nj; ++t) process(j + t);
        __syncthreads();
        if (*ring.abort) { ok = false; break; }
        if (threadIdx.x == 0)
            for (uint32_t t = 0; t < nj; ++t) col_issue<In, kRing>(ring, ar, j + t + kRing, nchunks, ncc, issued);
        j += nj;
    }
    if (!ok) {
        if (threadIdx.x == 0) atomicOr(&g_quant_timeout, 1u);
        ring_drain<kRing>(ring, j, issued);
    }
    if (AMAX) {
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            mr = max_nan(mr, __shfl_xor_sync(0xffffffffu, mr, o));
            mc = max_nan(mc, __shfl_xor_sync(0xffffffffu, mc, o));
        }
        __shared__ float s_red2[kThreads / 32];
        if ((threadIdx.x & 31) == 0) { s_red[threadIdx.x >> 5] = mr; s_red2[threadIdx.x >> 5] = mc; }
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int w = 1; w < kThreads / 32; ++w) { mr = max_nan(mr, s_red[w]); mc = max_nan(mc, s_red2[w]); }
            ar.partials_out[blockIdx.x] = RHT ? mr * 0.25f : mr;
            ac.partials_out[blockIdx.x] = RHT ? mc * 0.25f : mc;
        }
    } else {
        // row-wise result: padding blocks cols/16 .. kpad/16 - 1 of every row
        const uint32_t kvr = cols / 16, nbr = (uint32_t)(ar.kpad / 16) - kvr;
        const uint32_t npr = (uint32_t)ar.out_rows * nbr;
        for (uint32_t t = blockIdx.x * blockDim.x + threadIdx.x; t < npr; t += gridDim.x * blockDim.x) {
            const uint32_t r = t / nbr, b = kvr + (t - r * nbr);
            put_codes(ar, (size_t)r * csr + b * 8, make_uint2(0u, 0u));
            ar.scales[scale_offset32(r, b, nktr)] = 0;
        }
        zero_pad_rows(ar);
        // column-wise result: padding blocks past the last input row
        const uint32_t kvc = (uint32_t)(ac.rows / 16), nbc = (uint32_t)(ac.kpad / 16) - kvc;
        const uint32_t npc = (uint32_t)ac.out_rows * nbc;
        for (uint32_t t = blockIdx.x * blockDim.x + threadIdx.x; t < npc; t += gridDim.x * blockDim.x) {
            const uint32_t r = t / nbc, b = kvc + (t - r * nbc);
            put_codes(ac, (size_t)r * csc + b * 8, make_uint2(0u, 0u));
            ac.scales[scale_offset32(r, b, nktc)] = 0;
        }
        zero_pad_rows(ac);
    }
}

// BF16 inputs use square-ish tiles instead: 128 rows x 64 columns (16 KB) per
// ring stage, one TMA tile copy each.  Each tile is 8 row blocks deep, so the
// column-wise result of a column is 8 consecutive blocks (64 contiguous code
// bytes, two 4-byte scale words): the codes are staged in shared memory and
// leave as 16-byte stores, instead of 8-byte stores to 32 different rows per
// warp instruction.  Row-wise, a tile row is 4 blocks (32 code bytes).
constexpr uint32_t kTileRows = 128, kTileCols = 64;
constexpr uint32_t kTileBytes = kTileRows * kTileCols * 2;   // BF16
static_assert(kTileBytes == kChunk, "a tile fills one ring stage");
constexpr uint32_t kColStageBytes = 8 * kTileCols * 8 + 8 * kTileCols;   // codes [8][64] x 8 B + scales [8][64]
// k_dual_tile and k_dual_tile_grouped stage tile j's column-wise results in
// buffer j % 2 of two, so one CTA barrier per tile orders both the ring
// slot's reuse and the staging buffer's.  k_dual_tile's ring is 2 deep (4
// CTAs per SM fit, about 42 KB each; a third stage measured no faster with
// SR, whose registers allow 3 CTAs per SM); the grouped kernel keeps 3.
constexpr int kDualRing = 2;
template <int KRING> constexpr uint32_t dual_smem() { return KRING * kChunk + 64 + 2 * kColStageBytes; }

// Geometry of the dual-orientation tile kernels, fixed per launch.
struct DualGeom {
    uint32_t csr, nktr, csc, nktc;   // code row strides (bytes) and k atoms of the two results
    uint32_t cols, rows;             // the input
    uint32_t kvr, kbr, kbp;          // real row-wise blocks per row; real and padded column-wise blocks
    uint32_t cp, rb, q, bc;          // this thread's column pair / row block, and row / block column
};
// tid: the thread's index within the 256 threads that share one tile's work
__device__ __forceinline__ DualGeom dual_geom(const Args &ar, const Args &ac, uint32_t tid = threadIdx.x) {
    DualGeom g;
    g.csr = (uint32_t)(ar.kpad / 2); g.nktr = (uint32_t)ar.nkt;
    g.csc = (uint32_t)(ac.kpad / 2); g.nktc = (uint32_t)ac.nkt;
    g.cols = (uint32_t)ar.cols; g.rows = (uint32_t)ar.rows;
    g.kvr = g.cols / 16; g.kbr = g.rows / 16; g.kbp = (uint32_t)(ac.kpad / 16);
    g.cp = tid % 32; g.rb = tid / 32;
    g.q = tid / 4; g.bc = tid % 4;
    return g;
}

// Quantization of one 128 x 64 BF16 tile (rt, ct) held at shared address st,
// both orientations.  Column-wise: this thread's unit (columns c0 + 2 cp, +1;
// rows r0 + 16 rb .. + 15), staged in stage_codes / stage_scales when STAGE
// (written out by dual_tile_flush), else stored directly.  Row-wise: rows
// r0 + q and r0 + q + 64, block c0 / 16 + bc, stored directly.
// PARTS: 1 the column-wise unit only, 2 the row-wise blocks only, 3 both.
template <int GRID, int ROUND, bool RHT, bool STAGE, int PARTS = 3>
__device__ __forceinline__ void dual_tile_quant(const Args &ar, const Args &ac, const DualGeom &g, uint32_t st,
                                                uint32_t rt, uint32_t ct, const Signs &sgr, const Signs &sgc,
                                                float Sr, float Sc, const float *s_kr, const float *s_kc, bool fr,
                                                bool fc, uint8_t *stage_codes, uint8_t *stage_scales) {
    const uint32_t r0 = rt * kTileRows, c0 = ct * kTileCols;
    if (PARTS & 2) {
        const uint32_t r = r0 + g.q, b = ct * (kTileCols / 16) + g.bc;
        if (r < g.rows && b < g.kvr) {
            Raw<__nv_bfloat16> ra, rbw;
            ra.load_shared(st + g.q * (kTileCols * 2) + g.bc * 32);
            rbw.load_shared(st + (g.q + 64) * (kTileCols * 2) + g.bc * 32);
            // one block at a time (measured faster than the packed pair, which
            // holds twice the registers)
            quant_block_row<__nv_bfloat16, GRID, ROUND, RHT>(ar, ra, r, b, sgr, Sr, s_kr, g.csr, g.nktr, fr);
            if (r + 64 < g.rows)
                quant_block_row<__nv_bfloat16, GRID, ROUND, RHT>(ar, rbw, r + 64, b, sgr, Sr, s_kr, g.csr, g.nktr, fr);
        }
    }
    if (PARTS & 1) {
        const uint32_t c = c0 + 2 * g.cp, kb = rt * 8 + g.rb;
        ColRaw<__nv_bfloat16> raw;
        raw.load_shared(st + 16 * g.rb * (kTileCols * 2) + g.cp * 4, kTileCols * 2);
        if (STAGE) {
            uint2 w0 = make_uint2(0u, 0u), w1 = make_uint2(0u, 0u);
            uint32_t e0 = 0, e1 = 0;
            if (c < g.cols && kb < g.kbr)
                col_unit_words<__nv_bfloat16, GRID, ROUND, RHT>(ac, raw, kb, c, true, sgc, Sc, s_kc, fc, w0, w1, e0,
                                                                e1);
            // staging [rb][column] (consecutive columns -> consecutive words)
            reinterpret_cast<uint2 *>(stage_codes)[g.rb * kTileCols + 2 * g.cp] = w0;
            reinterpret_cast<uint2 *>(stage_codes)[g.rb * kTileCols + 2 * g.cp + 1] = w1;
            stage_scales[g.rb * kTileCols + 2 * g.cp] = (uint8_t)e0;
            stage_scales[g.rb * kTileCols + 2 * g.cp + 1] = (uint8_t)e1;
        } else if (c < g.cols && kb < g.kbp) {
            // padding blocks past the last row are written as zeros
            quant_unit_col<__nv_bfloat16, GRID, ROUND, RHT>(ac, raw, kb, c, kb < g.kbr, sgc, Sc, s_kc, g.csc, g.nktc,
                                                            fc);
        }
    }
}

// The staged column-wise results of tile (rt, ct): column c, blocks
// rt * 8 .. + 7 = 64 contiguous code bytes (16 per thread), and the scales as
// two 4-byte words of an atom.
__device__ __forceinline__ void dual_tile_flush(const Args &ac, const DualGeom &g, uint32_t rt, uint32_t ct,
                                                const uint8_t *stage_codes, const uint8_t *stage_scales) {
    const uint32_t c0 = ct * kTileCols, kb0 = rt * 8;
    {
        const uint32_t cl = threadIdx.x / 4, part = threadIdx.x % 4;
        const uint32_t c = c0 + cl, kb = kb0 + 2 * part;
        if (c < g.cols && kb < g.kbp) {
            const uint2 a0 = reinterpret_cast<const uint2 *>(stage_codes)[(2 * part) * kTileCols + cl];
            const uint2 a1 = reinterpret_cast<const uint2 *>(stage_codes)[(2 * part + 1) * kTileCols + cl];
            put_codes(ac, (size_t)c * g.csc + kb * 8, make_uint4(a0.x, a0.y, a1.x, a1.y));
        }
    }
    if (threadIdx.x < 2 * kTileCols) {
        const uint32_t cl = threadIdx.x / 2, h = threadIdx.x % 2;
        const uint32_t c = c0 + cl, kb = kb0 + 4 * h;
        if (c < g.cols && kb < g.kbp) {
            uint32_t w = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) w |= (uint32_t)stage_scales[(4 * h + k) * kTileCols + cl] << (8 * k);
            *reinterpret_cast<uint32_t *>(ac.scales + scale_offset32(c, kb, g.nktc)) = w;
        }
    }
}

// Row-wise padding blocks cols/16 .. kpad/16 - 1 of every row of a dual
// result, and the scale entries of both results' padding rows.
__device__ __forceinline__ void dual_padding(const Args &ar, const Args &ac, const DualGeom &g) {
    const uint32_t nbr = (uint32_t)(ar.kpad / 16) - g.kvr;
    const uint32_t npr = (uint32_t)ar.out_rows * nbr;
    for (uint32_t t = blockIdx.x * blockDim.x + threadIdx.x; t < npr; t += gridDim.x * blockDim.x) {
        const uint32_t r = t / nbr, b = g.kvr + (t - r * nbr);
        put_codes(ar, (size_t)r * g.csr + b * 8, make_uint2(0u, 0u));
        ar.scales[scale_offset32(r, b, g.nktr)] = 0;
    }
    zero_pad_rows(ar);
    zero_pad_rows(ac);   // column-wise padding blocks come from zero-filled tile rows
}

template <int GRID, int ROUND, bool RHT>
__global__ void __launch_bounds__(kThreads, kStagedMinCtas)
    k_dual_tile(const __grid_constant__ CUtensorMap tmx, Args ar, Args ac, uint32_t nct, uint32_t ntiles) {
    constexpr int kRing = kDualRing;
    extern __shared__ __align__(128) uint8_t dsm[];
    __shared__ float s_kr[256], s_kc[256];
    __shared__ float s_red[kThreads / 32];
    const RingCtl ring = ring_init<kRing>(dsm);
    // staging buffer b: codes [rb][cl] uint2, then scales [rb][cl] byte
    uint8_t *const stage0 = dsm + kRing * kChunk + 64;
    uint32_t issued = 0, j = 0;
    auto issue = [&](uint32_t jj) {
        const uint32_t i = blockIdx.x + jj * gridDim.x;
        if (i >= ntiles) return;
        const uint32_t rt = i / nct, ct = i - rt * nct;
        const uint32_t bar = ring.bars + 8u * (jj % kRing);
        ptx::mbar_arrive_expect_tx(bar, kTileBytes);   // out-of-range elements arrive as zeros
        ptx::tma_load_2d(ring.buf + (jj % kRing) * kChunk, &tmx, (int32_t)(ct * kTileCols),
                         (int32_t)(rt * kTileRows), bar);
        issued = jj + 1;
    };
    if (threadIdx.x == 0) {
        ptx::prefetch_tmap(&tmx);
        for (uint32_t t = 0; t < kRing; ++t) issue(t);
    }
    const float qmax = GRID == kE2M1 ? 6.0f : ar.uqmax;
    float Sr = 1.0f, Sc = 1.0f;
    bool fr = false, fc = false;
    float amr = 0.0f, amc = 0.0f;
    tensor_scale_prologue(ar, qmax, RHT ? 0.25f : 1.0f, s_kr, s_red, Sr, GRID == kE1M2 && ROUND == kRTNE, &fr, &amr);
    tensor_scale_prologue(ac, qmax, RHT ? 0.25f : 1.0f, s_kc, s_red, Sc, GRID == kE1M2 && ROUND == kRTNE, &fc, &amc);
    if (blockIdx.x == 0 && threadIdx.x == 0 && ar.status && !isfinite(amc)) *ar.status = 1u;
    const uint32_t smask = RHT ? rht_sign_mask(ar.rht_seed) : 0u;
    const Signs sgr = row_signs<__nv_bfloat16>(smask), sgc = col_signs<__nv_bfloat16>(smask);
    const uint32_t nloc = ntiles > blockIdx.x ? (ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    const DualGeom g = dual_geom(ar, ac);
    bool ok = true;
    for (; j < nloc; ++j) {
        // each thread waits for the tile itself; no CTA barrier before the work
        const bool mine = ring_wait_own<kRing>(ring, j);
        const uint32_t i = blockIdx.x + j * gridDim.x;
        const uint32_t rt = i / nct, ct = i - rt * nct;
        uint8_t *const stage_codes = stage0 + (j & 1) * kColStageBytes;
        uint8_t *const stage_scales = stage_codes + 8 * kTileCols * 8;
        if (mine)
            dual_tile_quant<GRID, ROUND, RHT, true>(ar, ac, g, ring.buf + (j % kRing) * kChunk, rt, ct, sgr, sgc, Sr,
                                                    Sc, s_kr, s_kc, fr, fc, stage_codes, stage_scales);
        // tile j consumed and its column-wise results staged; every thread has
        // also finished flushing tile j - 1, whose buffer tile j + 1 reuses
        __syncthreads();
        if (*ring.abort) { ok = false; break; }
        if (threadIdx.x == 0) issue(j + kRing);
        dual_tile_flush(ac, g, rt, ct, stage_codes, stage_scales);
    }
    if (!ok) {
        if (threadIdx.x == 0) atomicOr(&g_quant_timeout, 1u);
        ring_drain<kRing>(ring, j, issued);
    }
    dual_padding(ar, ac, g);
}

// ======================================== on-chip single pass (dual, BF16)
// For a tensor that fits in the GPU's shared memory (up to kResidentMax
// 128 x 64 tiles per SM), one cooperative launch of one CTA per SM reads it
// once: each CTA loads its tiles (TMA) and keeps them resident, computes both
// orientations' maxima from them -- with the transform through the same
// tensor-core products as k_amax_mma, so the result is bit for bit the
// two-pass one -- and writes one partial maximum per orientation; after a
// bounded grid barrier (a counter in the workspace that the launch zeroes)
// every CTA reduces all partials to the two tensor scales and quantizes its
// resident tiles.  The input's second read, and a launch, go away.
constexpr uint32_t kResidentMax = 14;
constexpr uint32_t kResidentSmem = kResidentMax * kTileBytes + 128;

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Maxima of |4 y| (or |x| without the transform) of one resident tile, row-wise
// blocks into mr and column-wise blocks into mc, by the CTA's NT threads.
// Elements outside the tensor arrive as zeros.
template <bool RHT, int NT>
__device__ __forceinline__ void tile_maxima(uint32_t st, uint32_t bl0, uint32_t bl1, uint32_t bh0, uint32_t bh1,
                                            float &mr, float &mc) {
    static_assert(NT == 256 || NT == 512, "one or two row blocks per thread; 32 A groups over the warps");
    const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (!RHT) {
        // the orientations share max |x|: the thread's row-wise blocks (rows
        // q and q + 64 with 256 threads, row q with 512)
        const uint32_t q = threadIdx.x / 4, bc = threadIdx.x % 4;
#pragma unroll
        for (uint32_t h = 0; h < 512 / NT; ++h) {
            Raw<__nv_bfloat16> ra;
            ra.load_shared(st + (q + 64 * h) * (kTileCols * 2) + bc * 32);
#pragma unroll
            for (int e = 0; e < 16; e += 2) mr = max3_nan(mr, fabsf(ra.get(e)), fabsf(ra.get(e + 1)));
        }
        mc = mr;
        return;
    }
#pragma unroll
    for (uint32_t u = 0; u < 32 / (NT / 32); ++u) {
        const uint32_t G = warp + (NT / 32) * u, band = G / 4, sft = G % 4;
        float d[4], e[4];
        uint32_t af[4];
        // row-wise: A row m = tile row 16 band + m, block column (sft + m) % 4
        {
            const uint32_t m = lane & 15, half = lane >> 4;
            ldsm_x4(st + (band * 16 + m) * (kTileCols * 2) + ((sft + m) & 3) * 32 + half * 16, af);
            mma_bf16(af, bl0, bl1, d);
            mma_bf16(af, bh0, bh1, e);
#pragma unroll
            for (int k = 0; k < 4; ++k) mr = max3_nan(mr, fabsf(d[k]), fabsf(e[k]));
        }
        // column-wise: A row m = column 16 sft + m, k = tile rows 16 band .. + 15
        {
            const uint32_t lrow = (lane & 7) + ((lane >> 4) << 3), lcol = ((lane >> 3) & 1) * 8;
            ldsm_x4_t(st + (band * 16 + lrow) * (kTileCols * 2) + (sft * 16 + lcol) * 2, af);
            mma_bf16(af, bl0, bl1, d);
            mma_bf16(af, bh0, bh1, e);
#pragma unroll
            for (int k = 0; k < 4; ++k) mc = max3_nan(mc, fabsf(d[k]), fabsf(e[k]));
        }
    }
}

// The single pass runs 512 threads per CTA (one CTA per SM): the maxima
// spread over 16 warps, and the quantization gives each tile's column-wise
// units to threads 0-255 and its row-wise blocks to threads 256-511, both
// stored directly, so the two halves need no barrier between them.
constexpr int kResidentThreads = 512;

template <int GRID, int ROUND, bool RHT>
__global__ void __launch_bounds__(kResidentThreads, 1)
    k_dual_resident(const __grid_constant__ CUtensorMap tmx, Args ar, Args ac, uint32_t nct, uint32_t ntiles,
                    uint32_t *arrive) {
    extern __shared__ __align__(128) uint8_t dsm[];
    __shared__ float s_kr[256], s_kc[256];
    __shared__ float s_red[kResidentThreads / 32], s_red2[kResidentThreads / 32];
    __shared__ int s_go;
    const uint32_t buf = ptx::smem_u32(dsm);
    const uint32_t bars = buf + kResidentMax * kTileBytes;
    const uint32_t nloc = ntiles > blockIdx.x ? (ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    auto tile_of = [&](uint32_t t, uint32_t &rt, uint32_t &ct) {
        const uint32_t i = blockIdx.x + t * gridDim.x;
        rt = i / nct;
        ct = i - rt * nct;
    };
    if (threadIdx.x == 0) {
        for (uint32_t t = 0; t < nloc; ++t) ptx::mbar_init(bars + 8u * t, 1);
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmx);
        for (uint32_t t = 0; t < nloc; ++t) {
            uint32_t rt, ct;
            tile_of(t, rt, ct);
            ptx::mbar_arrive_expect_tx(bars + 8u * t, kTileBytes);
            ptx::tma_load_2d(buf + t * kTileBytes, &tmx, (int32_t)(ct * kTileCols), (int32_t)(rt * kTileRows),
                             bars + 8u * t);
        }
    }
    __syncthreads();
    // 1. both orientations' maxima over the resident tiles
    const uint32_t smask = RHT ? rht_sign_mask(ar.rht_seed) : 0u;
    uint32_t bl0 = 0, bl1 = 0, bh0 = 0, bh1 = 0;
    if (RHT) {
        const uint32_t lane = threadIdx.x & 31, k0 = 2 * (lane & 3), n0 = lane >> 2;
        auto bv = [&](uint32_t n, uint32_t k) -> uint32_t {
            return ((__popc(n & k) ^ (smask >> k)) & 1u) ? 0xBF80u : 0x3F80u;
        };
        bl0 = bv(n0, k0) | (bv(n0, k0 + 1) << 16);
        bl1 = bv(n0, k0 + 8) | (bv(n0, k0 + 9) << 16);
        bh0 = bv(n0 + 8, k0) | (bv(n0 + 8, k0 + 1) << 16);
        bh1 = bv(n0 + 8, k0 + 8) | (bv(n0 + 8, k0 + 9) << 16);
    }
    float mr = 0.0f, mc = 0.0f;
    bool ok = true;
    for (uint32_t t = 0; t < nloc && ok; ++t) {
        ok = ptx::mbar_wait_bounded(bars + 8u * t, 0u, kRingWait);
        if (ok) tile_maxima<RHT, kResidentThreads>(buf + t * kTileBytes, bl0, bl1, bh0, bh1, mr, mc);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        mr = max_nan(mr, __shfl_xor_sync(0xffffffffu, mr, o));
        mc = max_nan(mc, __shfl_xor_sync(0xffffffffu, mc, o));
    }
    if ((threadIdx.x & 31) == 0) { s_red[threadIdx.x >> 5] = mr; s_red2[threadIdx.x >> 5] = mc; }
    ok = __syncthreads_and(ok) != 0;
    // 2. partial maxima out (NaN from a CTA whose copies did not land in time,
    // so that the others do not wait for it and see a non-finite amax), then
    // the grid barrier -- every CTA is resident (cooperative launch) -- bounded
    if (threadIdx.x == 0) {
        for (int w = 1; w < kResidentThreads / 32; ++w) { mr = max_nan(mr, s_red[w]); mc = max_nan(mc, s_red2[w]); }
        ar.partials_out[blockIdx.x] = ok ? (RHT ? mr * 0.25f : mr) : __int_as_float(0x7FFFFFFF);
        ac.partials_out[blockIdx.x] = ok ? (RHT ? mc * 0.25f : mc) : __int_as_float(0x7FFFFFFF);
        __threadfence();
        atomicAdd(arrive, 1u);
    }
    if (!ok) {
        // wait (bounded) for every copy of this CTA before leaving
        if (threadIdx.x == 0) {
            atomicOr(&g_quant_timeout, 1u);
            for (uint32_t t = 0; t < nloc; ++t)
                if (!ptx::mbar_wait_bounded(bars + 8u * t, 0u, kRingWait)) break;
        }
        return;
    }
    if (threadIdx.x == 0) {
        const long long t0 = clock64();
        bool go = true;
        while (ld_acquire_u32(arrive) < gridDim.x) {
            if (clock64() - t0 > kRingWait) { go = false; break; }
            __nanosleep(64);
        }
        s_go = go;
        if (!go) atomicOr(&g_quant_timeout, 1u);
    }
    __syncthreads();
    if (!s_go) return;
    // 3. tensor scales from all partial maxima, then the resident tiles
    const float qmax = GRID == kE2M1 ? 6.0f : ar.uqmax;
    float Sr = 1.0f, Sc = 1.0f;
    bool fr = false, fc = false;
    float amr = 0.0f, amc = 0.0f;
    tensor_scale_prologue(ar, qmax, RHT ? 0.25f : 1.0f, s_kr, s_red, Sr, GRID == kE1M2 && ROUND == kRTNE, &fr, &amr);
    tensor_scale_prologue(ac, qmax, RHT ? 0.25f : 1.0f, s_kc, s_red, Sc, GRID == kE1M2 && ROUND == kRTNE, &fc, &amc);
    if (blockIdx.x == 0 && threadIdx.x == 0 && ar.status && !isfinite(amc)) *ar.status = 1u;
    const Signs sgr = row_signs<__nv_bfloat16>(smask), sgc = col_signs<__nv_bfloat16>(smask);
    const bool col_half = threadIdx.x < 256;
    const DualGeom g = dual_geom(ar, ac, threadIdx.x & 255u);
    for (uint32_t t = 0; t < nloc; ++t) {
        uint32_t rt, ct;
        tile_of(t, rt, ct);
        if (col_half)
            dual_tile_quant<GRID, ROUND, RHT, false, 1>(ar, ac, g, buf + t * kTileBytes, rt, ct, sgr, sgc, Sr, Sc,
                                                        s_kr, s_kc, fr, fc, nullptr, nullptr);
        else
            dual_tile_quant<GRID, ROUND, RHT, false, 2>(ar, ac, g, buf + t * kTileBytes, rt, ct, sgr, sgc, Sr, Sc,
                                                        s_kr, s_kc, fr, fc, nullptr, nullptr);
    }
    dual_padding(ar, ac, g);
}

// ====================================================== grouped (MoE) path
// Segments are found by binary search over prefix tables copied into shared
// memory: find_seg returns the largest e with pre[e] <= u (empty segments are
// skipped because their start equals the next one's).
__device__ __forceinline__ int find_seg(const int64_t *pre, int n, int64_t u) {
    int lo = 0, hi = n;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pre[mid] <= u) lo = mid; else hi = mid;
    }
    return lo;
}

struct GroupSmem {
    int64_t in_row[kMaxGroups + 1];
    int64_t out_off[kMaxGroups];
    int64_t units[kMaxGroups + 1];
    float senc[kMaxGroups];
};

__device__ __forceinline__ void load_group_tables(const GroupQuant &gt, GroupSmem &sm) {
    for (int i = threadIdx.x; i <= gt.n; i += blockDim.x) {
        sm.in_row[i] = gt.in_row[i];
        sm.units[i] = gt.units[i];
        if (i < gt.n) sm.out_off[i] = gt.out_off[i];
    }
    __syncthreads();
}

__device__ __forceinline__ void seg_max_flush(uint32_t *slots, int e, float m) {
    if (e >= 0 && m > 0.0f) atomicMax(slots + e, __float_as_uint(m));
    else if (e >= 0 && !(m == m)) atomicMax(slots + e, 0x7FC00000u);   // NaN
}

// Per-segment maxima (row-wise: units are real 16-blocks, unit -> (row, block);
// column-wise: units are 16-row x 2-column pieces, unit -> (row block, pair)).
// Warp-contiguous chunks keep segment changes (and atomics) rare.
template <class In, bool RHT, bool COL>
__global__ void __launch_bounds__(kThreads) k_amax_grouped(Args a, const __grid_constant__ GroupQuant gt,
                                                           FastDiv div, uint32_t per_row, uint32_t *slots) {
    __shared__ GroupSmem sm;
    load_group_tables(gt, sm);
    const uint32_t smask = RHT ? rht_sign_mask(a.rht_seed) : 0u;
    const Signs sg = COL ? col_signs<In>(smask) : row_signs<In>(smask);
    const In *x = static_cast<const In *>(a.x);
    const int64_t total = sm.units[gt.n];
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t wid = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int64_t chunk = ((total + nwarps - 1) / nwarps + 31) / 32 * 32;
    const int lane = threadIdx.x & 31;
    int e_cur = -1;
    float m = 0.0f;
    const int64_t uend = total < (wid + 1) * chunk ? total : (wid + 1) * chunk;
    for (int64_t u = wid * chunk + lane; u < uend; u += 32) {
        const int e = (e_cur >= 0 && u < sm.units[e_cur + 1]) ? e_cur : find_seg(sm.units, gt.n, u);
        if (e != e_cur) {
            seg_max_flush(slots, e_cur, RHT ? m * 0.25f : m);
            e_cur = e;
            m = 0.0f;
        }
        const uint32_t lu = (uint32_t)(u - sm.units[e]);
        const uint32_t q = fdiv(lu, div), rem = lu - q * per_row;
        if (!COL) {
            Raw<In> raw;
            raw.load(x + (sm.in_row[e] + q) * a.ld + rem * 16);
            float lo[8], hi[8];
            block_values<In, RHT>(raw, sg, lo, hi);
#pragma unroll
            for (int j = 0; j < 8; ++j) m = max3_nan(m, fabsf(lo[j]), fabsf(hi[j]));
        } else {
            const int64_t seg_rows = sm.in_row[e + 1] - sm.in_row[e];
            const int64_t left = seg_rows - 16 * (int64_t)q;
            const int nvalid = left < 16 ? (int)left : 16;
            ColRaw<In> raw;
            raw.load_rows(x + (sm.in_row[e] + 16 * (int64_t)q) * a.ld + rem * 2, a.ld, nvalid);
            uint64_t P[16];
            col_values<In, RHT>(raw, sg, P);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float c0, c1;
                upk2(P[i], c0, c1);
                m = max3_nan(m, fabsf(c0), fabsf(c1));
            }
        }
    }
    seg_max_flush(slots, e_cur, RHT ? m * 0.25f : m);
}

// Quantization of every segment with its own tensor scale.  Row-wise units
// cover rows [0, rpad(T_e)) x all kpad/16 blocks of each segment (padding
// rows and blocks are written as zeros); column-wise units cover the
// segment's kpad(T_e)/16 row blocks x column pairs.
template <class In, int GRID, int ROUND, bool RHT, bool COL>
__global__ void __launch_bounds__(kThreads) k_quant_grouped(Args a, const __grid_constant__ GroupQuant gt,
                                                            FastDiv div, uint32_t per_row, const uint32_t *slots) {
    __shared__ GroupSmem sm;
    load_group_tables(gt, sm);
    const float qmax = GRID == kE2M1 ? 6.0f : a.uqmax;
    for (int e = threadIdx.x; e < gt.n; e += blockDim.x) {
        const float A_t = __uint_as_float(slots[e]);
        float se = 1.0f, sd = 1.0f;
        if (A_t > 0.0f) {
            const float num = 448.0f * qmax;
            se = __fdiv_rn(num, A_t);
            if (se > kFltMax) se = kFltMax;
            sd = __fdiv_rn(A_t, num);
        }
        sm.senc[e] = se;
        if (blockIdx.x == 0) {
            a.tensor_scale[e] = sd;
            if (!isfinite(A_t) && a.status) atomicOr(a.status, 1u);
        }
    }
    __syncthreads();
    const uint32_t smask = RHT ? rht_sign_mask(a.rht_seed) : 0u;
    const Signs sg = COL ? col_signs<In>(smask) : row_signs<In>(smask);
    const In *x = static_cast<const In *>(a.x);
    const int64_t total = sm.units[gt.n];
    const uint32_t cstride = (uint32_t)(a.kpad / 2), nkt = (uint32_t)a.nkt;
    const uint32_t kvb = (uint32_t)(a.k / 16);
    for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < total;
         u += (int64_t)gridDim.x * blockDim.x) {
        const int e = find_seg(sm.units, gt.n, u);
        const uint32_t lu = (uint32_t)(u - sm.units[e]);
        const uint32_t q = fdiv(lu, div), rem = lu - q * per_row;
        const int64_t seg_rows = sm.in_row[e + 1] - sm.in_row[e];
        const float S_enc = sm.senc[e];
        if (!COL) {
            // q: row within the segment, rem: block within the row
            Raw<In> raw;
            if ((int64_t)q < seg_rows && rem < kvb) raw.load(x + (sm.in_row[e] + q) * a.ld + rem * 16);
            else raw.zero();
            quant_block_row<In, GRID, ROUND, RHT>(a, raw, (uint32_t)(sm.out_off[e] + q), rem, sg, S_enc, nullptr,
                                                  cstride, nkt, false);
        } else {
            // q: row block within the segment, rem: column pair
            const int64_t left = seg_rows - 16 * (int64_t)q;
            const int nvalid = left <= 0 ? 0 : (left < 16 ? (int)left : 16);
            ColRaw<In> raw;
            if (nvalid > 0) raw.load_rows(x + (sm.in_row[e] + 16 * (int64_t)q) * a.ld + rem * 2, a.ld, nvalid);
            else raw.zero();
            quant_unit_col<In, GRID, ROUND, RHT>(a, raw, (uint32_t)(sm.out_off[e] / 16 + q), rem * 2, nvalid > 0,
                                                 sg, S_enc, nullptr, cstride, nkt, false);
        }
    }
    zero_pad_rows(a);
}

// Row-wise grouped quantization of a contiguous input through the staged
// ring: the segments are consecutive rows of one [sum T_e x cols] tensor, so
// its 16 KB chunks stream as in k_row_staged.  Each block finds its segment
// by input row (binary search over the prefix table in shared memory, cached
// between blocks), takes that segment's tensor scale and lands in the
// segment's output rows.  AMAX: per-segment maxima by atomicMax on the bit
// patterns; a CTA takes a contiguous run of chunks, so a thread meets one or
// two segments and flushes once per segment (strided chunks would visit every
// segment and flush per chunk).  The quantization pass then zeroes the
// padding blocks of every output row and every block of the segments'
// padding rows.
template <class In, int GRID, int ROUND, bool RHT, bool AMAX>
__global__ void __launch_bounds__(kThreads, kStagedMinCtas)
    k_row_grouped_staged(Args a, const __grid_constant__ GroupQuant gt, FastDiv bdiv, uint32_t kvb,
                         uint32_t nchunks, uint64_t total_bytes, uint32_t *slots) {
    constexpr int kRing = ring_depth<AMAX>();
    extern __shared__ __align__(128) uint8_t dsm[];
    __shared__ GroupSmem sm;
    const RingCtl ring = ring_init<kRing>(dsm);
    // chunk of local step j: contiguous runs (AMAX) or strided (quantization)
    const uint32_t per = AMAX ? (nchunks + gridDim.x - 1) / gridDim.x : 0u;
    const uint32_t nloc = AMAX ? (blockIdx.x * per < nchunks ? min(per, nchunks - blockIdx.x * per) : 0u)
                               : (nchunks > blockIdx.x ? (nchunks - blockIdx.x + gridDim.x - 1) / gridDim.x : 0u);
    auto chunk_of = [&](uint32_t jj) { return AMAX ? blockIdx.x * per + jj : blockIdx.x + jj * gridDim.x; };
    uint32_t issued = 0, j = 0;
    auto issue = [&](uint32_t jj) {
        if (jj >= nloc) return;
        const uint64_t off = (uint64_t)chunk_of(jj) * kChunk;
        const uint64_t rem = total_bytes - off;
        const uint32_t bytes = rem < kChunk ? (uint32_t)rem : kChunk;
        const uint32_t bar = ring.bars + 8u * (jj % kRing);
        ptx::mbar_arrive_expect_tx(bar, bytes);
        ptx::bulk_load(ring.buf + (jj % kRing) * kChunk, static_cast<const uint8_t *>(a.x) + off, bytes, bar);
        issued = jj + 1;
    };
    if (threadIdx.x == 0)
        for (uint32_t t = 0; t < kRing; ++t) issue(t);
    load_group_tables(gt, sm);
    if (!AMAX) {
        const float qmax = GRID == kE2M1 ? 6.0f : a.uqmax;
        for (int e = threadIdx.x; e < gt.n; e += blockDim.x) {
            const float A_t = __uint_as_float(slots[e]);
            float se = 1.0f, sd = 1.0f;
            if (A_t > 0.0f) {
                const float num = 448.0f * qmax;
                se = __fdiv_rn(num, A_t);
                if (se > kFltMax) se = kFltMax;
                sd = __fdiv_rn(A_t, num);
            }
            sm.senc[e] = se;
            if (blockIdx.x == 0) {
                a.tensor_scale[e] = sd;
                if (!isfinite(A_t) && a.status) atomicOr(a.status, 1u);
            }
        }
        __syncthreads();
    }
    const uint32_t smask = RHT ? rht_sign_mask(a.rht_seed) : 0u;
    const Signs sg = row_signs<In>(smask);
    const uint32_t total_blocks = (uint32_t)(total_bytes / (16 * sizeof(In)));
    constexpr uint32_t BPC = kChunk / (16 * sizeof(In));
    const uint32_t cstride = (uint32_t)(a.kpad / 2), nkt = (uint32_t)a.nkt;
    int e_cur = -1;
    float m = 0.0f;
    bool ok = true;
    for (; j < nloc; ++j) {
        if (!ring_wait<kRing>(ring, j)) { ok = false; break; }
        const uint32_t i = chunk_of(j);
        const uint32_t st = ring.buf + (j % kRing) * kChunk;
#pragma unroll
        for (uint32_t kk = 0; kk < (BPC + kThreads - 1) / kThreads; ++kk) {
            const uint32_t k = threadIdx.x + kk * kThreads;
            const uint32_t gb = i * BPC + k;
            if (k >= BPC || gb >= total_blocks) continue;
            const uint32_t r = fdiv(gb, bdiv);   // input row
            const bool same = e_cur >= 0 && (int64_t)r >= sm.in_row[e_cur] && (int64_t)r < sm.in_row[e_cur + 1];
            const int e = same ? e_cur : find_seg(sm.in_row, gt.n, (int64_t)r);
            Raw<In> raw;
            raw.load_shared(st + k * 16 * sizeof(In));
            if (AMAX) {
                if (e != e_cur) {
                    seg_max_flush(slots, e_cur, RHT ? m * 0.25f : m);
                    e_cur = e;
                    m = 0.0f;
                }
                float lo[8], hi[8];
                block_values<In, RHT>(raw, sg, lo, hi);
#pragma unroll
                for (int t = 0; t < 8; ++t) m = max3_nan(m, fabsf(lo[t]), fabsf(hi[t]));
            } else {
                e_cur = e;
                const uint32_t orow = (uint32_t)(sm.out_off[e] + ((int64_t)r - sm.in_row[e]));
                quant_block_row<In, GRID, ROUND, RHT>(a, raw, orow, gb - r * kvb, sg, sm.senc[e], nullptr,
                                                      cstride, nkt, false);
            }
        }
        __syncthreads();
        if (threadIdx.x == 0) issue(j + kRing);
    }
    if (!ok) {
        if (threadIdx.x == 0) atomicOr(&g_quant_timeout, 1u);
        ring_drain<kRing>(ring, j, issued);
    }
    if (AMAX) {
        seg_max_flush(slots, e_cur, RHT ? m * 0.25f : m);
    } else {
        const uint32_t nbk = (uint32_t)(a.kpad / 16);
        for (uint32_t ro = blockIdx.x * blockDim.x + threadIdx.x; ro < (uint32_t)a.out_rows;
             ro += gridDim.x * blockDim.x) {
            const int e = find_seg(sm.out_off, gt.n, (int64_t)ro);
            const bool pad_row = (int64_t)ro - sm.out_off[e] >= sm.in_row[e + 1] - sm.in_row[e];
            for (uint32_t b = pad_row ? 0u : kvb; b < nbk; ++b) {
                put_codes(a, (size_t)ro * cstride + b * 8, make_uint2(0u, 0u));
                a.scales[scale_offset32(ro, b, nkt)] = 0;
            }
        }
    }
}

template <bool AMAX, class K, class... P>
cudaError_t launch_staged(K kern, int64_t work_ctas, int *grid_out, cudaStream_t s, P... args);

// The round keys of Philox4x32-10 with key sr_seed (the key advances by the
// Weyl constants 0x9E3779B9 / 0xBB67AE85 after each round).
void set_sr_keys(Args &a) {
    uint32_t k0 = (uint32_t)a.sr_seed, k1 = (uint32_t)(a.sr_seed >> 32);
    for (int r = 0; r < 10; ++r) {
        a.srk[2 * r] = k0;
        a.srk[2 * r + 1] = k1;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
}

Args grouped_args(const QuantLaunch &q, void *ws) {
    Args a{};
    a.x = q.x; a.ld = q.ld; a.cols = q.cols;
    a.out_rows = q.out_rows; a.k = q.k; a.kpad = kpad_of(q.k); a.nkt = a.kpad / 64;
    a.rows = q.colwise ? q.k : q.rows;   // column-wise: the SR row length is the whole k
    a.rht_seed = q.rht_seed; a.sr_seed = q.sr_seed; a.sr_counter = q.sr_counter; a.elem_base = 0;
    set_sr_keys(a);
    a.status = reinterpret_cast<uint32_t *>(static_cast<char *>(ws) + kWsStatus);
    a.codes = q.codes; a.scales = q.scales; a.tensor_scale = q.tensor_scale;
    a.eplane = q.grid == kE1M2 ? q.eplane : nullptr;
    a.uqmax = q.grid == kE2M1C ? 2.0f : 3.5f;
    a.utop = grid_top(q.grid);
    return a;
}

template <class In>
cudaError_t quantize_grouped_typed(const QuantLaunch &q, const GroupQuant &gt, void *ws, cudaStream_t s) {
    Args a = grouped_args(q, ws);
    uint32_t *slots = reinterpret_cast<uint32_t *>(static_cast<char *>(ws) + kWsPartials);
    cudaError_t e = cudaMemsetAsync(ws, 0, kWsPartials + (size_t)gt.n * sizeof(uint32_t), s);
    if (e != cudaSuccess) return e;
    const bool col = q.colwise != 0;
    if (!col && q.ld == q.cols) {
        // contiguous row-wise: both passes stream the tensor through the staged ring
        const uint32_t kvb = (uint32_t)(q.cols / 16);
        const uint64_t tb = (uint64_t)q.rows * (uint64_t)q.cols * sizeof(In);
        const uint32_t nch = (uint32_t)((tb + kChunk - 1) / kChunk);
        const FastDiv bd = make_fastdiv(kvb);
        e = q.rht ? launch_staged<true>(k_row_grouped_staged<In, kE2M1, kRTNE, true, true>, nch, nullptr, s, a, gt,
                                        bd, kvb, nch, tb, slots)
                  : launch_staged<true>(k_row_grouped_staged<In, kE2M1, kRTNE, false, true>, nch, nullptr, s, a,
                                        gt, bd, kvb, nch, tb, slots);
        if (e != cudaSuccess) return e;
        const int kg = q.grid == kE2M1 ? kE2M1 : kE1M2;   // clamped E2M1 runs the uniform-grid kernels
#define UFP4_GR(GRID, ROUND, RHT)                                                                                 if (kg == GRID && q.round == ROUND && (q.rht != 0) == RHT)                                                    return launch_staged<false>(k_row_grouped_staged<In, GRID, ROUND, RHT, false>, nch, nullptr, s, a,                                         gt, bd, kvb, nch, tb, slots);
        UFP4_GR(kE2M1, kRTNE, false) UFP4_GR(kE2M1, kRTNE, true) UFP4_GR(kE2M1, kSR, false) UFP4_GR(kE2M1, kSR, true)
        UFP4_GR(kE1M2, kRTNE, false) UFP4_GR(kE1M2, kRTNE, true) UFP4_GR(kE1M2, kSR, false) UFP4_GR(kE1M2, kSR, true)
#undef UFP4_GR
        return cudaErrorInvalidValue;
    }
    // amax pass: units over real data only
    GroupQuant ga = gt;
    const uint32_t per_row_a = col ? (uint32_t)(q.cols / 2) : (uint32_t)(q.cols / 16);
    for (int i = 0; i < gt.n; ++i) {
        const int64_t T = gt.in_row[i + 1] - gt.in_row[i];
        ga.units[i + 1] = ga.units[i] + (col ? (T + 15) / 16 : T) * per_row_a;
    }
    const int64_t ta = ga.units[gt.n];
    const int sms = num_sms();
    if (ta > 0) {
        const int g = (int)std::min<int64_t>((ta + kThreads - 1) / kThreads, (int64_t)sms * 4);
#define UFP4_GA(COL, RHT) if (col == COL && (q.rht != 0) == RHT) k_amax_grouped<In, RHT, COL><<<g, kThreads, 0, s>>>(a, ga, make_fastdiv(per_row_a), per_row_a, slots);
        UFP4_GA(false, false) UFP4_GA(false, true) UFP4_GA(true, false) UFP4_GA(true, true)
#undef UFP4_GA
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    // quant pass: units include the padding rows / blocks
    const uint32_t per_row = col ? (uint32_t)(q.cols / 2) : (uint32_t)(a.kpad / 16);
    const int64_t tq = gt.units[gt.n];
    const int g = (int)std::min<int64_t>(std::max<int64_t>((tq + kThreads - 1) / kThreads, 1), (int64_t)sms * 8);
    const FastDiv fd = make_fastdiv(per_row);
    const int kgrid = q.grid == kE2M1 ? kE2M1 : kE1M2;   // clamped E2M1 runs the uniform-grid kernels
#define UFP4_GQ(COL, GRID, ROUND, RHT)                                                            \
    if (col == COL && kgrid == GRID && q.round == ROUND && (q.rht != 0) == RHT) {              \
        k_quant_grouped<In, GRID, ROUND, RHT, COL><<<g, kThreads, 0, s>>>(a, gt, fd, per_row, slots); \
        return cudaGetLastError();                                                               \
    }
    UFP4_GQ(false, kE2M1, kRTNE, false) UFP4_GQ(false, kE2M1, kRTNE, true)
    UFP4_GQ(false, kE2M1, kSR, false)   UFP4_GQ(false, kE2M1, kSR, true)
    UFP4_GQ(false, kE1M2, kRTNE, false) UFP4_GQ(false, kE1M2, kRTNE, true)
    UFP4_GQ(false, kE1M2, kSR, false)   UFP4_GQ(false, kE1M2, kSR, true)
    UFP4_GQ(true, kE2M1, kRTNE, false)  UFP4_GQ(true, kE2M1, kRTNE, true)
    UFP4_GQ(true, kE2M1, kSR, false)    UFP4_GQ(true, kE2M1, kSR, true)
    UFP4_GQ(true, kE1M2, kRTNE, false)  UFP4_GQ(true, kE1M2, kRTNE, true)
    UFP4_GQ(true, kE1M2, kSR, false)    UFP4_GQ(true, kE1M2, kSR, true)
#undef UFP4_GQ
    return cudaErrorInvalidValue;
}

// ======================================= grouped, both orientations (BF16)
// The segments of a grouped tensor are cut into segment-aligned 128 x 64
// tiles: segment e's rows are split into ceil(T_e / 128) row tiles starting at
// its first row, so no tile straddles two segments, and tile rows past the
// segment's end are read as zeros (the zero padding of the column-wise
// layout; padding rows of the row-wise layout).  Tiles are numbered segment
// by segment (the GroupDual prefix table) and every CTA takes a contiguous
// run of them through the TMA ring, so it meets few segments and the
// segment lookup is uniform across the CTA.  AMAX: each thread keeps the
// row-wise and column-wise block maxima of its current segment and the CTA's
// warps flush them (atomicMax on the bit patterns) when the segment changes.
// Otherwise both results as k_dual_tile, each block with its segment's
// tensor scales.

// Tensor-scale encode factor S_enc of a segment from its amax slot.
__device__ __forceinline__ float senc_of(uint32_t slot, float qmax) {
    const float A_t = __uint_as_float(slot);
    float se = 1.0f;
    if (A_t > 0.0f) {
        se = __fdiv_rn(448.0f * qmax, A_t);
        if (se > kFltMax) se = kFltMax;
    }
    return se;
}

// One segment-aligned tile at shared address st: `nvalid` of its rows belong
// to the segment, its row-wise output starts at row `orow`, its column-wise
// blocks at k-block `kb0`, of which the first `nkb` (4 or 8) lie in the
// segment's k range.
template <int GRID, int ROUND, bool RHT, bool AMAX>
__device__ __forceinline__ void dual_tile_grouped(const Args &ar, const Args &ac, const DualGeom &g, uint32_t st,
                                                  int nvalid, uint32_t orow, uint32_t kb0, uint32_t nkb, uint32_t ct,
                                                  const Signs &sgr, const Signs &sgc, float Sr, float Sc,
                                                  const float *s_kr, const float *s_kc, bool fr, bool fc,
                                                  uint8_t *stage_codes, uint8_t *stage_scales, float &mr, float &mc) {
    const uint32_t c0 = ct * kTileCols;
    {
        const uint32_t c = c0 + 2 * g.cp;
        const int left = nvalid - 16 * (int)g.rb;   // rows of this unit inside the segment
        ColRaw<__nv_bfloat16> raw;
        const uint32_t sa = st + 16 * g.rb * (kTileCols * 2) + g.cp * 4;
        if (left >= 16) raw.load_shared(sa, kTileCols * 2);   // (warp-uniform branches)
        else if (left > 0) raw.load_shared_rows(sa, kTileCols * 2, left);
        else raw.zero();
        if (AMAX) {
            if (c < g.cols && left > 0) {
                uint64_t P[16];
                col_values<__nv_bfloat16, RHT>(raw, sgc, P);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float a, b;
                    upk2(P[i], a, b);
                    mc = max3_nan(mc, fabsf(a), fabsf(b));
                }
            }
        } else {
            uint2 w0 = make_uint2(0u, 0u), w1 = make_uint2(0u, 0u);
            uint32_t e0 = 0, e1 = 0;
            if (c < g.cols && g.rb < nkb)
                col_unit_words<__nv_bfloat16, GRID, ROUND, RHT>(ac, raw, kb0 + g.rb, c, left > 0, sgc, Sc, s_kc, fc,
                                                                w0, w1, e0, e1);
            reinterpret_cast<uint2 *>(stage_codes)[g.rb * kTileCols + 2 * g.cp] = w0;
            reinterpret_cast<uint2 *>(stage_codes)[g.rb * kTileCols + 2 * g.cp + 1] = w1;
            stage_scales[g.rb * kTileCols + 2 * g.cp] = (uint8_t)e0;
            stage_scales[g.rb * kTileCols + 2 * g.cp + 1] = (uint8_t)e1;
        }
    }
    {
        const uint32_t b = ct * (kTileCols / 16) + g.bc;
        if (b < g.kvr) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = (int)g.q + 64 * h;
                Raw<__nv_bfloat16> ra;
                if (row < nvalid) ra.load_shared(st + (uint32_t)row * (kTileCols * 2) + g.bc * 32);
                else ra.zero();
                if (AMAX) {
                    if (row < nvalid) {
                        float lo[8], hi[8];
                        block_values<__nv_bfloat16, RHT>(ra, sgr, lo, hi);
#pragma unroll
                        for (int j = 0; j < 8; ++j) mr = max3_nan(mr, fabsf(lo[j]), fabsf(hi[j]));
                    }
                } else {
                    // rows past the segment's end are the layout's zero padding rows
                    quant_block_row<__nv_bfloat16, GRID, ROUND, RHT>(ar, ra, orow + (uint32_t)row, b, sgr, Sr,
                                                                     s_kr, g.csr, g.nktr, fr);
                }
            }
        }
    }
}

template <int GRID, int ROUND, bool RHT, bool AMAX>
__global__ void __launch_bounds__(kThreads, kStagedMinCtas)
    k_dual_tile_grouped(const __grid_constant__ CUtensorMap tmx, Args ar, Args ac,
                        const __grid_constant__ GroupDual gd, uint32_t nct, uint32_t *slots) {
    // slots: [0, n) row-wise maxima, [n, 2n) column-wise maxima (fp32 bits)
    constexpr int kRing = ring_depth<false>();
    extern __shared__ __align__(128) uint8_t dsm[];
    __shared__ float s_kr[256], s_kc[256];   // the current segment's per-code multipliers
    const RingCtl ring = ring_init<kRing>(dsm);
    // staging buffer b: codes [rb][cl] uint2, then scales [rb][cl] byte
    uint8_t *const stage0 = dsm + kRing * kChunk + 64;
    const uint32_t total = (uint32_t)gd.tiles[gd.n];
    const uint32_t per = (total + gridDim.x - 1) / gridDim.x;
    const uint32_t t0 = blockIdx.x * per;
    const uint32_t nloc = t0 < total ? min(per, total - t0) : 0u;
    uint32_t issued = 0, j = 0;
    // Position of the CTA's consecutive tiles (segment, row tile, column tile),
    // advanced one tile at a time: a binary search only when a segment ends.
    struct Cursor {
        int e;
        uint32_t rt, ct;
    };
    auto seek = [&](uint32_t i) {
        Cursor c;
        c.e = find_seg(gd.tiles, gd.n, (int64_t)i);
        const uint32_t lt = (uint32_t)(i - gd.tiles[c.e]);
        c.rt = lt / nct;
        c.ct = lt - c.rt * nct;
        return c;
    };
    auto next = [&](Cursor &c, uint32_t i_next) {   // i_next: the tile after c's
        if (i_next >= (uint32_t)gd.tiles[c.e + 1]) {
            if (i_next < total) c = seek(i_next);
            return;
        }
        if (++c.ct == nct) { c.ct = 0; ++c.rt; }
    };
    Cursor icur = seek(t0);   // the issuing thread's, kRing tiles ahead
    auto issue = [&](uint32_t jj) {
        if (jj >= nloc) return;
        const uint32_t bar = ring.bars + 8u * (jj % kRing);
        ptx::mbar_arrive_expect_tx(bar, kTileBytes);   // rows past the tensor arrive as zeros
        ptx::tma_load_2d(ring.buf + (jj % kRing) * kChunk, &tmx, (int32_t)(icur.ct * kTileCols),
                         (int32_t)(gd.in_row[icur.e] + (int64_t)icur.rt * kTileRows), bar);
        issued = jj + 1;
        next(icur, t0 + jj + 1);
    };
    if (threadIdx.x == 0) {
        ptx::prefetch_tmap(&tmx);
        for (uint32_t t = 0; t < kRing; ++t) issue(t);
    }
    const float qmax = GRID == kE2M1 ? 6.0f : ar.uqmax;
    if (!AMAX && blockIdx.x == 0) {
        // every segment's S_dec, and the non-finite flag
        for (int e = threadIdx.x; e < gd.n; e += blockDim.x) {
            const float ar_t = __uint_as_float(slots[e]), ac_t = __uint_as_float(slots[gd.n + e]);
            ar.tensor_scale[e] = ar_t > 0.0f ? __fdiv_rn(ar_t, 448.0f * qmax) : 1.0f;
            ac.tensor_scale[e] = ac_t > 0.0f ? __fdiv_rn(ac_t, 448.0f * qmax) : 1.0f;
            if ((!isfinite(ar_t) || !isfinite(ac_t)) && ar.status) atomicOr(ar.status, 1u);
        }
    }
    const uint32_t smask = RHT ? rht_sign_mask(ar.rht_seed) : 0u;
    const Signs sgr = row_signs<__nv_bfloat16>(smask), sgc = col_signs<__nv_bfloat16>(smask);
    const DualGeom g = dual_geom(ar, ac);
    float mr = 0.0f, mc = 0.0f;
    int e_cur = -1;
    float Sr = 1.0f, Sc = 1.0f;
    bool fr = false, fc = false;
    // a segment's tables k = min(S_enc / E4M3(e), FLT_MAX) x (1/4 with the
    // transform) x (2^-8 where the E1M2 RTNE rounding folds it), as the
    // single-tensor prologue builds them; rebuilt when the CTA's run of tiles
    // enters the next segment (every thread has left the previous tile)
    auto tables = [&](int e) {
        Sr = senc_of(slots[e], qmax);
        Sc = senc_of(slots[gd.n + e], qmax);
        fr = GRID == kE1M2 && ROUND == kRTNE && Sr >= 1.5407439555097887e-33f;
        fc = GRID == kE1M2 && ROUND == kRTNE && Sc >= 1.5407439555097887e-33f;
        const float kf = RHT ? 0.25f : 1.0f;
        for (int c = threadIdx.x; c < 256; c += blockDim.x) {
            const float d = e4m3_to_f32((uint32_t)c);
            float kr = 0.0f, kc = 0.0f;
            if (d > 0.0f) {
                kr = fminf(__fdiv_rn(Sr, d), kFltMax);
                kc = fminf(__fdiv_rn(Sc, d), kFltMax);
            } else if (!(d == 0.0f)) {
                kr = kc = d;   // NaN code: only reachable from non-finite input
            }
            s_kr[c] = kr * (fr ? kf * 0.00390625f : kf);
            s_kc[c] = kc * (fc ? kf * 0.00390625f : kf);
        }
        __syncthreads();
    };
    bool ok = true;
    Cursor cur = seek(t0);
    for (; j < nloc; ++j) {
        const bool mine = ring_wait_own<kRing>(ring, j);
        const uint32_t i = t0 + j;
        const int e = cur.e;
        const uint32_t rt = cur.rt, ct = cur.ct;
        next(cur, i + 1);
        const uint32_t T = (uint32_t)(gd.in_row[e + 1] - gd.in_row[e]);   // rows fit 32 bits (checked on the host)
        const uint32_t left = T - rt * kTileRows;
        const int nvalid = left < kTileRows ? (int)left : (int)kTileRows;
        // column-wise blocks of the segment's k range (kpad(T) / 16, a multiple of 4) in this tile
        const uint32_t kbl = (T + 63) / 64 * 4 - rt * 8;
        const uint32_t nkb = kbl < 8 ? kbl : 8u;
        const uint32_t kb0 = (uint32_t)(gd.koff[e] / 16) + rt * 8;
        // (the tables are read only by the quantization, which every thread
        // finished before the previous tile's barrier)
        if (!AMAX && e != e_cur) tables(e);   // uniform across the CTA
        e_cur = e;
        uint8_t *const stage_codes = stage0 + (j & 1) * kColStageBytes;
        uint8_t *const stage_scales = stage_codes + 8 * kTileCols * 8;
        if (mine)
            dual_tile_grouped<GRID, ROUND, RHT, AMAX>(ar, ac, g, ring.buf + (j % kRing) * kChunk, nvalid,
                                                      (uint32_t)gd.roff[e] + rt * kTileRows, kb0, nkb, ct, sgr, sgc,
                                                      Sr, Sc, s_kr, s_kc, fr, fc, stage_codes, stage_scales, mr, mc);
        // tile j consumed and its column-wise results staged; every thread has
        // also finished flushing tile j - 1, whose buffer tile j + 1 reuses
        __syncthreads();
        if (*ring.abort) { ok = false; break; }
        if (threadIdx.x == 0) issue(j + kRing);
        if (AMAX) {
            // the segment's last tile in this CTA: flush its maxima, one atomic per warp
            if (j + 1 == nloc || cur.e != e) {
#pragma unroll
                for (int o = 16; o; o >>= 1) {
                    mr = max_nan(mr, __shfl_xor_sync(0xffffffffu, mr, o));
                    mc = max_nan(mc, __shfl_xor_sync(0xffffffffu, mc, o));
                }
                if ((threadIdx.x & 31) == 0) {
                    seg_max_flush(slots, e, RHT ? mr * 0.25f : mr);
                    seg_max_flush(slots + gd.n, e, RHT ? mc * 0.25f : mc);
                }
                mr = mc = 0.0f;
            }
        } else {
            // the staged column-wise results: column c, blocks kb0 .. kb0 + nkb - 1
            {
                const uint32_t cl = threadIdx.x / 4, part = threadIdx.x % 4;
                const uint32_t c = ct * kTileCols + cl;
                if (c < g.cols && 2 * part < nkb) {
                    const uint2 a0 = reinterpret_cast<const uint2 *>(stage_codes)[(2 * part) * kTileCols + cl];
                    const uint2 a1 = reinterpret_cast<const uint2 *>(stage_codes)[(2 * part + 1) * kTileCols + cl];
                    put_codes(ac, (size_t)c * g.csc + (size_t)(kb0 + 2 * part) * 8,
                              make_uint4(a0.x, a0.y, a1.x, a1.y));
                }
            }
            if (threadIdx.x < 2 * kTileCols) {
                const uint32_t cl = threadIdx.x / 2, h = threadIdx.x % 2;
                const uint32_t c = ct * kTileCols + cl;
                if (c < g.cols && 4 * h < nkb) {
                    uint32_t w = 0;
#pragma unroll
                    for (int k = 0; k < 4; ++k) w |= (uint32_t)stage_scales[(4 * h + k) * kTileCols + cl] << (8 * k);
                    *reinterpret_cast<uint32_t *>(ac.scales + scale_offset32(c, kb0 + 4 * h, g.nktc)) = w;
                }
            }
        }
    }
    if (!ok) {
        if (threadIdx.x == 0) atomicOr(&g_quant_timeout, 1u);
        ring_drain<kRing>(ring, j, issued);
    }
    if (!AMAX) dual_padding(ar, ac, g);
}

// ============================================================= statistics
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
            const float e = scale_value(grid, a.scales[scale_offset(p.r, p.c >> 1, a.nkt)]);
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
    const uint32_t smask = RHT ? rht_sign_mask(a.rht_seed) : 0u;
    const Signs sg = col_signs<In>(smask);
    const uint32_t ncp = (uint32_t)(a.cols / 2), nkb = (uint32_t)(a.rows / 16);
    const uint32_t total = ncp * nkb, cstride = (uint32_t)(a.kpad / 2), nkt = (uint32_t)a.nkt;
    const In *x = static_cast<const In *>(a.x);
    Acc acc;
    for (uint32_t u = blockIdx.x * blockDim.x + threadIdx.x; u < total; u += gridDim.x * blockDim.x) {
        const uint32_t kb = u / ncp, c = (u - kb * ncp) * 2;
        ColRaw<In> raw;
        raw.load(x + (int64_t)kb * 16 * a.ld + c, a.ld);
        uint64_t P[16];
        col_values<In, RHT>(raw, sg, P);
        float v[2][16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            upk2(P[i], v[0][i], v[1][i]);
            if (RHT) { v[0][i] *= 0.25f; v[1][i] *= 0.25f; }
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const uint2 w = *reinterpret_cast<const uint2 *>(a.codes + (size_t)(c + j) * cstride + kb * 8);
            const float e = scale_value(grid, a.scales[scale_offset32(c + j, kb, nkt)]);
            acc_block8(acc, &v[j][0], w.x, e, S_dec, grid, qmax);
            acc_block8(acc, &v[j][8], w.y, e, S_dec, grid, qmax);
        }
    }
    stats_reduce(acc, a.stats_out);
}

// ================================================================== MXFP4
// The OCP microscaling format MXFP4: blocks of 32 elements along k share one
// E8M0 scale 2^s, s = floor(log2(max |y|)) - 2 (2 = the exponent of E2M1's
// largest normal 6), clamped to [-127, 127] (-127 for an all-zero block);
// elements are E2M1 codes of y * 2^-s (RTNE saturating at 6, or SR).  No
// tensor scale (tensor_scale is written as 1).  The scale byte s + 127 is
// stored at both of the block's 16-block places of the scale layout, so the
// dequantizer and the statistics read it like any block scale.  One thread
// per block; with the transform, each 16-element half is rotated.

// Scale byte s + 127 of a block maximum: the fp32 exponent field minus 2,
// at least 0 (zero or subnormal maxima, and exponents below -125, clamp to
// s = -127).
__device__ __forceinline__ uint32_t mx_scale_byte(float amax) {
    const uint32_t ef = (__float_as_uint(amax) >> 23) & 0xFFu;
    return ef > 2u ? ef - 2u : 0u;
}

template <int ROUND>
__device__ __forceinline__ void mx_store(const Args &a, float v[32], uint32_t r, uint32_t b, uint64_t i0,
                                         uint32_t cstride, uint32_t nkt) {
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 32; j += 2) amax = max3_nan(amax, fabsf(v[j]), fabsf(v[j + 1]));
    if (!(amax <= kFltMax) && a.status) atomicOr(a.status, 1u);
    const uint32_t sb = mx_scale_byte(amax);
    const float f = __uint_as_float((254u - min(sb, 253u)) << 23);   // 2^-s, exact
    uint32_t w[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        float q[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) q[j] = __fmul_rn(v[8 * t + j], f);
        w[t] = codes8<kE2M1, ROUND>(q, a, i0 + 8 * t);
    }
    *reinterpret_cast<uint4 *>(a.codes + (size_t)r * cstride + b * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint16_t *>(a.scales + scale_offset32(r, 2 * b, nkt)) = (uint16_t)(sb | (sb << 8));
}

__device__ __forceinline__ void mx_store_zero(const Args &a, uint32_t r, uint32_t b, uint32_t cstride,
                                              uint32_t nkt) {
    *reinterpret_cast<uint4 *>(a.codes + (size_t)r * cstride + b * 16) = make_uint4(0u, 0u, 0u, 0u);
    *reinterpret_cast<uint16_t *>(a.scales + scale_offset32(r, 2 * b, nkt)) = 0;
}

// Row-wise: unit u = r * (kpad / 32) + b; blocks b >= k / 32 are padding.
template <class In, int ROUND, bool RHT>
__global__ void __launch_bounds__(kThreads) k_quant_mx_row(Args a) {
    const uint32_t nbp = (uint32_t)(a.kpad / 32), nbk = (uint32_t)(a.k / 32);
    const uint32_t cstride = (uint32_t)(a.kpad / 2), nkt = (uint32_t)a.nkt;
    const uint64_t total = (uint64_t)a.out_rows * nbp;
    const uint32_t smask = RHT ? rht_sign_mask(a.rht_seed) : 0u;
    const In *x = static_cast<const In *>(a.x);
    if (blockIdx.x == 0 && threadIdx.x == 0) *a.tensor_scale = 1.0f;
    for (uint64_t u = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; u < total;
         u += (uint64_t)gridDim.x * blockDim.x) {
        const uint32_t r = (uint32_t)(u / nbp), b = (uint32_t)(u - (uint64_t)r * nbp);
        if (b >= nbk) { mx_store_zero(a, r, b, cstride, nkt); continue; }
        float v[32];
        const In *p = x + (int64_t)r * a.ld + (int64_t)b * 32;
#pragma unroll
        for (int t = 0; t < 4; ++t) load8(p + 8 * t, RHT ? (smask >> (8 * (t & 1))) & 0xFFu : 0u, v + 8 * t);
        if (RHT) {
            fwht16(v);
            fwht16(v + 16);
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] *= 0.25f;
        }
        mx_store<ROUND>(a, v, r, b, ((uint64_t)r * a.k + (uint64_t)b * 32), cstride, nkt);
    }
    zero_pad_rows(a);
}

// Column-wise (the quantization of X^T): unit u = b * cols + c, column c of
// the input is output row c, and rows 32b..32b+31 its block b; adjacent
// threads read adjacent columns.
template <class In, int ROUND, bool RHT>
__global__ void __launch_bounds__(kThreads) k_quant_mx_col(Args a) {
    const uint32_t cols = (uint32_t)a.cols;
    const uint32_t nbp = (uint32_t)(a.kpad / 32), nbk = (uint32_t)(a.k / 32);
    const uint32_t cstride = (uint32_t)(a.kpad / 2), nkt = (uint32_t)a.nkt;
    const uint64_t total = (uint64_t)nbp * cols;
    const uint32_t smask = RHT ? rht_sign_mask(a.rht_seed) : 0u;
    const In *x = static_cast<const In *>(a.x);
    if (blockIdx.x == 0 && threadIdx.x == 0) *a.tensor_scale = 1.0f;
    for (uint64_t u = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; u < total;
         u += (uint64_t)gridDim.x * blockDim.x) {
        const uint32_t b = (uint32_t)(u / cols), c = (uint32_t)(u - (uint64_t)b * cols);
        if (b >= nbk) { mx_store_zero(a, c, b, cstride, nkt); continue; }
        float v[32];
        const In *p = x + (int64_t)b * 32 * a.ld + c;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float e = (float)p[(int64_t)i * a.ld];
            v[i] = (RHT && ((smask >> (i & 15)) & 1u)) ? -e : e;
        }
        if (RHT) {
            fwht16(v);
            fwht16(v + 16);
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] *= 0.25f;
        }
        mx_store<ROUND>(a, v, c, b, ((uint64_t)c * a.k + (uint64_t)b * 32), cstride, nkt);
    }
    zero_pad_rows(a);
}

template <class In>
cudaError_t quantize_mx_typed(const QuantLaunch &q, const Args &a, cudaStream_t s) {
    const uint64_t units = (uint64_t)q.out_rows * (uint64_t)(a.kpad / 32);
    const int g = (int)std::min<uint64_t>(std::max<uint64_t>((units + kThreads - 1) / kThreads, 1),
                                          (uint64_t)num_sms() * 8);
#define UFP4_MX(COL, RND, R)                                                                     \
    if (q.colwise == COL && q.round == RND && (q.rht != 0) == R) {                               \
        if (COL) k_quant_mx_col<In, RND, R><<<g, kThreads, 0, s>>>(a);                           \
        else k_quant_mx_row<In, RND, R><<<g, kThreads, 0, s>>>(a);                               \
        return cudaGetLastError();                                                               \
    }
    UFP4_MX(0, kRTNE, false) UFP4_MX(0, kRTNE, true) UFP4_MX(0, kSR, false) UFP4_MX(0, kSR, true)
    UFP4_MX(1, kRTNE, false) UFP4_MX(1, kRTNE, true) UFP4_MX(1, kSR, false) UFP4_MX(1, kSR, true)
#undef UFP4_MX
    return cudaErrorInvalidValue;
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
            const float e = scale_value(grid, scales[scale_offset(p.r, p.c >> 1, nkt)]);
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
// Launch of a staged kernel: opt in to the ring's dynamic shared memory once
// per kernel, persistent grid of the CTAs that fit at once.
template <class K, class... P>
cudaError_t launch_staged_smem(K kern, size_t smem, int64_t work_ctas, int *grid_out, cudaStream_t s, P... args) {
    static std::mutex mu;
    static std::vector<const void *> done;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (std::find(done.begin(), done.end(), (const void *)kern) == done.end()) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            done.push_back((const void *)kern);
        }
    }
    const int g = resident_grid(kern, work_ctas, smem);
    if (grid_out) *grid_out = g;
    kern<<<g, kThreads, smem, s>>>(args...);
    return cudaGetLastError();
}
template <bool AMAX, class K, class... P>
cudaError_t launch_staged(K kern, int64_t work_ctas, int *grid_out, cudaStream_t s, P... args) {
    return launch_staged_smem(kern, ring_smem<AMAX>(), work_ctas, grid_out, s, args...);
}

template <class In, int GRID, int ROUND, bool RHT>
cudaError_t quant_pass(const QuantLaunch &q, const Args &a, bool staged, cudaStream_t s) {
    const bool col = q.colwise != 0;
    if (!col) {
        if (staged) {
            const uint32_t kvb = (uint32_t)(a.k / 16);
            const uint64_t tb = (uint64_t)a.rows * a.cols * sizeof(In);
            const uint32_t nch = (uint32_t)((tb + kChunk - 1) / kChunk);
            return launch_staged<false>(k_row_staged<In, GRID, ROUND, RHT, false>, nch, nullptr, s, a,
                                 make_fastdiv(kvb), kvb, nch, tb);
        }
        const uint32_t bpr = (uint32_t)(a.kpad / 16), total = (uint32_t)(a.out_rows * bpr);
        auto kern = k_quant_rowwise<In, GRID, ROUND, RHT>;
        kern<<<resident_grid(kern, (total + 2 * kThreads - 1) / (2 * kThreads)), kThreads, 0, s>>>(
            a, make_fastdiv(bpr), bpr, total);
        return cudaGetLastError();
    }
    if (staged) {
        constexpr uint32_t CW = kChunk / (16 * sizeof(In));
        const uint32_t ncc = (uint32_t)((a.cols + CW - 1) / CW), nch = (uint32_t)(a.rows / 16) * ncc;
        return launch_staged<false>(k_col_staged<In, GRID, ROUND, RHT, false>, nch, nullptr, s, a, ncc, nch);
    }
    const uint32_t ncp = (uint32_t)(a.cols / 2), ctotal = (uint32_t)((a.kpad / 16) * ncp);
    auto kern = k_quant_colwise<In, GRID, ROUND, RHT>;
    kern<<<resident_grid(kern, (ctotal + kThreads - 1) / kThreads), kThreads, 0, s>>>(a, make_fastdiv(ncp), ncp,
                                                                                        ctotal);
    return cudaGetLastError();
}

template <class In, bool RHT>
cudaError_t amax_pass(const QuantLaunch &q, Args &a, bool staged, cudaStream_t s) {
    const bool col = q.colwise != 0;
    int g = 1;
    cudaError_t e;
    if constexpr (std::is_same<In, __nv_bfloat16>::value && RHT) {
        // BF16 with the transform: the tensor-core amax (rows as 16-byte pieces)
        if ((a.cols * 2) % 16 == 0) {
            const uint32_t ncc = (uint32_t)((a.cols + kMmaCW - 1) / kMmaCW);
            const uint32_t nch = (uint32_t)((a.rows + 15) / 16) * ncc;
            e = col ? launch_staged_smem(k_amax_mma<false, true>, kMmaSmem, nch, &g, s, a, a, ncc, nch)
                    : launch_staged_smem(k_amax_mma<true, false>, kMmaSmem, nch, &g, s, a, a, ncc, nch);
            a.n_partials = g;
            return e;
        }
    }
    if (!col) {
        if (staged) {
            const uint64_t tb = (uint64_t)a.rows * a.cols * sizeof(In);
            const uint32_t nch = (uint32_t)((tb + kChunk - 1) / kChunk);
            e = launch_staged<true>(k_row_staged<In, 0, 0, RHT, true>, nch, &g, s, a, FastDiv{0, 0}, 0u, nch, tb);
        } else {
            const uint32_t bpr = (uint32_t)(a.k / 16), total = (uint32_t)(a.out_rows * bpr);
            auto kern = k_amax_rowwise<In, RHT>;
            g = resident_grid(kern, (total + 2 * kThreads - 1) / (2 * kThreads));
            kern<<<g, kThreads, 0, s>>>(a, make_fastdiv(bpr), bpr, total);
            e = cudaGetLastError();
        }
    } else {
        if (staged) {
            constexpr uint32_t CW = kChunk / (16 * sizeof(In));
            const uint32_t ncc = (uint32_t)((a.cols + CW - 1) / CW), nch = (uint32_t)(a.rows / 16) * ncc;
            e = launch_staged<true>(k_col_staged<In, 0, 0, RHT, true>, nch, &g, s, a, ncc, nch);
        } else {
            const uint32_t ncp = (uint32_t)(a.cols / 2), total = (uint32_t)((a.rows / 16) * ncp);
            auto kern = k_amax_colwise<In, RHT>;
            g = resident_grid(kern, (total + kThreads - 1) / kThreads);
            kern<<<g, kThreads, 0, s>>>(a, make_fastdiv(ncp), ncp, total);
            e = cudaGetLastError();
        }
    }
    a.n_partials = g;
    return e;
}

template <class In>
cudaError_t quantize_typed(const QuantLaunch &q, Args &a, void *ws, cudaStream_t s) {
    const bool col = q.colwise != 0;
    // The bulk-copy path needs 16-byte pieces: the whole (contiguous) tensor
    // row-wise, each row segment column-wise.
    const bool staged = col ? ((a.cols * (int64_t)sizeof(In)) % 16 == 0) : (a.ld == a.cols);
    if (!q.amax_in) {
        a.partials_out = reinterpret_cast<float *>(static_cast<char *>(ws) + kWsPartials);
        a.partials = a.partials_out;
        cudaError_t e = q.rht ? amax_pass<In, true>(q, a, staged, s) : amax_pass<In, false>(q, a, staged, s);
        if (e != cudaSuccess) return e;
    }
    const int kgrid = q.grid == kE2M1 ? kE2M1 : kE1M2;   // clamped E2M1 runs the uniform-grid kernels
#define UFP4_Q(GRID, ROUND, RHT)                                                   \
    if (kgrid == GRID && q.round == ROUND && (q.rht != 0) == RHT)                  \
        return quant_pass<In, GRID, ROUND, RHT>(q, a, staged, s);
    UFP4_Q(kE2M1, kRTNE, false) UFP4_Q(kE2M1, kRTNE, true)
    UFP4_Q(kE2M1, kSR, false)   UFP4_Q(kE2M1, kSR, true)
    UFP4_Q(kE1M2, kRTNE, false) UFP4_Q(kE1M2, kRTNE, true)
    UFP4_Q(kE1M2, kSR, false)   UFP4_Q(kE1M2, kSR, true)
#undef UFP4_Q
    return cudaErrorInvalidValue;
}

// Cooperative launch of a single-pass kernel over `grid` CTAs of
// kResidentThreads with kResidentSmem bytes of shared memory, after zeroing
// its grid-barrier counter.  cudaErrorNotSupported when the CTAs cannot all
// be resident.
template <class K, class... P>
cudaError_t launch_resident(K kern, uint32_t grid, uint32_t *arrive, cudaStream_t s, P... args) {
    static std::mutex mu;
    static std::vector<const void *> done;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (std::find(done.begin(), done.end(), (const void *)kern) == done.end()) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kResidentSmem);
            if (e != cudaSuccess) return e;
            done.push_back((const void *)kern);
        }
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kResidentThreads, kResidentSmem) != cudaSuccess ||
        (int64_t)per_sm * num_sms() < (int64_t)grid)
        return cudaErrorNotSupported;
    cudaError_t e = cudaMemsetAsync(arrive, 0, sizeof(uint32_t), s);
    if (e != cudaSuccess) return e;
    void *argv[] = {static_cast<void *>(&args)...};
    e = cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(kern), dim3(grid), dim3(kResidentThreads), argv,
                                    kResidentSmem, s);
    if (e == cudaErrorCooperativeLaunchTooLarge) {
        cudaGetLastError();   // not sticky: take the two-pass route
        return cudaErrorNotSupported;
    }
    return e;
}

// Both orientations of one tensor from one read per pass (k_dual_staged).
// The row-wise and column-wise partial maxima take the two halves of the
// workspace's partial area.
template <class In>
cudaError_t quantize_dual_typed(const QuantLaunch &qr, const QuantLaunch &qc, Args &ar, Args &ac, void *ws,
                                cudaStream_t s) {
    if constexpr (std::is_same<In, __nv_bfloat16>::value) {
        // BF16: 128 x 64 tiles by TMA (k_dual_tile)
        alignas(64) CUtensorMap tm;
        if (!make_input_tile_map(&tm, ar.x, ar.rows, ar.cols, ar.ld, kTileCols, kTileRows))
            return cudaErrorInvalidValue;
        const uint32_t nct = (uint32_t)((ar.cols + kTileCols - 1) / kTileCols);
        const uint32_t ntiles = (uint32_t)((ar.rows + kTileRows - 1) / kTileRows) * nct;
        ac.status = nullptr;   // the row-wise prologue reports both
        if (!qr.amax_in && !qc.amax_in) {
            // small enough to stay in shared memory: one cooperative single pass
            const int sms = num_sms();
            const uint32_t grid = (uint32_t)std::min<int64_t>(sms, ntiles);
            if ((ntiles + grid - 1) / grid <= kResidentMax) {
                ar.partials_out = reinterpret_cast<float *>(static_cast<char *>(ws) + kWsPartials);
                ac.partials_out = ar.partials_out + kMaxPartials / 2;
                ar.partials = ar.partials_out;
                ac.partials = ac.partials_out;
                ar.n_partials = ac.n_partials = (int)grid;
                uint32_t *arrive = reinterpret_cast<uint32_t *>(static_cast<char *>(ws) + kWsArrive);
                const int kgrid = qr.grid == kE2M1 ? kE2M1 : kE1M2;
#define UFP4_R(GRID, ROUND, RHT)                                                                         \
                if (kgrid == GRID && qr.round == ROUND && (qr.rht != 0) == RHT) {                        \
                    cudaError_t e = launch_resident(k_dual_resident<GRID, ROUND, RHT>, grid, arrive, s, tm, \
                                                    ar, ac, nct, ntiles, arrive);                          \
                    if (e != cudaErrorNotSupported) return e;                                             \
                }
                UFP4_R(kE2M1, kRTNE, false) UFP4_R(kE2M1, kRTNE, true)
                UFP4_R(kE2M1, kSR, false)   UFP4_R(kE2M1, kSR, true)
                UFP4_R(kE1M2, kRTNE, false) UFP4_R(kE1M2, kRTNE, true)
                UFP4_R(kE1M2, kSR, false)   UFP4_R(kE1M2, kSR, true)
#undef UFP4_R
                // (not co-resident on this device: the two-pass route below)
            }
        }
        if (!qr.amax_in || !qc.amax_in) {
            // the amax pass streams with little arithmetic: 16-row x 1 KB
            // chunks (contiguous kilobyte rows) read faster than 128-byte
            // tile rows, and the maxima do not depend on the traversal
            constexpr uint32_t CW = kChunk / 32;
            const uint32_t ncc = (uint32_t)((ar.cols + CW - 1) / CW), nch = (uint32_t)(ar.rows / 16) * ncc;
            ar.partials_out = reinterpret_cast<float *>(static_cast<char *>(ws) + kWsPartials);
            ac.partials_out = ar.partials_out + kMaxPartials / 2;
            int g = 1;
            cudaError_t e;
            if (qr.rht) {
                // the tensor-core amax of both orientations (CW = kMmaCW: same chunking)
                static_assert(CW == kMmaCW, "chunk widths");
                auto kern = k_amax_mma<true, true>;
                if (resident_grid(kern, nch, kMmaSmem) > kMaxPartials / 2) return cudaErrorInvalidValue;
                e = launch_staged_smem(kern, kMmaSmem, nch, &g, s, ar, ac, ncc, nch);
            } else {
                auto kern = k_dual_staged<In, 0, 0, false, true>;
                if (resident_grid(kern, nch, ring_smem<true>()) > kMaxPartials / 2) return cudaErrorInvalidValue;
                e = launch_staged<true>(kern, nch, &g, s, ar, ac, ncc, nch);
            }
            if (e != cudaSuccess) return e;
            ar.partials = ar.partials_out;
            ac.partials = ac.partials_out;
            ar.n_partials = ac.n_partials = g;
        }
        const int kgrid = qr.grid == kE2M1 ? kE2M1 : kE1M2;   // clamped E2M1 runs the uniform-grid kernels
#define UFP4_T(GRID, ROUND, RHT)                                                                          \
        if (kgrid == GRID && qr.round == ROUND && (qr.rht != 0) == RHT)                                   \
            return launch_staged_smem(k_dual_tile<GRID, ROUND, RHT>, dual_smem<kDualRing>(), ntiles, nullptr, s,  \
                                      tm, ar, ac, nct, ntiles);
        UFP4_T(kE2M1, kRTNE, false) UFP4_T(kE2M1, kRTNE, true)
        UFP4_T(kE2M1, kSR, false)   UFP4_T(kE2M1, kSR, true)
        UFP4_T(kE1M2, kRTNE, false) UFP4_T(kE1M2, kRTNE, true)
        UFP4_T(kE1M2, kSR, false)   UFP4_T(kE1M2, kSR, true)
#undef UFP4_T
        return cudaErrorInvalidValue;
    } else {
    constexpr uint32_t CW = kChunk / (16 * sizeof(In));
    const uint32_t ncc = (uint32_t)((ar.cols + CW - 1) / CW), nch = (uint32_t)(ar.rows / 16) * ncc;
    ac.status = nullptr;   // the row-wise prologue reports both
    if (!qr.amax_in || !qc.amax_in) {
        ar.partials_out = reinterpret_cast<float *>(static_cast<char *>(ws) + kWsPartials);
        ac.partials_out = ar.partials_out + kMaxPartials / 2;
        auto kern = qr.rht ? k_dual_staged<In, 0, 0, true, true> : k_dual_staged<In, 0, 0, false, true>;
        if (resident_grid(kern, nch, ring_smem<true>()) > kMaxPartials / 2) return cudaErrorInvalidValue;
        int g = 1;
        cudaError_t e = launch_staged<true>(kern, nch, &g, s, ar, ac, ncc, nch);
        if (e != cudaSuccess) return e;
        ar.partials = ar.partials_out;
        ac.partials = ac.partials_out;
        ar.n_partials = ac.n_partials = g;
    }
    const int kgrid = qr.grid == kE2M1 ? kE2M1 : kE1M2;   // clamped E2M1 runs the uniform-grid kernels
#define UFP4_D(GRID, ROUND, RHT)                                                                         \
    if (kgrid == GRID && qr.round == ROUND && (qr.rht != 0) == RHT)                                      \
        return launch_staged<false>(k_dual_staged<In, GRID, ROUND, RHT, false>, nch, nullptr, s, ar, ac, ncc, nch);
    UFP4_D(kE2M1, kRTNE, false) UFP4_D(kE2M1, kRTNE, true)
    UFP4_D(kE2M1, kSR, false)   UFP4_D(kE2M1, kSR, true)
    UFP4_D(kE1M2, kRTNE, false) UFP4_D(kE1M2, kRTNE, true)
    UFP4_D(kE1M2, kSR, false)   UFP4_D(kE1M2, kSR, true)
#undef UFP4_D
    return cudaErrorInvalidValue;
    }
}

Args make_args(const QuantLaunch &q, void *ws) {
    Args a{};
    a.x = q.x;
    a.rows = q.rows; a.cols = q.cols; a.ld = q.ld;
    a.out_rows = q.out_rows; a.k = q.k; a.kpad = kpad_of(q.k); a.nkt = a.kpad / 64;
    a.rht_seed = q.rht_seed; a.sr_seed = q.sr_seed; a.sr_counter = q.sr_counter;
    set_sr_keys(a);
    a.elem_base = q.elem_base;
    a.amax_in = q.amax_in;
    a.status = ws ? reinterpret_cast<uint32_t *>(static_cast<char *>(ws) + kWsStatus) : nullptr;
    a.codes = q.codes; a.scales = q.scales; a.tensor_scale = q.tensor_scale;
    a.eplane = q.grid == kE1M2 ? q.eplane : nullptr;
    a.uqmax = q.grid == kE2M1C ? 2.0f : 3.5f;
    a.utop = grid_top(q.grid);
    return a;
}

// Both orientations of a grouped BF16 tensor: the amax pass and the
// quantization pass of k_dual_tile_grouped, one read of x each.
cudaError_t quantize_grouped_dual_bf16(const QuantLaunch &qr, const QuantLaunch &qc, const GroupDual &gd, void *ws,
                                       cudaStream_t s) {
    Args ar = grouped_args(qr, ws), ac = grouped_args(qc, ws);
    ac.status = nullptr;   // the row-wise side reports both
    alignas(64) CUtensorMap tm;
    if (!make_input_tile_map(&tm, qr.x, qr.rows, qr.cols, qr.ld, kTileCols, kTileRows)) return cudaErrorInvalidValue;
    const uint32_t nct = (uint32_t)((qr.cols + kTileCols - 1) / kTileCols);
    const int64_t ntiles = gd.tiles[gd.n];
    uint32_t *slots = reinterpret_cast<uint32_t *>(static_cast<char *>(ws) + kWsPartials);
    cudaError_t e = cudaMemsetAsync(ws, 0, kWsPartials + 2 * (size_t)gd.n * sizeof(uint32_t), s);
    if (e != cudaSuccess || ntiles == 0) return e;
    constexpr uint32_t smem = dual_smem<ring_depth<false>()>();
    e = qr.rht ? launch_staged_smem(k_dual_tile_grouped<kE2M1, kRTNE, true, true>, smem, ntiles, nullptr, s, tm, ar,
                                    ac, gd, nct, slots)
               : launch_staged_smem(k_dual_tile_grouped<kE2M1, kRTNE, false, true>, smem, ntiles, nullptr, s, tm, ar,
                                    ac, gd, nct, slots);
    if (e != cudaSuccess) return e;
    const int kgrid = qr.grid == kE2M1 ? kE2M1 : kE1M2;   // clamped E2M1 runs the uniform-grid kernels
#define UFP4_GD(GRID, ROUND, RHT)                                                                             \
    if (kgrid == GRID && qr.round == ROUND && (qr.rht != 0) == RHT)                                          \
        return launch_staged_smem(k_dual_tile_grouped<GRID, ROUND, RHT, false>, smem, ntiles, nullptr, s, tm, ar, ac,  \
                                  gd, nct, slots);
    UFP4_GD(kE2M1, kRTNE, false) UFP4_GD(kE2M1, kRTNE, true)
    UFP4_GD(kE2M1, kSR, false)   UFP4_GD(kE2M1, kSR, true)
    UFP4_GD(kE1M2, kRTNE, false) UFP4_GD(kE1M2, kRTNE, true)
    UFP4_GD(kE1M2, kSR, false)   UFP4_GD(kE1M2, kSR, true)
#undef UFP4_GD
    return cudaErrorInvalidValue;
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

cudaError_t read_quant_timeout_flag(uint32_t *flag, cudaStream_t s) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(flag, g_quant_timeout, sizeof(uint32_t), 0,
                                              cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess && *flag) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbolAsync(g_quant_timeout, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    }
    return e;
}

cudaError_t launch_quantize(const QuantLaunch &q, void *ws, cudaStream_t s) {
    Args a = make_args(q, ws);
    if (q.grid == kMXFP4) {
        // status word only (no tensor amax): clear it like the other passes do
        if (a.status) {
            cudaError_t e = cudaMemsetAsync(a.status, 0, sizeof(uint32_t), s);
            if (e != cudaSuccess) return e;
        }
        return q.dtype == 0 ? quantize_mx_typed<__nv_bfloat16>(q, a, s) : quantize_mx_typed<float>(q, a, s);
    }
    if (q.dtype == 0) return quantize_typed<__nv_bfloat16>(q, a, ws, s);
    return quantize_typed<float>(q, a, ws, s);
}

cudaError_t launch_quantize_stats(const QuantLaunch &q, void *ws, int *n_ctas, cudaStream_t s) {
    const int64_t esz = q.dtype == 0 ? 2 : 4;
    *n_ctas = 0;
    // one pass: the staged row-wise quantization (contiguous input), whose
    // CTAs fit the workspace's partial sums
    if (q.grid != kMXFP4 && !q.colwise && q.ld == q.cols) {
        Args a = make_args(q, ws);
        a.stats_out = reinterpret_cast<double *>(static_cast<char *>(ws) + kWsStats);
        if (!q.amax_in) {
            a.partials_out = reinterpret_cast<float *>(static_cast<char *>(ws) + kWsPartials);
            a.partials = a.partials_out;
            cudaError_t e = q.rht ? (esz == 2 ? amax_pass<__nv_bfloat16, true>(q, a, true, s)
                                              : amax_pass<float, true>(q, a, true, s))
                                  : (esz == 2 ? amax_pass<__nv_bfloat16, false>(q, a, true, s)
                                              : amax_pass<float, false>(q, a, true, s));
            if (e != cudaSuccess) return e;
        }
        const uint32_t kvb = (uint32_t)(a.k / 16);
        const uint64_t tb = (uint64_t)a.rows * a.cols * esz;
        const uint32_t nch = (uint32_t)((tb + kChunk - 1) / kChunk);
        const int kgrid = q.grid == kE2M1 ? kE2M1 : kE1M2;
#define UFP4_QS(IN, GRID, ROUND, RHT)                                                                        \
        if ((esz == sizeof(IN)) && kgrid == GRID && q.round == ROUND && (q.rht != 0) == RHT) {              \
            auto kern = k_row_staged<IN, GRID, ROUND, RHT, false, true>;                                     \
            if (resident_grid(kern, nch, ring_smem<false>()) <= kMaxStatsCtas)                               \
                return launch_staged<false>(kern, nch, n_ctas, s, a, make_fastdiv(kvb), kvb, nch, tb);      \
        }
        UFP4_QS(__nv_bfloat16, kE2M1, kRTNE, false) UFP4_QS(__nv_bfloat16, kE2M1, kRTNE, true)
        UFP4_QS(__nv_bfloat16, kE2M1, kSR, false)   UFP4_QS(__nv_bfloat16, kE2M1, kSR, true)
        UFP4_QS(__nv_bfloat16, kE1M2, kRTNE, false) UFP4_QS(__nv_bfloat16, kE1M2, kRTNE, true)
        UFP4_QS(__nv_bfloat16, kE1M2, kSR, false)   UFP4_QS(__nv_bfloat16, kE1M2, kSR, true)
        UFP4_QS(float, kE2M1, kRTNE, false) UFP4_QS(float, kE2M1, kRTNE, true)
        UFP4_QS(float, kE2M1, kSR, false)   UFP4_QS(float, kE2M1, kSR, true)
        UFP4_QS(float, kE1M2, kRTNE, false) UFP4_QS(float, kE1M2, kRTNE, true)
        UFP4_QS(float, kE1M2, kSR, false)   UFP4_QS(float, kE1M2, kSR, true)
#undef UFP4_QS
        // (the amax pass, if any, has run: the two-pass route below repeats it)
    }
    // two passes: quantization, then the statistics kernels
    cudaError_t e = launch_quantize(q, ws, s);
    if (e != cudaSuccess) return e;
    return launch_stats(q, ws, n_ctas, s);
}

cudaError_t launch_quantize_dual(const QuantLaunch &qr, const QuantLaunch &qc, void *ws, cudaStream_t s) {
    const int64_t esz = qr.dtype == 0 ? 2 : 4;
    const bool same = qr.grid == qc.grid && qr.round == qc.round && qr.rht == qc.rht &&
                      (!qr.rht || qr.rht_seed == qc.rht_seed);
    // one read serves both when every 16-row chunk row is a whole number of
    // 16-byte pieces; otherwise two ordinary quantizations
    if (!same || (qr.cols * esz) % 16 != 0 || qr.rows % 16 != 0) {
        cudaError_t e = launch_quantize(qr, ws, s);
        return e != cudaSuccess ? e : launch_quantize(qc, ws, s);
    }
    Args ar = make_args(qr, ws), ac = make_args(qc, ws);
    if (qr.dtype == 0) return quantize_dual_typed<__nv_bfloat16>(qr, qc, ar, ac, ws, s);
    return quantize_dual_typed<float>(qr, qc, ar, ac, ws, s);
}

cudaError_t launch_quantize_grouped(const QuantLaunch &q, const GroupQuant &gt, void *ws, cudaStream_t s) {
    if (q.dtype == 0) return quantize_grouped_typed<__nv_bfloat16>(q, gt, ws, s);
    return quantize_grouped_typed<float>(q, gt, ws, s);
}

cudaError_t launch_quantize_grouped_dual(const QuantLaunch &qr, const QuantLaunch &qc, const GroupDual &gd,
                                         void *ws, cudaStream_t s) {
    if (qr.dtype != 0) return cudaErrorInvalidValue;
    return quantize_grouped_dual_bf16(qr, qc, gd, ws, s);
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
    else work = ((a.cols / 2) * (a.rows / 16) + kThreads - 1) / kThreads;
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

#ifdef UFP4_PROBE
#include "probe_entry.inc"
#endif
