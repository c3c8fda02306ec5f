// common.cuh -- device helpers shared by the libufp4 kernels (sm_103a).
//
// Method sources: the pages on arXiv:2606.20381 ("Rethinking Shrinkage Bias
// in LLM FP4 Pretraining"), cited as [ZC] zhichai.net post, [AN]
// autonainews.com article, [HP] hotpaper.ai card.  Formats and layouts that
// the pages leave open follow the contract stated in include/ufp4.h.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace ufp4 {

constexpr int kE2M1 = 0;
constexpr int kE1M2 = 1;
// E2M1 restricted to its uniform part {0, .5, 1, 1.5, 2} (codes 0..4): the
// clamped-E2M1 ablation.  It quantizes through the uniform-grid (E1M2)
// kernels with qmax 2 and top index 4; its codes are E2M1 codes.
constexpr int kE2M1C = 2;
// MXFP4 (OCP microscaling): E2M1 elements, one E8M0 scale 2^s per 32
// elements (stored at both of its 16-blocks' places), no tensor scale.
constexpr int kMXFP4 = 3;
constexpr int kRTNE = 0;
constexpr int kSR = 1;
constexpr float kFltMax = 3.402823466e38f;

__host__ __device__ __forceinline__ float grid_qmax(int grid) {
    return (grid == kE2M1 || grid == kMXFP4) ? 6.0f : (grid == kE1M2 ? 3.5f : 2.0f);
}
// Largest magnitude index of the grid.
__host__ __device__ __forceinline__ uint32_t grid_top(int grid) { return grid == kE2M1C ? 4u : 7u; }

__host__ __device__ __forceinline__ int64_t kpad_of(int64_t k) { return (k + 63) / 64 * 64; }
__host__ __device__ __forceinline__ int64_t rpad_of(int64_t r) { return (r + 127) / 128 * 128; }

// Byte offset of block scale (row r, 16-block b) in the tensor-core scale
// layout: 512-byte atoms of 128 rows x 4 blocks, atoms ordered (row tile,
// block group); inside an atom row r sits at (r%32)*16 + ((r%128)/32)*4.
__host__ __device__ __forceinline__ int64_t scale_offset(int64_t r, int64_t b, int64_t nkt) {
    return (((r >> 7) * nkt + (b >> 2)) << 9) + ((r & 31) << 4) + (((r >> 5) & 3) << 2) + (b & 3);
}

// ---------------------------------------------------------------- Philox
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of the 4x32
// S-box with multipliers 0xD2511F53 / 0xCD9E8D57 and key increments
// 0x9E3779B9 / 0xBB67AE85.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
        const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
        k.x += 0x9E3779B9u;
        k.y += 0xBB67AE85u;
    }
    return c;
}

// The same generator with its ten round keys given (rk[2r], rk[2r + 1] for
// round r: the key after r increments), e.g. precomputed on the host.
__device__ __forceinline__ uint4 philox4x32_10_keys(uint4 c, const uint32_t (&rk)[20]) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
        const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(hi1 ^ c.y ^ rk[2 * r], lo1, hi0 ^ c.w ^ rk[2 * r + 1], lo0);
    }
    return c;
}

// RHT sign pattern d as a 16-bit mask (bit j set <=> d_j = -1): bits 0..15
// of word 0 of Philox4x32-10(key = seed, counter = 0).
__device__ __forceinline__ uint32_t rht_sign_mask(uint64_t seed) {
    const uint4 w = philox4x32_10(make_uint4(0u, 0u, 0u, 0u),
                                  make_uint2((uint32_t)seed, (uint32_t)(seed >> 32)));
    return w.x & 0xFFFFu;
}

// ------------------------------------------------------------- E4M3 codec
// fp32 -> E4M3, round to nearest even, saturating to +-448 (hardware cvt).
__device__ __forceinline__ uint32_t e4m3_from_f32(float v) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
    return r & 0xFFu;
}

// E4M3 -> fp32 (exact; via the hardware f16 path).
__device__ __forceinline__ float e4m3_to_f32(uint32_t c) {
    uint32_t h2;
    const uint16_t in = (uint16_t)(c & 0xFFu);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// E8M0 -> fp32: 2^(b - 127) (b = 0 is 2^-127, a subnormal; 255, NaN, is
// never written).
__device__ __forceinline__ float e8m0_to_f32(uint32_t b) {
    b &= 0xFFu;
    return b ? __uint_as_float(b << 23) : __uint_as_float(0x00400000u);
}

// Value of a stored block-scale byte: E8M0 for MXFP4, E4M3 otherwise.
__device__ __forceinline__ float scale_value(int grid, uint32_t c) {
    return grid == kMXFP4 ? e8m0_to_f32(c) : e4m3_to_f32(c);
}

// --------------------------------------------------------------- bf16 bits
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// NaN-propagating max of magnitudes.
__device__ __forceinline__ float max_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}
// max_nan(a, max_nan(b, c)) in one instruction (the same value: NaN if any
// input is NaN, else the exact maximum, in any order).
__device__ __forceinline__ float max3_nan(float a, float b, float c) {
    float r;
    asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// ------------------------------------------------------------- grid codes
// E2M1 round-to-nearest-even of a pair, satfinite; first argument goes to
// the LOW nibble of the returned byte.
__device__ __forceinline__ uint32_t e2m1x2_rn(float lo, float hi) {
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
        "cvt.u32.u8 %0, t;\n\t}"
        : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// E1M2 round-to-nearest-even of q (grid units): m = rint(min(2|q|, 7)); 2|q|
// is exact (or +inf, which clamps to 7).  Adding 2^23 rounds a value in
// [0, 8) to an integer with ties to even, leaving it in the low mantissa bits.
__device__ __forceinline__ uint32_t e1m2_rn(float q, float top = 7.0f) {
    const float a2 = fminf(fabsf(q) * 2.0f, top);
    const uint32_t m = __float_as_uint(__fadd_rn(a2, 8388608.0f)) & 7u;
    return m | ((__float_as_uint(q) >> 28) & 8u);
}

// Stochastic rounding of q (in grid units) with 16 random bits r (< 2^16):
// floor to the grid point below |q| (clamped to qmax), then up with
// probability p = (a - lo) / (hi - lo) against u = r * 2^-16.  Returns the code.
template <int GRID>
__device__ __forceinline__ uint32_t sr_code(float q, uint32_t r, uint32_t top = 7u) {
    // The decision "up iff r 2^-16 < p", p the position of |q| between its
    // grid neighbours, is taken in fixed point: with t = |q| scaled so that
    // the neighbours are consecutive integers, T = ceil(t 2^16) holds the
    // lower neighbour's index in its top bits and ceil(p 2^16) in its low 16
    // (a p above 1 - 2^-16 carries into the index: always up), and
    // r < ceil(p 2^16) iff r < T mod 2^16.  Exact: t 2^16 is an fp32 value
    // below 2^19 and the conversion rounds up; one conversion per element.
    const uint32_t sgn = (__float_as_uint(q) >> 28) & 8u;
    if (GRID == kE1M2) {
        const float t = fminf(fabsf(q) * 131072.0f, (float)(top << 16));   // 2|q| 2^16, at most top 2^16
        const uint32_t T = __float2uint_ru(t);
        // the same decision as an addition: T + (2^16 - 1 - r) carries into
        // bit 16 iff r < T mod 2^16 (T < 2^19, so nothing overflows)
        return sgn | ((T + 0xFFFFu - r) >> 16);
    } else {
        const float a = fabsf(q);
        if (!(a < 6.0f)) return sgn | 7u;   // also NaN (non-finite input)
        // neighbours 0.5 apart below 2, 1 apart below 4, 2 apart above: ip
        // counts the steps, and the lower neighbour's E2M1 index is ip,
        // ip + 2, ip + 4
        const float mul = a < 2.0f ? 131072.0f : (a < 4.0f ? 65536.0f : 32768.0f);
        const uint32_t T = __float2uint_ru(a * mul);
        const uint32_t base = (T >> 16) + (a < 2.0f ? 0u : (a < 4.0f ? 2u : 4u));
        return sgn | (base + (r < (T & 0xFFFFu) ? 1u : 0u));
    }
}

// sr_code<kE1M2> of q given as qs = q 2^17 (the caller's packed multiply;
// exact: a power-of-two factor, and an overflow to inf clamps the same).
__device__ __forceinline__ uint32_t sr_code_e1m2_scaled(float qs, uint32_t r, uint32_t top) {
    const uint32_t sgn = (__float_as_uint(qs) >> 28) & 8u;
    const uint32_t T = __float2uint_ru(fminf(fabsf(qs), (float)(top << 16)));
    return sgn | ((T + 0xFFFFu - r) >> 16);
}

// Grid value of a magnitude index.
// E2M1: 0, .5, 1, 1.5, 2, 3, 4, 6;  E1M2: m / 2.
__device__ __forceinline__ float grid_value(int grid, uint32_t m) {
    m &= 7u;
    if (grid == kE1M2 || m < 4u) return 0.5f * (float)m;
    return m == 7u ? 6.0f : (float)(m - 2u);
}

// E1M2 as two E2M1 planes: the value m/2 of an E1M2 code equals (R + E)/2,
// R the code's nibble read as an E2M1 code ({0,.5,1,1.5,2,3,4,6}[m]) and E
// the correction plane {0,.5,1,1.5,2,2,2,1}[m] as E2M1 codes, sign kept.
// E plane of 8 packed nibbles s|b2 b1 b0 (m = 4 b2 + 2 b1 + b0): E2M1 code m
// for m < 4, 4 (value 2) for m in {4,5,6}, 2 (value 1) for m = 7.  Per
// nibble the E code is the input masked by: bit 0 kept iff !b2, bit 1 iff
// (!b2 | b0), bit 2 iff !(b0 & b1), bit 3 (sign) always -- the shifted
// copies line the other bits up with each position.
__device__ __forceinline__ uint32_t e1m2_eplane(uint32_t w) {
    const uint32_t u = w >> 1, v = w << 1, t = w >> 2, x = w << 2;
    const uint32_t keep = (~t & 0x11111111u) | ((~u | v) & 0x22222222u) | (~(x & v) & 0x44444444u) | 0x88888888u;
    return w & keep;
}

// ---------------------------------------------------------- in-register FWHT
// Unnormalised 8-point Walsh-Hadamard butterflies (Sylvester order):
// v_i <- sum_j (-1)^popcount(i&j) v_j.
__device__ __forceinline__ void fwht8(float v[8]) {
#pragma unroll
    for (int s = 1; s < 8; s <<= 1) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if ((i & s) == 0) {
                const float a = v[i], b = v[i + s];
                v[i] = a + b;
                v[i + s] = a - b;
            }
        }
    }
}

__device__ __forceinline__ void fwht16(float v[16]) {
#pragma unroll
    for (int s = 1; s < 16; s <<= 1) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if ((i & s) == 0) {
                const float a = v[i], b = v[i + s];
                v[i] = a + b;
                v[i + s] = a - b;
            }
        }
    }
}

}  // namespace ufp4
