// nvfp4_device.cuh -- device primitives of the sm_103a NVFP4 quantizer.
//
// Every rounding the method pins is spelled out here so no compiler lowering
// can change a bit ("Add NVFP4 four-over-six (row-wise) quantization to the
// training prototype", CuTe DSL kernel (SM100), Design):
//   - fp32 multiply / add / divide with explicit round-to-nearest intrinsics
//     (no contraction into FMA; the build also passes -fmad=false);
//   - E4M3 scale encode with cvt.rn.satfinite.e4m3x2.f32, exact decode with
//     cvt.rn.f16x2.e4m3x2;
//   - e2m1 encode with cvt.rn.satfinite.e2m1x2.f32 (NaN -> +6), exact decode
//     with cvt.rn.f16x2.e2m1x2;
//   - NaN-dropping fmaxf / fminf for amaxes and the 448 caps.
#pragma once

#include <cstdint>
#include <cfloat>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include "nvfp4_params.h"

namespace nvfp4 {

// ---- pinned fp32 arithmetic --------------------------------------------------------------
__device__ __forceinline__ float mul_rn(float a, float b) { return __fmul_rn(a, b); }
__device__ __forceinline__ float add_rn(float a, float b) { return __fadd_rn(a, b); }
__device__ __forceinline__ float sub_rn(float a, float b) { return __fsub_rn(a, b); }
__device__ __forceinline__ float div_rn(float a, float b) { return __fdiv_rn(a, b); }
__device__ __forceinline__ float max_nd(float a, float b) { return fmaxf(a, b); }
__device__ __forceinline__ float min_nd(float a, float b) { return fminf(a, b); }
// NaN-dropping maximum of two pairs of bf16 magnitudes: max.bf16x2 (no .NaN)
// returns the other operand where one is NaN, and keeps subnormals; the
// maximum is one of its inputs, so it is exact.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t acc, uint32_t w) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(acc), "r"(w & 0x7FFF7FFFu));
    return r;
}

// ---- E4M3 block scales -----------------------------------------------------------------
// RN-even to E4M3FN with saturation to +-448 (NaN stays NaN).
__device__ __forceinline__ uint32_t e4m3_encode(float s) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(s));
    return r & 0xFFu;
}

// Two scales in one conversion: the bytes of sa and sb.
__device__ __forceinline__ void e4m3_encode2(float sa, float sb, uint32_t& a, uint32_t& b) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(sb), "f"(sa));
    a = r & 0xFFu;
    b = static_cast<uint32_t>(r) >> 8;
}

// The exact values of two E4M3 bytes in one conversion.
__device__ __forceinline__ void e4m3_decode2(uint32_t a, uint32_t b, float& da, float& db) {
    uint32_t h2;
    const uint16_t in = static_cast<uint16_t>((a & 0xFFu) | ((b & 0xFFu) << 8));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
    da = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
    db = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16)));
}

// Exact value of an E4M3 byte (every E4M3 value is an fp16 normal or zero).
__device__ __forceinline__ float e4m3_decode(uint32_t b) {
    uint32_t h2;
    const uint16_t in = static_cast<uint16_t>(b & 0xFFu);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
}

// ---- e2m1 elements -----------------------------------------------------------------------
// Eight values -> eight 4-bit codes, element i in nibble i (element 2j in the
// low nibble of byte j).
__device__ __forceinline__ uint32_t e2m1_encode8(const float* v) {
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(r)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return r;
}

// One code byte (two 4-bit codes) -> an f16 pair of grid values, low nibble in
// the low half.  The byte is taken with an explicit cvt.u8.u32 of the shifted
// word: decoding straight from a four-byte vector unpack of the word was
// observed to read zeros for some byte positions.
__device__ __forceinline__ uint32_t e2m1_decode_byte(uint32_t w, int byte) {
    uint32_t h;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
        : "=r"(h)
        : "r"(w >> (8 * byte)));
    return h;
}

// Eight 4-bit codes -> their exact signed grid values.
__device__ __forceinline__ void e2m1_decode8(uint32_t w, float* q) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t h = e2m1_decode_byte(w, i);
        q[2 * i] = __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xFFFFu)));
        q[2 * i + 1] = __half2float(__ushort_as_half(static_cast<unsigned short>(h >> 16)));
    }
}

// ---- counter-based generator: Philox4x32-10 (Salmon et al., SC'11) -------------------
__device__ __forceinline__ uint64_t mul_wide_u32(uint32_t a, uint32_t b) {
    uint64_t p;
    asm("mul.wide.u32 %0, %1, %2;" : "=l"(p) : "r"(a), "r"(b));
    return p;
}

// Words for global element indices idx0 .. idx0+15 (idx0 a multiple of 16):
// element idx uses word idx % 4 of the block with counter (idx / 4, step).
// Round r: (x, y, z, w) <- (hi(M1 z) ^ y ^ k0[r], lo(M1 z), hi(M0 x) ^ w ^ k1[r],
// lo(M0 x)); round 0's step terms and the round keys come from pk.
__device__ __forceinline__ void sr_words16(uint64_t idx0, const PhiloxKeys& pk, uint32_t* w) {
    const uint64_t b0 = idx0 >> 2;                         // a multiple of 4
    const uint32_t hi = static_cast<uint32_t>(b0 >> 32);   // shared by the four counters
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint64_t p = mul_wide_u32(kPhiloxM0, static_cast<uint32_t>(b0) + j);
        uint4 c = make_uint4(pk.r0x ^ hi, pk.r0y, static_cast<uint32_t>(p >> 32) ^ pk.r0z, static_cast<uint32_t>(p));
#pragma unroll
        for (int r = 1; r < 10; ++r) {
            const uint64_t p0 = mul_wide_u32(kPhiloxM0, c.x);
            const uint64_t p1 = mul_wide_u32(kPhiloxM1, c.z);
            c = make_uint4(static_cast<uint32_t>(p1 >> 32) ^ c.y ^ pk.k0[r], static_cast<uint32_t>(p1),
                           static_cast<uint32_t>(p0 >> 32) ^ c.w ^ pk.k1[r], static_cast<uint32_t>(p0));
        }
        w[4 * j + 0] = c.x;
        w[4 * j + 1] = c.y;
        w[4 * j + 2] = c.z;
        w[4 * j + 3] = c.w;
    }
}

// ---- packed pairs of fp32 (one instruction, two IEEE round-to-nearest results) ----
__device__ __forceinline__ uint64_t pack2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void unpack2(uint64_t r, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// Stochastic rounding of one magnitude a = |v| to a grid value ("fp4-train",
// Method): with G[k] <= a < G[k+1], take G[k+1] when u < p, p = (a - G[k]) /
// (G[k+1] - G[k]), u = (word >> 8) * 2^-24.  The grid spacing is 0.5 on
// [0,2), 1 on [2,4) and 2 on [4,6]: sp = 2^(max(E,0) - 1) for a's binary
// exponent E.  Its reciprocal's bits are min(~bits(a) & 0x7F800000, bits(2)):
// the complemented exponent field is 0x7F800000 minus the field.  t = a / sp
// is exact and lies in [0,4); with fl = floor(t) and p = t - fl, the rounded
// index fl + [u < p] equals ceil(t - u) (t - u lies in (fl, fl+1) when u < p,
// in (fl-1, fl] otherwise), and ceil(RU(t - u)) = ceil(t - u) because
// rounding upward never passes the integer above, so one fused multiply-add
// rounded upward, t - (word >> 8) * 2^-24, and a ceiling give the index.  a >= 6,
// infinity and NaN give 6 (the NaN-dropping min after clamping a); the
// caller restores the sign (a zero result may come out as -0).
__device__ __forceinline__ uint32_t sr_inv_bits(float a) {
    return min(~__float_as_uint(a) & 0x7F800000u, 0x40000000u);
}

__device__ __forceinline__ float sr_grid_value(float a, uint32_t word) {
    a = min_nd(a, 6.0f);
    const uint32_t ib = sr_inv_bits(a);
    const float t = mul_rn(a, __uint_as_float(ib));
    const float k = ceilf(__fmaf_ru(static_cast<float>(word >> 8), -5.9604644775390625e-08f, t));
    return mul_rn(k, __uint_as_float(0x7F000000u - ib));
}

__device__ __forceinline__ uint64_t fma2_ru(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rp.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// sr_grid_value on two magnitudes at once (same arithmetic, paired fp32 ops)
__device__ __forceinline__ void sr_grid_value2(float a0, float a1, uint32_t w0, uint32_t w1, float& g0, float& g1) {
    a0 = min_nd(a0, 6.0f);
    a1 = min_nd(a1, 6.0f);
    const uint32_t i0 = sr_inv_bits(a0), i1 = sr_inv_bits(a1);
    const uint64_t T = mul2(pack2(a0, a1), pack2(__uint_as_float(i0), __uint_as_float(i1)));
    const uint64_t U = pack2(static_cast<float>(w0 >> 8), static_cast<float>(w1 >> 8));
    float k0, k1;
    unpack2(fma2_ru(U, pack2(-5.9604644775390625e-08f, -5.9604644775390625e-08f), T), k0, k1);
    const uint64_t SP = pack2(__uint_as_float(0x7F000000u - i0), __uint_as_float(0x7F000000u - i1));
    unpack2(mul2(pack2(ceilf(k0), ceilf(k1)), SP), g0, g1);
}

// ---- exact division from a reciprocal ---------------------------------------------------
// RN(a / b) given r = RN(1 / b): q0 = a*r, then two correction steps
// q <- q + (a - b*q) * r with fused multiply-adds (P. Markstein, IBM J. R&D 34(1),
// 1990; Muller et al., Handbook of Floating-Point Arithmetic, ch. 4).  The first
// step makes q faithful, so the second remainder is exact and the second step
// returns the correctly rounded quotient.  Valid while b, a / b and the
// remainders stay normal (the callers' guards keep them so), with the sign of
// a restored on a zero result.  Checked against IEEE
// division exhaustively over the mantissas of every E4M3 divisor.
__device__ __forceinline__ float div_by_recip(float a, float b, float r) {
    float q = mul_rn(a, r);
    float e = __fmaf_rn(-q, b, a);
    q = __fmaf_rn(e, r, q);
    e = __fmaf_rn(-q, b, a);
    return __fmaf_rn(e, r, q);
}

// RN(a / b) given r = RN(1 / b) with ONE correction step.  Exact when b's
// significand is one of the eight E4M3 significands 1 + k/8 (checked
// exhaustively over every fp32 significand of a, both quotient binades), under
// the same range conditions as div_by_recip.
__device__ __forceinline__ float div_by_recip1(float a, float b, float r) {
    const float q = mul_rn(a, r);
    const float e = __fmaf_rn(-q, b, a);
    return __fmaf_rn(e, r, q);
}

// RN(|a| / b) and the sign of a / b: the two-step (or, for E4M3 divisors,
// one-step) sequence on a signed a gives the exact magnitude, while its first
// product a * r carries the quotient's sign also for a = -0 (where the
// correction's sum would be +0) and is a positive NaN for NaN a.
__device__ __forceinline__ float sign_of_first(float q0, float mag) {
    return __uint_as_float((__float_as_uint(mag) & 0x7FFFFFFFu) | (__float_as_uint(q0) & 0x80000000u));
}


// RN(b / 6) for a block amax b >= 0 (6 = 1.5 * 4 has an E4M3 significand, so
// one correction step is exact while b is in range).
__device__ __forceinline__ float div6(float b) {
    if (b >= 7.8886090522101181e-31f && b < 8.5070591730234616e+37f)   // [2^-100, 2^126)
        return div_by_recip1(b, 6.0f, 0.16666667163372040f);             // RN(1/6)
    return div_rn(b, 6.0f);
}

// ---- global scales ("Add NVFP4 four-over-six ...", What) ------------------------------
// S_enc = min(6*bound / A, FLT_MAX), 1 when A is not a positive finite number;
// S_dec = 1 / S_enc.
__device__ __forceinline__ void global_scales(float A, float bound, float& enc, float& dec) {
    if (!(A > 0.0f) || isinf(A)) enc = 1.0f;
    else enc = min_nd(div_rn(mul_rn(6.0f, bound), A), FLT_MAX);
    dec = div_rn(1.0f, enc);
}

// ---- four-over-six candidate data ----------------------------------------------------------
// For one candidate scale byte sf (decoded d): the encode reciprocal
// enc = min(1/(d*S_dec), FLT_MAX) and the error values of the grid points.
// The error value of code q is ((q*d)*A)/C with C = 6*bound.  q*d is exact and
// q = 2^e * m with m in {1, 1.5}, e in -1..2, so while RN(m*d*A) stays normal
// far from the range ends, ((q*d)*A)/C = 2^e * X_m exactly, with
// X_1 = RN(RN(d*A)/C) and X_1.5 = RN(RN(1.5*d*A)/C).  `fast` records whether
// that holds (also for zero, infinite or NaN products, where the scaling is
// exact as well); when it does not, the error value is computed literally.
struct Cand {
    float enc, X1, DX;      // DX = X_1.5 - X_1, exact (Sterbenz: X_1.5 ~ 1.5 X_1)
    uint32_t fast;
};

__device__ __forceinline__ bool scalable(float Y) {
    const float a = fabsf(Y);
    return a == 0.0f || (a >= 7.8886090522101181e-31f && a <= 1.2676506002282294e+30f);
}

__device__ __forceinline__ Cand make_cand(uint32_t sf, float Sdec, float A, float C) {
    const float d = e4m3_decode(sf);
    Cand c;
    c.enc = min_nd(div_rn(1.0f, mul_rn(d, Sdec)), FLT_MAX);
    const float Y1 = mul_rn(d, A);
    const float Y15 = mul_rn(mul_rn(1.5f, d), A);
    c.X1 = div_rn(Y1, C);
    c.DX = sub_rn(div_rn(Y15, C), c.X1);
    c.fast = (scalable(Y1) && scalable(Y15)) ? 1u : 0u;
    return c;
}

// q - v for the two halves of an f16 pair q (a code pair's grid values) and
// two fp32 values v, each rounded once to fp32: the mixed-precision subtract
// takes its f16 operand exactly (no separate conversion).
__device__ __forceinline__ void sub_f16x2_f32(uint32_t q, float v0, float v1, float& d0, float& d1) {
    asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "sub.rn.f32.f16 %0, lo, %3;\n\tsub.rn.f32.f16 %1, hi, %4;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "r"(q), "f"(v0), "f"(v1));
}

// Eight values -> eight 4-bit codes (as e2m1_encode8) AND the codes' grid
// values as four f16 pairs, each byte decoded straight from the register the
// encode wrote.
__device__ __forceinline__ uint32_t e2m1_encode8_dec(const float* v, uint32_t* h) {
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %8, %7;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %10, %9;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %12, %11;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %4, b3;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(r), "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return r;
}

// Four values -> four 4-bit codes (the low 16 bits, element i in nibble i)
// and the codes' grid values as two f16 pairs, as e2m1_encode8_dec.
__device__ __forceinline__ uint32_t e2m1_encode4_dec(const float* v, uint32_t* h) {
    uint16_t r;
    asm("{\n\t.reg .b8 b0, b1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %6, %5;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b1;\n\t"
        "mov.b16 %0, {b0, b1};\n\t}"
        : "=h"(r), "=r"(h[0]), "=r"(h[1])
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]));
    return r;
}

// Error values of 8 codes given as f16 pairs of grid values (q = 2^e * m):
// dq = p * X_m with p = q without its 1.5 bit and X_m = X_1 + s * DX, s = 1
// for m = 1.5 (exact: X_1 + DX = X_1.5).  s is built from the 1.5 bit by an
// integer multiply (bit 9 * 0x1FC000 = the bits of 1.0f; the other half's
// bit 25 overflows out), so the selection needs no compare or select.
__device__ __forceinline__ void error_values8(const uint32_t* h, float X1, float DX, float* dq) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t sb = h[i] & 0x02000200u;           // the 1.5 bits of both halves
        const uint32_t pw = h[i] ^ sb;                    // p values
        const float plo = __half2float(__ushort_as_half(static_cast<unsigned short>(pw & 0xFFFFu)));
        const float phi = __half2float(__ushort_as_half(static_cast<unsigned short>(pw >> 16)));
        const float slo = __uint_as_float(sb * 0x1FC000u);
        const float shi = __uint_as_float(__umulhi(sb, 0x10000u) * 0x1FC000u);
        dq[2 * i] = mul_rn(plo, __fmaf_rn(slo, DX, X1));
        dq[2 * i + 1] = mul_rn(phi, __fmaf_rn(shi, DX, X1));
    }
}

// ---- 16x16 nibble transpose -----------------------------------------------------------------
// An 8x8 matrix of 4-bit codes, row r in w[r] (column c in nibble c), is
// transposed in place by swapping 4x4, 2x2 and 1x1 blocks (masked xor swaps).
__device__ __forceinline__ void transpose8x8_nibbles(uint32_t* w) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {               // 4x4 blocks: 16-bit fields
        const uint32_t t = ((w[r] >> 16) ^ w[r + 4]) & 0x0000FFFFu;
        w[r + 4] ^= t;
        w[r] ^= t << 16;
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {               // 2x2 blocks: 8-bit fields
        if (r & 2) continue;
        const uint32_t t = ((w[r] >> 8) ^ w[r + 2]) & 0x00FF00FFu;
        w[r + 2] ^= t;
        w[r] ^= t << 8;
    }
#pragma unroll
    for (int r = 0; r < 8; r += 2) {            // 1x1 blocks: 4-bit fields
        const uint32_t t = ((w[r] >> 4) ^ w[r + 1]) & 0x0F0F0F0Fu;
        w[r + 1] ^= t;
        w[r] ^= t << 4;
    }
}

// ---- asynchronous global -> shared copies (per thread) --------------------------------------
// Each thread copies its own 16-byte pieces and waits only for its own groups
// (cp.async.wait_group), so a per-thread multi-stage pipeline needs neither a
// barrier nor a spin-wait.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---- programmatic dependent launch -------------------------------------------------------------
// Every kernel is launched with programmatic stream serialization allowed
// (launch_pdl): it may start while the previous kernel in the stream is
// finishing, so its launch and its input-independent set-up (shared tables
// that need no input, barrier initialisation) overlap that kernel's last
// CTAs.  pdl_wait() blocks until the previous kernel has completed and its
// memory is visible; a kernel calls it before its first global-memory access.
// pdl_trigger() lets the next kernel launch; a kernel calls it once its CTA
// has no work left.  Launched without the attribute, both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---- loads and stores ----------------------------------------------------------------------
template <int DT>
__device__ __forceinline__ void load16(const void* base, int64_t elem0, float* y) {
    if (DT == NVFP4_BF16) {
        const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + elem0);
        const uint4 a = __ldg(p), b = __ldg(p + 1);
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            y[2 * i] = __uint_as_float(w[i] << 16);
            y[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    } else {
        const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + elem0);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 f = __ldg(p + i);
            y[4 * i] = f.x;
            y[4 * i + 1] = f.y;
            y[4 * i + 2] = f.z;
            y[4 * i + 3] = f.w;
        }
    }
}

// A thread's slot of P 16-byte pieces (P = 2 or 4) in a per-thread copy ring,
// with piece c stored at position c ^ swz: each 32-byte sector keeps its two
// pieces together (so the copies fill whole sectors), while a quarter warp's
// 16-byte reads of one piece fall into eight distinct 16-byte bank groups.
template <int P>
__device__ __forceinline__ uint32_t piece_swizzle(int tid) {
    return static_cast<uint32_t>(tid >> (P == 2 ? 2 : 1)) & (P - 1);
}

// 16 elements from a swizzled slot (piece c of the group at c ^ swz)
template <int DT>
__device__ __forceinline__ void lds16_swz(const unsigned char* slot, uint32_t swz, float* y) {
    if (DT == NVFP4_BF16) {
        const uint4 a = *reinterpret_cast<const uint4*>(slot + ((0 ^ swz) << 4));
        const uint4 b = *reinterpret_cast<const uint4*>(slot + ((1 ^ swz) << 4));
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            y[2 * i] = __uint_as_float(w[i] << 16);
            y[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 f = *reinterpret_cast<const float4*>(slot + ((i ^ swz) << 4));
            y[4 * i] = f.x;
            y[4 * i + 1] = f.y;
            y[4 * i + 2] = f.z;
            y[4 * i + 3] = f.w;
        }
    }
}

// 16 elements from shared memory (the layout load16 reads from global memory)
template <int DT>
__device__ __forceinline__ void lds16(const void* p, float* y) {
    if (DT == NVFP4_BF16) {
        const uint4 a = reinterpret_cast<const uint4*>(p)[0], b = reinterpret_cast<const uint4*>(p)[1];
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            y[2 * i] = __uint_as_float(w[i] << 16);
            y[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 f = reinterpret_cast<const float4*>(p)[i];
            y[4 * i] = f.x;
            y[4 * i + 1] = f.y;
            y[4 * i + 2] = f.z;
            y[4 * i + 3] = f.w;
        }
    }
}

__device__ __forceinline__ void load16_f32(const float* base, int64_t elem0, float* r) {
    const float4* p = reinterpret_cast<const float4*>(base + elem0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 f = p[i];
        r[4 * i] = f.x;
        r[4 * i + 1] = f.y;
        r[4 * i + 2] = f.z;
        r[4 * i + 3] = f.w;
    }
}

__device__ __forceinline__ void store16_f32(float* base, int64_t elem0, const float* r) {
    float4* p = reinterpret_cast<float4*>(base + elem0);
#pragma unroll
    for (int i = 0; i < 4; ++i) p[i] = make_float4(r[4 * i], r[4 * i + 1], r[4 * i + 2], r[4 * i + 3]);
}

__device__ __forceinline__ void store16_bf16(uint16_t* base, int64_t elem0, const float* v) {
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(v[2 * i]));
        const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(v[2 * i + 1]));
        w[i] = lo | (hi << 16);
    }
    uint4* p = reinterpret_cast<uint4*>(base + elem0);
    p[0] = make_uint4(w[0], w[1], w[2], w[3]);
    p[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

}  // namespace nvfp4
