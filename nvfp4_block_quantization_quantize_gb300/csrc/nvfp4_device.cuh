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

// ---- E4M3 block scales -----------------------------------------------------------------
// RN-even to E4M3FN with saturation to +-448 (NaN stays NaN).
__device__ __forceinline__ uint32_t e4m3_encode(float s) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(s));
    return r & 0xFFu;
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

// Eight 4-bit codes -> their exact signed grid values.
__device__ __forceinline__ void e2m1_decode8(uint32_t w, float* q) {
    uint32_t h0, h1, h2, h3;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
        : "r"(w));
    const uint32_t h[4] = {h0, h1, h2, h3};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        q[2 * i] = __half2float(__ushort_as_half(static_cast<unsigned short>(h[i] & 0xFFFFu)));
        q[2 * i + 1] = __half2float(__ushort_as_half(static_cast<unsigned short>(h[i] >> 16)));
    }
}

// ---- counter-based generator: Philox4x32-10 (Salmon et al., SC'11) -------------------
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
        const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
        const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    }
    return c;
}

// Words for global element indices idx0 .. idx0+15 (idx0 a multiple of 16):
// element idx uses word idx % 4 of the block with counter (idx / 4, step).
__device__ __forceinline__ void sr_words16(uint64_t idx0, uint64_t seed, uint64_t step,
                                           uint32_t* w) {
    const uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
    const uint32_t s0 = static_cast<uint32_t>(step), s1 = static_cast<uint32_t>(step >> 32);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint64_t blk = (idx0 >> 2) + j;
        const uint4 o = philox4x32_10(
            make_uint4(static_cast<uint32_t>(blk), static_cast<uint32_t>(blk >> 32), s0, s1), k0, k1);
        w[4 * j + 0] = o.x;
        w[4 * j + 1] = o.y;
        w[4 * j + 2] = o.z;
        w[4 * j + 3] = o.w;
    }
}

// Stochastic rounding of one value to a 4-bit code ("fp4-train", Method): with
// G[k] <= |v| < G[k+1], pick k+1 when u < p, p = (|v| - G[k]) / (G[k+1] - G[k])
// (exact: Sterbenz subtraction, power-of-two gap), u = (word >> 8) * 2^-24.
__device__ __forceinline__ uint32_t e2m1_encode_sr(float v, uint32_t word) {
    if (v != v) return 7u;                              // NaN -> +6
    const float a = fabsf(v);
    const uint32_t sign = (__float_as_uint(v) >> 31) << 3;
    if (a >= 6.0f) return sign | 7u;
    const uint32_t k = (a >= 0.5f) + (a >= 1.0f) + (a >= 1.5f) + (a >= 2.0f) + (a >= 3.0f) +
                       (a >= 4.0f);
    const float lo = (k < 4) ? 0.5f * static_cast<float>(k) : static_cast<float>(k - 2);
    const float inv_gap = (k < 4) ? 2.0f : ((k < 6) ? 1.0f : 0.5f);
    const float p = mul_rn(sub_rn(a, lo), inv_gap);
    const float u = mul_rn(static_cast<float>(word >> 8), 5.9604644775390625e-08f);  // 2^-24
    return sign | (k + (u < p ? 1u : 0u));
}

// ---- global scales ("Add NVFP4 four-over-six ...", What) ------------------------------
// S_enc = min(6*bound / A, FLT_MAX), 1 when A is not a positive finite number;
// S_dec = 1 / S_enc.
__device__ __forceinline__ void global_scales(float A, float bound, float& enc, float& dec) {
    if (!(A > 0.0f) || isinf(A)) enc = 1.0f;
    else enc = min_nd(div_rn(mul_rn(6.0f, bound), A), FLT_MAX);
    dec = div_rn(1.0f, enc);
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
