// nvfp4_block.cuh -- quantization of one 16-value group, shared by the kernels.
//
// Method: "fp4-train" (Method: block_absmax/6 scale in e4m3, division by the
// decoded scale, e2m1 grid, stochastic rounding, error feedback) and "Add NVFP4
// four-over-six (row-wise) quantization to the training prototype" (What;
// CuTe DSL kernel (SM100), Design: the (b/6)*S_enc association, the 1.5x
// map-to-4 scale, encode reciprocals, the 6*bound error denominator,
// element-order error sums, the width-16 tree, strict err4 < err6).
#pragma once

#include <type_traits>

#include "nvfp4_device.cuh"

namespace nvfp4 {

constexpr unsigned kFullMask = 0xFFFFFFFFu;

// Global scale of one tensor or row.
struct GScale {
    float A, Senc, Sdec;
};

// Block scale s6f = (b / 6) * S_enc.  Without a global scale S_enc = 1 and the
// product is the identity.
template <bool GS>
__device__ __forceinline__ float block_s6f(float b, float Senc) {
    const float s = div6(b);
    return GS ? mul_rn(s, Senc) : s;
}

// Width-16 tree over a half warp's 16 lanes, broadcast to all of them:
// (((e0+e8)+(e4+e12))+((e2+e10)+(e6+e14))) + (((e1+e9)+(e5+e13))+((e3+e11)+(e7+e15))).
// The xor butterfly forms exactly these pairs (commuted on some lanes).
__device__ __forceinline__ float tree16_lanes(float E) {
    E = add_rn(E, __shfl_xor_sync(kFullMask, E, 8));
    E = add_rn(E, __shfl_xor_sync(kFullMask, E, 4));
    E = add_rn(E, __shfl_xor_sync(kFullMask, E, 2));
    E = add_rn(E, __shfl_xor_sync(kFullMask, E, 1));
    return E;
}

// The same tree over 16 values held by one thread.
__device__ __forceinline__ float tree16_regs(const float* e) {
    return add_rn(add_rn(add_rn(add_rn(e[0], e[8]), add_rn(e[4], e[12])),
                         add_rn(add_rn(e[2], e[10]), add_rn(e[6], e[14]))),
                  add_rn(add_rn(add_rn(e[1], e[9]), add_rn(e[5], e[13])),
                         add_rn(add_rn(e[3], e[11]), add_rn(e[7], e[15]))));
}

__device__ __forceinline__ float max16_lanes(float m) {
    m = max_nd(m, __shfl_xor_sync(kFullMask, m, 8));
    m = max_nd(m, __shfl_xor_sync(kFullMask, m, 4));
    m = max_nd(m, __shfl_xor_sync(kFullMask, m, 2));
    m = max_nd(m, __shfl_xor_sync(kFullMask, m, 1));
    return m;
}

__device__ __forceinline__ float absmax16(const float* y) {
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) m = max_nd(m, fabsf(y[i]));
    return m;
}

// ---- plain path ---------------------------------------------------------------------------
// The plain path's division y / D.  2^-20 <= D <= 2^20 and |y| <= b <= 2^60
// keep quotients and remainders normal for |y| >= 2^-80, so the reciprocal
// sequence is exact there; below that the quotient is under 2^-60 and its
// nearest code is the signed zero either way, while stochastic rounding (EXACT)
// takes the IEEE division.  Outside the range: IEEE division throughout.
__device__ __forceinline__ bool plain_fast(float D, float b) {
    return D >= 9.5367431640625e-07f && D <= 1048576.0f && b <= 1.152921504606847e+18f;
}

// RN(y / D) from r = RN(1/D) up to the sign of a zero result; q0 = y * r
// (the sign source).  One correction step is exact when D is a decoded E4M3
// scale (E4), two in general.
template <bool E4>
__device__ __forceinline__ float recip_quotient(float y, float D, float r, float& q0) {
    q0 = mul_rn(y, r);
    float e = __fmaf_rn(-q0, D, y);
    float q = __fmaf_rn(e, r, q0);
    if (!E4) {
        e = __fmaf_rn(-q, D, y);
        q = __fmaf_rn(e, r, q);
    }
    return q;
}

// One signed quotient RN(y / D), as plain_quotients16 computes it per element.
template <bool EXACT, bool E4 = false>
__device__ __forceinline__ float plain_quotient(float y, float D, float r, bool fast) {
    if (!fast) {
        const float q = div_rn(y, D);
        return q == q ? q : fabsf(q);
    }
    float q0;
    float q = recip_quotient<E4>(y, D, r, q0);
    if (EXACT && fabsf(y) < 8.271806125530277e-25f) q = div_rn(y, D);
    return sign_of_first(q0, q);
}

// RN(1/d) for every non-negative E4M3 byte (entry 0 unused: a zero scale
// zeroes the block), filled once per CTA.
__device__ __forceinline__ void fill_recip_table(float* rt) {
    for (int i = threadIdx.x; i < 128; i += blockDim.x) rt[i] = div_rn(1.0f, e4m3_decode(static_cast<uint32_t>(i)));
    __syncthreads();
}

// The nearest path's quotients outside the reciprocal sequence's range: IEEE
// divisions, out of line (the blocks that need them are rare, and the fast
// path is inlined many times in the tile kernels).
static __device__ __noinline__ void plain_quotients16_ieee(const float* y, float D, float* v) {
    for (int i = 0; i < 16; ++i) v[i] = plain_quotient<false>(y[i], D, 0.0f, false);
}

// codes of y / D (D = decoded scale * S_dec), nearest or stochastic; a zero
// divisor zeroes the block.  b is the block amax (bounds |y|).  rt: the
// reciprocal table when D is a bare E4M3 scale sf (no global scale), else
// null.  With wq, stochastic rounding also returns the codes' signed grid
// values in q (nearest rounding leaves q alone).
// get_words(wd) fills the 16 elements' stochastic-rounding words (called
// only for stochastic rounding, where the words are needed).
// BF16_E4: y is a bf16 input value (no residual added) and D a bare E4M3
// scale (no global scale).  Then a nonzero y is at least 2^-133 (the least
// bf16 subnormal) and D at most 448, so y / D is at least 2^-142 and the
// reciprocal sequence's quotient is nonzero exactly when y is; below 2^-25 a
// quotient's stochastic rounding depends on nothing else (the distance to
// the grid, 2|q| * 2^24, is under 1, so it rounds up only on the zero draw,
// and only if q != 0), and from 2^-25 up y is at least 2^-34, where the
// sequence is exact.  So the tiny-element check is not needed.
template <int RND, bool BF16_E4 = false, class GetWords>
__device__ __forceinline__ void encode_plain16_impl(const float* y, float D, float b, GetWords get_words,
                                                    uint32_t& w0, uint32_t& w1, const float* rt,
                                                    uint32_t sf, float* q, bool wq) {
    const bool fast = plain_fast(D, b);
    const float r = rt ? rt[sf] : (fast ? div_rn(1.0f, D) : 0.0f);
    if (RND != NVFP4_SR) {                      // nearest (either scale association)
        float v[16];
        if (fast) {                             // the reciprocal sequence on pairs (per-lane IEEE)
            const uint64_t R2 = pack2(r, r), ND2 = pack2(-D, -D);
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
                const uint64_t Y = pack2(y[i], y[i + 1]);
                const uint64_t Q0 = mul2(Y, R2);
                uint64_t Q = fma2(fma2(Q0, ND2, Y), R2, Q0);
                if (!rt) Q = fma2(fma2(Q, ND2, Y), R2, Q);
                float q0a, q0b, qa, qb;
                unpack2(Q0, q0a, q0b);
                unpack2(Q, qa, qb);
                v[i] = sign_of_first(q0a, qa);
                v[i + 1] = sign_of_first(q0b, qb);
            }
        } else {                                // copies, so that y and v stay in registers
            float yl[16], vl[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) yl[i] = y[i];
            plain_quotients16_ieee(yl, D, vl);
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = vl[i];
        }
        w0 = e2m1_encode8(v);
        w1 = e2m1_encode8(v + 8);
    } else {
        uint32_t wd[16];
        get_words(wd);
        // blocks holding an element 0 < |y| < 2^-80 (or zeros) take the per-element checked path
        bool tiny = false;
        if (!BF16_E4) {
#pragma unroll
            for (int i = 0; i < 16; ++i) tiny |= fabsf(y[i]) < 8.271806125530277e-25f;
        }
        float g[16];
        if (fast && !tiny) {
            const uint64_t R2 = pack2(r, r), ND2 = pack2(-D, -D);
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
                const uint64_t Y = pack2(y[i], y[i + 1]);
                const uint64_t Q0 = mul2(Y, R2);
                uint64_t Q = fma2(fma2(Q0, ND2, Y), R2, Q0);
                if (!rt) Q = fma2(fma2(Q, ND2, Y), R2, Q);
                float q0a, q0b, qa, qb, ga, gb;
                unpack2(Q0, q0a, q0b);
                unpack2(Q, qa, qb);
                sr_grid_value2(fabsf(qa), fabsf(qb), wd[i], wd[i + 1], ga, gb);
                g[i] = sign_of_first(q0a, ga);
                g[i + 1] = sign_of_first(q0b, gb);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float v = rt ? plain_quotient<true, true>(y[i], D, r, fast) : plain_quotient<true>(y[i], D, r, fast);
                g[i] = sign_of_first(v, sr_grid_value(fabsf(v), wd[i]));
            }
        }
        w0 = e2m1_encode8(g);
        w1 = e2m1_encode8(g + 8);
        if (wq) {
#pragma unroll
            for (int i = 0; i < 16; ++i) q[i] = g[i];
        }
    }
    if (D == 0.0f) {
        w0 = 0;
        w1 = 0;
        if (RND == NVFP4_SR && wq) {
#pragma unroll
            for (int i = 0; i < 16; ++i) q[i] = 0.0f;
        }
    }
}

// elements idx0 .. idx0 + 15 of x (the stochastic-rounding counter)
template <int RND, bool BF16_E4 = false>
__device__ __forceinline__ void encode_plain16(const float* y, float D, float b, uint64_t idx0,
                                               const PhiloxKeys& pk, uint32_t& w0,
                                               uint32_t& w1, const float* rt, uint32_t sf,
                                               float* q, bool wq) {
    encode_plain16_impl<RND, BF16_E4>(
        y, D, b, [&](uint32_t* wd) { sr_words16(idx0, pk, wd); }, w0, w1, rt, sf, q, wq);
}

// the same with the words given (wd[16], read only for stochastic rounding)
template <int RND, bool BF16_E4 = false>
__device__ __forceinline__ void encode_plain16_words(const float* y, float D, float b, const uint32_t* wd,
                                                     uint32_t& w0, uint32_t& w1, const float* rt,
                                                     uint32_t sf, float* q, bool wq) {
    encode_plain16_impl<RND, BF16_E4>(
        y, D, b,
        [&](uint32_t* out) {
#pragma unroll
            for (int i = 0; i < 16; ++i) out[i] = wd[i];
        },
        w0, w1, rt, sf, q, wq);
}

// The block scale before E4M3 rounding: (b / 6) * S_enc, or with the standard
// NVFP4 association (std_assoc) b * (S_enc * (1/6)), 1/6 the nearest fp32
// ("Add NVFP4 four-over-six (row-wise) quantization to the training
// prototype", Two load-bearing numeric details).
template <bool GS>
__device__ __forceinline__ float block_scale(float b, float Senc, bool std_assoc) {
    if (std_assoc) return mul_rn(b, mul_rn(Senc, 0.16666667163372040f));
    return block_s6f<GS>(b, Senc);
}

// y[i] += r[i] (the error-feedback sum), two elements per instruction
__device__ __forceinline__ void add16(float* y, const float* r) {
#pragma unroll
    for (int i = 0; i < 16; i += 2) unpack2(add2(pack2(y[i], y[i + 1]), pack2(r[i], r[i + 1])), y[i], y[i + 1]);
}

// Error-feedback residual r = y - q * d of a block without a global scale,
// from the codes' signed grid values q: q * d has at most 7 significant bits
// (a grid value times an E4M3 value, both normal or zero), so it is exact and
// the fused y + (-q) * d rounds once, as y - RN(q * d) does.
__device__ __forceinline__ void residual_q16(const float* y, const float* q, float d, float* r) {
    const uint64_t ND = pack2(-d, -d);
#pragma unroll
    for (int i = 0; i < 16; i += 2)
        unpack2(fma2(pack2(q[i], q[i + 1]), ND, pack2(y[i], y[i + 1])), r[i], r[i + 1]);
}

// dequantized values (q * d) * S_dec from signed grid values
template <bool GS>
__device__ __forceinline__ void dequant_q16(const float* q, float d, float Sdec, float* dq) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float v = mul_rn(q[i], d);
        dq[i] = GS ? mul_rn(v, Sdec) : v;
    }
}

// ---- four-over-six --------------------------------------------------------------------------
// One candidate over 8 values: codes of y * enc, and the per-element errors
// |dq - y| (MAE) or (dq - y)^2 (MSE) of its error values dq = ((q*d)*A)/C.
template <int ERR>
__device__ __forceinline__ void candidate8(const float* y, const Cand& c, float d, float A, float C,
                                           uint32_t& w, float* e) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = mul_rn(y[i], c.enc);
    uint32_t h[4];
    w = e2m1_encode8_dec(v, h);
    float dq[8];
    if (c.fast) {
        error_values8(h, c.X1, c.DX, dq);
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float qlo = __half2float(__ushort_as_half(static_cast<unsigned short>(h[i] & 0xFFFFu)));
            const float qhi = __half2float(__ushort_as_half(static_cast<unsigned short>(h[i] >> 16)));
            dq[2 * i] = div_rn(mul_rn(mul_rn(qlo, d), A), C);
            dq[2 * i + 1] = div_rn(mul_rn(mul_rn(qhi, d), A), C);
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float diff = sub_rn(dq[i], y[i]);
        e[i] = (ERR == NVFP4_ERR_MAE) ? fabsf(diff) : mul_rn(diff, diff);
    }
}

// The same over 16 values (two 8-value halves).
template <int ERR>
__device__ __forceinline__ void candidate16(const float* y, const Cand& c, float d, float A, float C,
                                            uint32_t& w0, uint32_t& w1, float* e) {
    candidate8<ERR>(y, c, d, A, C, w0, e);
    candidate8<ERR>(y + 8, c, d, A, C, w1, e + 8);
}

// sequential sum e[0] + ... + e[15] from 0
__device__ __forceinline__ float seq_sum16(const float* e) {
    float E = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) E = add_rn(E, e[i]);
    return E;
}

// Per-tensor four-over-six table, for a global scale shared by the tensor:
// enc[sf] = min(1/(dec(sf) * S_dec), FLT_MAX) and dq[k][sf] = ((G[k] * dec(sf))
// * A) / (6 * bound), the error-value magnitude of grid index k under scale
// byte sf (every block scale is a non-negative E4M3 byte <= 0x7E).  A code
// with index k stands for +-dq[k][sf] with the sign of its y (y * enc keeps
// y's sign), so its error |dq - y| is | dq[k][sf] - |y| | exactly, and the
// square likewise.  The row stride 132 spreads the 8 rows of one scale byte
// over distinct banks.
constexpr int kDqStride = 132;
struct O6Tab {
    float enc[128];
    float dq[8 * kDqStride];
    float2 ek[128];                             // (enc[sf], dq[grid value 1][sf]): one load per candidate
};

// the shared table of a kernel instance, or nothing when it has no four-over-six
struct NoTab {};
template <int ERR>
using O6TabOf = typename std::conditional<ERR != NVFP4_ERR_NONE, O6Tab, NoTab>::type;

__device__ __forceinline__ void fill_o6_table(O6Tab* tab, float Sdec, float A, float C) {
    const float G[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
    for (int i = threadIdx.x; i < 128; i += blockDim.x) {
        const float d = e4m3_decode(static_cast<uint32_t>(i));
        tab->enc[i] = min_nd(div_rn(1.0f, mul_rn(d, Sdec)), FLT_MAX);
#pragma unroll
        for (int k = 0; k < 8; ++k) tab->dq[k * kDqStride + i] = div_rn(mul_rn(mul_rn(G[k], d), A), C);
        tab->ek[i] = make_float2(tab->enc[i], tab->dq[2 * kDqStride + i]);
    }
    __syncthreads();
}

// One candidate over 16 values from the table: codes of y * enc and the
// per-element errors (dq: the table column of the candidate's scale byte).
template <int ERR>
__device__ __forceinline__ void candidate16_tab(const float* y, float enc, const float* dq, uint32_t& w0,
                                                uint32_t& w1, float* e) {
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = mul_rn(y[i], enc);
    w0 = e2m1_encode8(v);
    w1 = e2m1_encode8(v + 8);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t k = ((i < 8 ? w0 : w1) >> (4 * (i & 7))) & 7u;
        const float diff = sub_rn(dq[k * kDqStride], fabsf(y[i]));
        e[i] = (ERR == NVFP4_ERR_MAE) ? fabsf(diff) : mul_rn(diff, diff);
    }
}

// The exact error sum of one candidate from its codes (the per-element
// errors of candidate16_tab, summed in element order from 0 as seq_sum16).
template <int ERR>
__device__ __forceinline__ float errsum16_tab(const float* y, uint32_t w0, uint32_t w1, const float* dq) {
    float E = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t k = ((i < 8 ? w0 : w1) >> (4 * (i & 7))) & 7u;
        const float diff = sub_rn(dq[k * kDqStride], fabsf(y[i]));
        E = add_rn(E, (ERR == NVFP4_ERR_MAE) ? fabsf(diff) : mul_rn(diff, diff));
    }
    return E;
}

// Approximate error sum of one candidate, no table lookups, in the scaled
// domain: v = RN(y * enc) is the value the encode rounds to a grid value q
// (signed like y), an element's approximate error is |RN(q - v)| (one mixed
// f16/f32 subtract; squared for MSE, fused into its addition), summed as two
// interleaved chains (even and odd elements, paired instructions) that are
// then added, and the sum S' is scaled back by K, the error value of grid
// value 1 (((1 * d) * A) / C): E^ = RN(K * S'), or RN(RN(K * K) * S') for
// MSE.  The codes are the candidate's exact codes.
template <int ERR>
__device__ __forceinline__ float errsum16_approx(const float* y, float enc, float K, uint32_t& w0,
                                                 uint32_t& w1) {
    float v[16];
    const uint64_t ENC2 = pack2(enc, enc);
#pragma unroll
    for (int i = 0; i < 16; i += 2) unpack2(mul2(pack2(y[i], y[i + 1]), ENC2), v[i], v[i + 1]);
    uint32_t h[8];
    w0 = e2m1_encode8_dec(v, h);
    w1 = e2m1_encode8_dec(v + 8, h + 4);
    uint64_t S2 = pack2(0.0f, 0.0f);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float e0, e1;
        sub_f16x2_f32(h[j], v[2 * j], v[2 * j + 1], e0, e1);
        const uint64_t D = ERR == NVFP4_ERR_MSE ? pack2(e0, e1) : pack2(fabsf(e0), fabsf(e1));
        S2 = ERR == NVFP4_ERR_MSE ? fma2(D, D, S2) : add2(S2, D);
    }
    float s0, s1;
    unpack2(S2, s0, s1);
    const float S = add_rn(s0, s1);
    return ERR == NVFP4_ERR_MAE ? mul_rn(K, S) : mul_rn(mul_rn(K, K), S);
}

// Whether approximate sums E6^, E4^ (errsum16_approx) decide E4 < E6 as the
// exact sums E6, E4 do.  With u = 2^-24, K_r = d*A/C, q an element's grid
// value (|q| <= 6) and b the block amax (>= |y|):
//   an error value dq = ((q*d)*A)/C (q*d exact, two roundings) lies within
//   2.01u |q| K_r of |q| K_r, and its difference with |y| is rounded once;
//   v = y * enc with enc = RN(1 / RN(d * S_dec)) and S_dec = RN(1 / RN(C / A))
//   is y / K_r within 5.05u |y| / K_r, q - v is rounded once, the sums add
//   gamma_15 <= 15.01u of their terms (the exact sum in element order; the
//   approximate one passes each term through at most 9 additions, its MSE
//   squares fused into them), and K * S' (K within 2.01u of K_r) adds 3.02u:
//   MAE  |E - E^| <= 35.04u E^ + 193u K + 80.8u b   (sum |q| <= 96, sum |y| <= 16 b);
//   MSE  |d_t^2 - (K_r d_a)^2| = ||d_t| - K_r|d_a|| (|d_t| + K_r|d_a|), with the
//        first factor <= 12.06u K + 5.05u b + u (|d_t| + K_r|d_a|) and sum |d|
//        <= 4 sqrt(sum d^2) over 16 terms:
//        |E - E^| <= 96.5u K sqrt(E^) + 40.4u b sqrt(E^) + 42u E^.
// Per candidate, with the constants rounded up to powers of two,
// 2^6 u E^ + 2^8 u K + 2^7 u b and 2^7 u K sqrt(E^) + 2^6 u b sqrt(E^) +
// 2^6 u E^; the threshold is twice the two candidates' bounds together plus
// 2^-120 for the absolute errors of subnormal results, with the square roots
// bounded by the AM-GM inequality: K sqrt(E^) <= (E^ + K^2) / 2 and
// b sqrt(E^) <= 3 E^ + b^2 / 12.  A NaN or infinite sum, K or b gives a NaN
// difference or an infinite threshold: the test fails and the caller takes
// the exact sums.
template <int ERR>
__device__ __forceinline__ bool approx_decides(float E6, float E4, float K6, float K4, float b) {
    float T;
    if (ERR == NVFP4_ERR_MAE) {
        T = add_rn(mul_rn(add_rn(E6, E4), 7.62939453125e-06f),
                   mul_rn(add_rn(add_rn(K6, K4), b), 3.0517578125e-05f));
    } else {
        const float R = add_rn(add_rn(mul_rn(5.0f, add_rn(E6, E4)), __fmaf_rn(K6, K6, mul_rn(K4, K4))),
                               mul_rn(mul_rn(b, b), 0.1875f));
        T = mul_rn(R, 7.62939453125e-06f);
    }
    T = add_rn(T, 7.52316384526264e-37f);
    return fabsf(sub_rn(E6, E4)) > T;
}

// The same test for a 16x16 tile's sums over its 256 elements (rowwise: the
// width-16 tree of the rows' element-order sums; columnwise: of the
// columns'), each element's error passing at most 15 + 4 additions: with
// sum |q| <= 1536, sum |y| <= 256 b and gamma_19, |E - E^| <= 43.04u E^ +
// 3087u K + 1293u b for MAE and, with sum |d| <= 16 sqrt(sum d^2) over 256
// terms, <= 386u K sqrt(E^) + 162u b sqrt(E^) + 50u E^ for MSE; per
// candidate 2^6 u E^ + 2^12 u K + 2^11 u b and 2^9 u K sqrt(E^) + 2^8 u b
// sqrt(E^) + 2^6 u E^, the threshold twice the two candidates' bounds
// together plus 2^-120, with K sqrt(E^) <= (E^ + 16 K^2) / 8 and
// b sqrt(E^) <= (E^ + b^2) / 2.
template <int ERR>
__device__ __forceinline__ bool tile_sums_decide(float E6, float E4, float K6, float K4, float b) {
    float T;
    if (ERR == NVFP4_ERR_MAE) {
        T = add_rn(mul_rn(add_rn(E6, E4), 7.62939453125e-06f),
                   mul_rn(add_rn(add_rn(K6, K4), b), 4.8828125e-04f));
    } else {
        const float R = add_rn(add_rn(add_rn(E6, E4), mul_rn(4.0f, __fmaf_rn(K6, K6, mul_rn(K4, K4)))),
                               mul_rn(b, b));
        T = mul_rn(R, 3.0517578125e-05f);
    }
    T = add_rn(T, 7.52316384526264e-37f);
    return fabsf(sub_rn(E6, E4)) > T;
}

// CERT (a 1x16 block, whose error sums are its own): the sums come from
// errsum16_approx wherever approx_decides, otherwise from the table
// (per-tensor scale) or the per-block exact form (per-row scale).
template <int ERR, bool CERT = false, class TileSums>
__device__ __forceinline__ void four_over_six16(const float* y, float b, const GScale& g, float C,
                                                const O6Tab* tab, uint32_t& w0, uint32_t& w1,
                                                uint32_t& sf, float& d, TileSums tile_sums) {
    const float s6f = block_s6f<true>(b, g.Senc);
    uint32_t sf6, sf4;
    e4m3_encode2(min_nd(s6f, 448.0f), min_nd(mul_rn(s6f, 1.5f), 448.0f), sf6, sf4);
    float d6, d4;
    e4m3_decode2(sf6, sf4, d6, d4);
    uint32_t a0, a1, b0, b1;
    float e[16], E6, E4;
    if (CERT && tab) {                          // per-tensor global scale, 1x16
        const float2 ek6 = tab->ek[sf6], ek4 = tab->ek[sf4];
        const float K6 = ek6.y, K4 = ek4.y;
        E6 = errsum16_approx<ERR>(y, ek6.x, K6, a0, a1);
        E4 = errsum16_approx<ERR>(y, ek4.x, K4, b0, b1);
        if (!approx_decides<ERR>(E6, E4, K6, K4, b)) {
            E6 = errsum16_tab<ERR>(y, a0, a1, tab->dq + sf6);
            E4 = errsum16_tab<ERR>(y, b0, b1, tab->dq + sf4);
        }
    } else if (tab) {                           // per-tensor global scale: table lookups
        candidate16_tab<ERR>(y, tab->enc[sf6], tab->dq + sf6, a0, a1, e);
        E6 = seq_sum16(e);
        candidate16_tab<ERR>(y, tab->enc[sf4], tab->dq + sf4, b0, b1, e);
        E4 = seq_sum16(e);
    } else if (CERT) {                          // per-row global scale, 1x16, certified
        // K and enc as make_cand's X1 and enc (the error value of grid value
        // 1, and the encode reciprocal); the exact form only where undecided
        const float K6 = div_rn(mul_rn(d6, g.A), C), K4 = div_rn(mul_rn(d4, g.A), C);
        const float enc6 = min_nd(div_rn(1.0f, mul_rn(d6, g.Sdec)), FLT_MAX);
        const float enc4 = min_nd(div_rn(1.0f, mul_rn(d4, g.Sdec)), FLT_MAX);
        E6 = errsum16_approx<ERR>(y, enc6, K6, a0, a1);
        E4 = errsum16_approx<ERR>(y, enc4, K4, b0, b1);
        if (!approx_decides<ERR>(E6, E4, K6, K4, b)) {
            const Cand c6 = make_cand(sf6, g.Sdec, g.A, C), c4 = make_cand(sf4, g.Sdec, g.A, C);
            candidate16<ERR>(y, c6, d6, g.A, C, a0, a1, e);
            E6 = seq_sum16(e);
            candidate16<ERR>(y, c4, d4, g.A, C, b0, b1, e);
            E4 = seq_sum16(e);
        }
    } else {                                    // per-row global scale: candidates per block
        const Cand c6 = make_cand(sf6, g.Sdec, g.A, C), c4 = make_cand(sf4, g.Sdec, g.A, C);
        candidate16<ERR>(y, c6, d6, g.A, C, a0, a1, e);
        E6 = seq_sum16(e);
        candidate16<ERR>(y, c4, d4, g.A, C, b0, b1, e);
        E4 = seq_sum16(e);
    }
    tile_sums(E6, E4);
    const bool pick4 = E4 < E6;                 // ties and NaN keep map-to-6
    w0 = pick4 ? b0 : a0;
    w1 = pick4 ? b1 : a1;
    sf = pick4 ? sf4 : sf6;
    d = pick4 ? d4 : d6;
}

// TREE: the tile's 16 rows are the 16 lanes of the caller's half warp;
// otherwise a 1x16 block (certified sums).
template <int ERR, bool TREE>
__device__ __forceinline__ void four_over_six16(const float* y, float b, const GScale& g, float C,
                                                const O6Tab* tab, uint32_t& w0, uint32_t& w1,
                                                uint32_t& sf, float& d) {
    four_over_six16<ERR, !TREE>(y, b, g, C, tab, w0, w1, sf, d, [](float& E6, float& E4) {
        if (TREE) {
            E6 = tree16_lanes(E6);
            E4 = tree16_lanes(E4);
        }
    });
}

// dequantized values (q * d) * S_dec of 16 codes
template <bool GS>
__device__ __forceinline__ void dequant16(uint32_t w0, uint32_t w1, float d, float Sdec, float* dq) {
    float q[16];
    e2m1_decode8(w0, q);
    e2m1_decode8(w1, q + 8);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float v = mul_rn(q[i], d);
        dq[i] = GS ? mul_rn(v, Sdec) : v;
    }
}

}  // namespace nvfp4
