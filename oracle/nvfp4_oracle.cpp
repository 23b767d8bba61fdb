/*
 * nvfp4_oracle.cpp -- plain, slow CPU oracle for NVFP4 block quantization.
 *
 * TEST INFRASTRUCTURE ONLY: called by the tests, the smoke check and the
 * benchmark's CPU-baseline leg, never by the product library.  No blocking,
 * no fusion, no reordering: each step is written in the order the pages give
 * it so a reader can check it against them by eye.  Citation tags are
 * explained in nvfp4_oracle.h.
 *
 * Build: g++ -O2 -ffp-contract=off -fno-fast-math (fp32 ops must round once,
 * exactly as written; orc_fp_env_ok() checks that subnormals survive).
 *
 * Parity unpinned: two steps rest on a reading that no value on the pages
 * fixes, so only this restatement and the GPU's agreement check them: the
 * association of the four-over-six error value ((q * d) * A) / (6 * bound)
 * when S_enc != 1 (planted mistakes q * (d * A) and (q * d) * (A / C) pass
 * every pin), and the S_enc = 1 fallback for a global amax that is 0, Inf,
 * NaN or negative (pinned only against that reading).  Every other step is
 * pinned by tests/test_oracle_pins.py, each pin checked by a planted mistake
 * in tests/test_oracle_mutations.py.
 */
#include "nvfp4_oracle.h"

#include <algorithm>
#include <cfloat>
#include <cmath>
#include <cstring>
#include <thread>
#include <vector>

namespace {

/* Worker threads for the loops over independent rows, bands and elements.
 * Each block's arithmetic is the same whichever thread runs it, and the only
 * cross-block combination (the tensor amax) is a NaN-dropping maximum of
 * non-negative values, which is exact in any order; so every thread count
 * gives the same bytes.  1 (the default) runs everything on the calling
 * thread. */
int g_threads = 1;

/* f(lo, hi) over [0, n), split into at most g_threads contiguous chunks. */
template <class F>
void parallel_for(int64_t n, F f) {
    const int64_t T = std::min<int64_t>(g_threads, n);
    if (T <= 1) {
        if (n > 0) f(int64_t{0}, n);
        return;
    }
    std::vector<std::thread> pool;
    for (int64_t t = 0; t < T; ++t) {
        const int64_t lo = n * t / T, hi = n * (t + 1) / T;
        pool.emplace_back([=] { f(lo, hi); });
    }
    for (auto& th : pool) th.join();
}

/* The signed e2m1 grid magnitudes, index k = 0..7 [fp4-train, Method]. */
const double kGrid[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

/* NaN-dropping max / min (IEEE maxNum / minNum): the block amax ignores NaN
 * and the 448 cap ignores NaN [4o6 PR, Design]. */
float max_nd(float a, float b) { return std::fmax(a, b); }
float min_nd(float a, float b) { return std::fmin(a, b); }

float widen(const void* x, int dtype, int64_t i) {
    if (dtype == ORC_BF16) return orc_bf16_to_f32(static_cast<const uint16_t*>(x)[i]);
    return static_cast<const float*>(x)[i];
}

/* Global encode / decode scales of one tensor or row.  NONE mode: both 1. */
struct GScale {
    float A;      /* the global amax the 4o6 error term multiplies by */
    float S_enc;
    float S_dec;
};

/* Map-to-6 block scale: s6f = (b / 6) * S_enc, capped at 448 with a
 * NaN-dropping min, then RN-even to E4M3 ([fp4-train, Method] "block_absmax / 6
 * encoded to e4m3"; [4o6 PR, Two load-bearing numeric details] the
 * (block_amax / 6) * S_enc association; [4o6 PR, Design] the 448 cap). */
float block_s6f(float b, float S_enc) { return (b / 6.0f) * S_enc; }

/* The standard NVFP4 association the four-over-six page contrasts with its own
 * ([4o6 PR, Two load-bearing numeric details]): b * (S_enc * (1/6)), with 1/6
 * the fp32 constant nearest to it.  It rounds differently from (b / 6) * S_enc
 * on some blocks. */
float block_s6f_std(float b, float S_enc) { return b * (S_enc * (1.0f / 6.0f)); }

/* Error sum of one candidate over a block ([4o6 PR, Design]): elements of a
 * 16-group are added strictly in order 0..15 starting from 0; a 16x16 tile
 * combines its 16 row sums with the fixed width-16 tree
 * (((e0+e8)+(e4+e12))+((e2+e10)+(e6+e14))) + (((e1+e9)+(e5+e13))+((e3+e11)+(e7+e15))). */
float block_error(const float* e, int n) {
    if (n == 16) {
        float E = 0.0f;
        for (int t = 0; t < 16; ++t) E = E + e[t];
        return E;
    }
    float R[16];
    for (int r = 0; r < 16; ++r) {
        float E = 0.0f;
        for (int t = 0; t < 16; ++t) E = E + e[16 * r + t];
        R[r] = E;
    }
    return (((R[0] + R[8]) + (R[4] + R[12])) + ((R[2] + R[10]) + (R[6] + R[14]))) +
           (((R[1] + R[9]) + (R[5] + R[13])) + ((R[3] + R[11]) + (R[7] + R[15])));
}

struct PlaneArgs {
    const float* y;           /* R x C fp32 plane */
    int64_t R, C;
    bool transposed;          /* the plane is x^T: SR draws are keyed on x's index */
    int block, rounding, err_mode;
    float bound;
    const GScale* gs;         /* per row of the plane (all equal for per-tensor) */
    uint64_t seed, step;
    int64_t row_offset;       /* global row index of plane row 0 (SR counter) */
    uint8_t* codes;           /* R x C/2  */
    uint8_t* scales;          /* R x C/16 */
    float* dq32;              /* R x C, optional: dequantized value of the stored code */
};

void store_code(uint8_t* codes, int64_t C, int64_t r, int64_t c, uint8_t code) {
    uint8_t& byte = codes[r * (C / 2) + c / 2];
    if (c % 2 == 0) byte = static_cast<uint8_t>((byte & 0xF0) | code);         /* even: low nibble */
    else            byte = static_cast<uint8_t>((byte & 0x0F) | (code << 4));  /* odd: high nibble */
}

/* Quantize one block of the plane; positions are (row, col) pairs. */
void quantize_block(const PlaneArgs& P, const int64_t* rows, const int64_t* cols, int n) {
    const GScale& g = P.gs[rows[0]];
    /* block absmax, NaN dropped, all-NaN -> 0 [fp4-train, Method; 4o6 PR, Design] */
    float b = 0.0f;
    for (int i = 0; i < n; ++i) b = max_nd(b, std::fabs(P.y[rows[i] * P.C + cols[i]]));

    const float s6f = (P.rounding == ORC_RTN_STD) ? block_s6f_std(b, g.S_enc) : block_s6f(b, g.S_enc);
    const uint8_t sf6 = orc_e4m3_encode(min_nd(s6f, 448.0f));
    const float d6 = orc_e4m3_decode(sf6);

    uint8_t code[256];
    uint8_t sf_out;
    float d_out;
    if (P.err_mode == ORC_ERR_NONE) {
        /* plain path: divide by the decoded scale, round to the grid
         * [fp4-train, Method]; a zero scale quantizes the block to zero
         * [fp4-train, Requirements and limits] */
        const float D = d6 * g.S_dec;
        for (int i = 0; i < n; ++i) {
            const float yv = P.y[rows[i] * P.C + cols[i]];
            if (D == 0.0f) { code[i] = 0; continue; }
            const float v = yv / D;
            if (P.rounding != ORC_SR) {
                code[i] = orc_e2m1_encode_rn(v);
            } else {
                /* the draw is keyed on the element's global index in x (row-major,
                 * row_offset rows before this tensor), also for the x^T plane, so
                 * x and x^T round each element the same way [Stable FP4 Training
                 * via Transposition-Invariant Block Quantization, abstract] */
                const int64_t xr = P.transposed ? cols[i] : rows[i];
                const int64_t xc = P.transposed ? rows[i] : cols[i];
                const int64_t xK = P.transposed ? P.R : P.C;
                const uint64_t idx = static_cast<uint64_t>(P.row_offset + xr) * static_cast<uint64_t>(xK) +
                                     static_cast<uint64_t>(xc);
                code[i] = orc_e2m1_encode_sr(v, orc_sr_uniform(P.seed, P.step, idx));
            }
        }
        sf_out = sf6;
        d_out = d6;
    } else {
        /* four-over-six [4o6 PR, What + Design]: a second candidate whose
         * pre-rounding scale is expanded by exactly 1.5x, both encoded with the
         * reciprocal min(1/(scale * S_dec), FLT_MAX), each judged by its
         * dequantization error ((q * d) * A) / (6 * bound) against y */
        const uint8_t sf4 = orc_e4m3_encode(min_nd(s6f * 1.5f, 448.0f));
        const float d4 = orc_e4m3_decode(sf4);
        const float denom = 6.0f * P.bound;
        const float dc[2] = {d6, d4};
        uint8_t cc[2][256];
        float E[2];
        for (int cand = 0; cand < 2; ++cand) {
            const float enc = min_nd(1.0f / (dc[cand] * g.S_dec), FLT_MAX);
            float err[256];
            for (int i = 0; i < n; ++i) {
                const float yv = P.y[rows[i] * P.C + cols[i]];
                cc[cand][i] = orc_e2m1_encode_rn(yv * enc);
                const float q = orc_e2m1_value(cc[cand][i]);
                const float dq = ((q * dc[cand]) * g.A) / denom;
                const float diff = dq - yv;
                err[i] = (P.err_mode == ORC_ERR_MAE) ? std::fabs(diff) : diff * diff;
            }
            E[cand] = block_error(err, n);
        }
        /* strict E4 < E6 picks map-to-4; ties and NaN pick map-to-6 */
        const int pick = (E[1] < E[0]) ? 1 : 0;
        for (int i = 0; i < n; ++i) code[i] = cc[pick][i];
        sf_out = pick ? sf4 : sf6;
        d_out = dc[pick];
    }

    for (int i = 0; i < n; ++i) {
        store_code(P.codes, P.C, rows[i], cols[i], code[i]);
        if (P.dq32) {
            /* dequantized value: (q * scale) * S_dec [fp4-train, API dequantize] */
            const float q = orc_e2m1_value(code[i]);
            P.dq32[rows[i] * P.C + cols[i]] = (q * d_out) * g.S_dec;
        }
    }
    /* one scale byte per 16 columns of each row; a 16x16 tile writes its byte
     * on each of its 16 rows */
    for (int i = 0; i < n; i += 16) P.scales[rows[i] * (P.C / 16) + cols[i] / 16] = sf_out;
}

void quantize_plane(const PlaneArgs& P) {
    if (P.block == ORC_BLOCK_1X16) {
        parallel_for(P.R, [&](int64_t r0, int64_t r1) {
            int64_t rows[16], cols[16];
            for (int64_t r = r0; r < r1; ++r)
                for (int64_t j = 0; j < P.C / 16; ++j) {
                    for (int t = 0; t < 16; ++t) { rows[t] = r; cols[t] = 16 * j + t; }
                    quantize_block(P, rows, cols, 16);
                }
        });
    } else {
        parallel_for(P.R / 16, [&](int64_t i0, int64_t i1) {
            int64_t rows[256], cols[256];
            for (int64_t i = i0; i < i1; ++i)
                for (int64_t j = 0; j < P.C / 16; ++j) {
                    for (int t = 0; t < 16; ++t)
                        for (int u = 0; u < 16; ++u) {
                            rows[16 * t + u] = 16 * i + t;
                            cols[16 * t + u] = 16 * j + u;
                        }
                    quantize_block(P, rows, cols, 256);
                }
        });
    }
}

bool valid_bound(float b) { return b > 0.0f && b <= 448.0f; }

/* Argument rules shared by quantize and qdq (see the product header). */
bool args_ok(int64_t M, int64_t K, int dtype, int block, int rounding, const float* residual,
             int gamax_mode, int err_mode, float bound, bool colwise) {
    if (M < 0 || K < 0 || K % 16 != 0) return false;
    if (dtype != ORC_F32 && dtype != ORC_BF16) return false;
    if (block != ORC_BLOCK_1X16 && block != ORC_BLOCK_16X16) return false;
    if (rounding != ORC_RTN && rounding != ORC_SR && rounding != ORC_RTN_STD) return false;
    if (gamax_mode < ORC_GAMAX_NONE || gamax_mode > ORC_GAMAX_ROW_GIVEN) return false;
    if (err_mode < ORC_ERR_NONE || err_mode > ORC_ERR_MSE) return false;
    if (!valid_bound(bound)) return false;
    if ((block == ORC_BLOCK_16X16 || colwise) && M % 16 != 0) return false;
    const bool rowmode = gamax_mode == ORC_GAMAX_ROW || gamax_mode == ORC_GAMAX_ROW_GIVEN;
    if (rowmode && (block == ORC_BLOCK_16X16 || colwise)) return false;
    if (err_mode != ORC_ERR_NONE) {
        if (rounding != ORC_RTN || residual) return false;
        if (gamax_mode == ORC_GAMAX_NONE) return false;
        if (bound != 256.0f && bound != 448.0f) return false;
    }
    if (colwise && residual) return false;
    return true;
}

}  // namespace

extern "C" {

/* ---- scalar codecs -------------------------------------------------- */

/* E4M3FN: sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent 15 with
 * mantissa 7 is NaN, there is no infinity; subnormals m * 2^-9. */
float orc_e4m3_decode(uint8_t b) {
    const int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
    if (e == 15 && m == 7) return NAN;
    const double mag = (e == 0) ? std::ldexp(static_cast<double>(m), -9)
                                : std::ldexp(1.0 + m / 8.0, e - 7);
    return static_cast<float>(s ? -mag : mag);
}

/* Round to the nearest E4M3FN value, ties to the even code; magnitudes at or
 * beyond the largest finite value 448 saturate to 448; NaN stays NaN. */
uint8_t orc_e4m3_encode(float s) {
    if (std::isnan(s)) return 0x7F;
    const uint8_t sign = std::signbit(s) ? 0x80 : 0x00;
    const double a = std::fabs(static_cast<double>(s));
    if (a >= 448.0) return static_cast<uint8_t>(sign | 0x7E);
    for (int c = 0; c < 0x7E; ++c) {
        const double lo = orc_e4m3_decode(static_cast<uint8_t>(c));
        const double hi = orc_e4m3_decode(static_cast<uint8_t>(c + 1));
        if (a >= lo && a < hi) {
            const double twice = 2.0 * a, sum = lo + hi;   /* both exact */
            int pick;
            if (twice < sum) pick = c;
            else if (twice > sum) pick = c + 1;
            else pick = (c % 2 == 0) ? c : c + 1;
            return static_cast<uint8_t>(sign | pick);
        }
    }
    return static_cast<uint8_t>(sign | 0x7E);  /* unreachable */
}

float orc_e2m1_value(uint8_t code) {
    const double mag = kGrid[code & 7];
    return static_cast<float>((code & 8) ? -mag : mag);
}

/* Nearest grid point; exact midpoints go to the even index k; |v| >= 6 and
 * infinities saturate to 6; NaN encodes to +6 ([4o6 PR, Design]).  The sign
 * bit is kept, so negative values that round to zero give code 0x8. */
uint8_t orc_e2m1_encode_rn(float v) {
    if (std::isnan(v)) return 0x7;
    const uint8_t sign = std::signbit(v) ? 0x8 : 0x0;
    const double a = std::fabs(static_cast<double>(v));
    if (a >= 6.0) return static_cast<uint8_t>(sign | 7);
    for (int k = 0; k < 7; ++k) {
        if (a >= kGrid[k] && a < kGrid[k + 1]) {
            const double twice = 2.0 * a, sum = kGrid[k] + kGrid[k + 1];
            int pick;
            if (twice < sum) pick = k;
            else if (twice > sum) pick = k + 1;
            else pick = (k % 2 == 0) ? k : k + 1;
            return static_cast<uint8_t>(sign | pick);
        }
    }
    return static_cast<uint8_t>(sign | 7);  /* unreachable */
}

/* Stochastic rounding [fp4-train, Method]: between grid points G[k] < |v| <
 * G[k+1] the higher one is chosen with probability equal to the fractional
 * distance p = (|v| - G[k]) / (G[k+1] - G[k]), i.e. when u < p.  Grid points,
 * |v| >= 6 and NaN are handled as in RN. */
uint8_t orc_e2m1_encode_sr(float v, double u) {
    if (std::isnan(v)) return 0x7;
    const uint8_t sign = std::signbit(v) ? 0x8 : 0x0;
    const double a = std::fabs(static_cast<double>(v));
    if (a >= 6.0) return static_cast<uint8_t>(sign | 7);
    for (int k = 0; k < 7; ++k) {
        if (a >= kGrid[k] && a < kGrid[k + 1]) {
            if (a == kGrid[k]) return static_cast<uint8_t>(sign | k);
            const double p = (a - kGrid[k]) / (kGrid[k + 1] - kGrid[k]);  /* exact */
            return static_cast<uint8_t>(sign | (u < p ? k + 1 : k));
        }
    }
    return static_cast<uint8_t>(sign | 7);  /* unreachable */
}

float orc_bf16_to_f32(uint16_t h) {
    const uint32_t u = static_cast<uint32_t>(h) << 16;   /* exact widening */
    float f;
    std::memcpy(&f, &u, 4);
    return f;
}

/* fp32 -> bf16 round-to-nearest-even on the dropped 16 bits. */
uint16_t orc_f32_to_bf16(float f) {
    uint32_t u;
    std::memcpy(&u, &f, 4);
    if (std::isnan(f)) return static_cast<uint16_t>((u >> 16) | 0x0040);
    const uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return static_cast<uint16_t>(u >> 16);
}

/* ---- Philox4x32-10 -------------------------------------------------- */
/* Salmon et al., "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11):
 * each round multiplies words 0 and 2 by the two round multipliers, and the
 * next state is (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2), hi(M0*c0) ^ c3 ^ k1,
 * lo(M0*c0)); the key is bumped by the two Weyl constants between rounds. */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) { k0 += W0; k1 += W1; }
        const uint64_t p0 = static_cast<uint64_t>(M0) * c0;
        const uint64_t p1 = static_cast<uint64_t>(M1) * c2;
        const uint32_t n0 = static_cast<uint32_t>(p1 >> 32) ^ c1 ^ k0;
        const uint32_t n1 = static_cast<uint32_t>(p1);
        const uint32_t n2 = static_cast<uint32_t>(p0 >> 32) ^ c3 ^ k1;
        const uint32_t n3 = static_cast<uint32_t>(p0);
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The counter-based (seed, step, global-index) draw of [fp4-train, Method]:
 * key = (lo32(seed), hi32(seed)), counter = (lo32(idx/4), hi32(idx/4),
 * lo32(step), hi32(step)); element idx uses output word idx % 4, whose top
 * 24 bits give u = (word >> 8) * 2^-24. */
double orc_sr_uniform(uint64_t seed, uint64_t step, uint64_t idx) {
    const uint64_t blk = idx >> 2;
    const uint32_t ctr[4] = {static_cast<uint32_t>(blk), static_cast<uint32_t>(blk >> 32),
                             static_cast<uint32_t>(step), static_cast<uint32_t>(step >> 32)};
    const uint32_t key[2] = {static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32)};
    uint32_t out[4];
    orc_philox4x32_10(ctr, key, out);
    return std::ldexp(static_cast<double>(out[idx & 3] >> 8), -24);
}

/* ---- global scale ---------------------------------------------------- */
/* S_enc = min(6 * bound / A, FLT_MAX) with a true division, falling back to 1
 * when A is not a positive finite number; S_dec = 1 / S_enc
 * ([4o6 PR, What + Design]: bound 256 by default, 448 allowed; FLT_MAX clamps). */
void orc_global_scales(float A, float bound, float* S_enc, float* S_dec) {
    float enc;
    if (!(A > 0.0f) || std::isinf(A)) enc = 1.0f;
    else enc = min_nd((6.0f * bound) / A, FLT_MAX);
    *S_enc = enc;
    *S_dec = 1.0f / enc;
}

void orc_amax(const void* x, int64_t M, int64_t K, int dtype, const float* residual,
              int mode, float* out) {
    if (mode == ORC_GAMAX_TENSOR) {
        /* max over rows of the row maxima: the same value as one running max
         * (the NaN-dropping maximum of non-negative values is order-free) */
        std::vector<float> part(static_cast<size_t>(M > 0 ? M : 1), 0.0f);
        orc_amax(x, M, K, dtype, residual, ORC_GAMAX_ROW, part.data());
        float A = 0.0f;
        for (int64_t r = 0; r < M; ++r) A = max_nd(A, part[r]);
        out[0] = A;
    } else {
        parallel_for(M, [&](int64_t r0, int64_t r1) {
            for (int64_t r = r0; r < r1; ++r) {
                float A = 0.0f;
                for (int64_t c = 0; c < K; ++c) {
                    float y = widen(x, dtype, r * K + c);
                    if (residual) y = y + residual[r * K + c];
                    A = max_nd(A, std::fabs(y));
                }
                out[r] = A;
            }
        });
    }
}

/* ---- quantize --------------------------------------------------------- */
int orc_quantize(const void* x, int64_t M, int64_t K, int dtype, int block, int rounding,
                 float* residual, uint64_t seed, uint64_t step, int64_t row_offset,
                 int gamax_mode, float* gamax, int err_mode, float scale_bound,
                 uint8_t* codes, uint8_t* scales, uint8_t* codes_col, uint8_t* scales_col) {
    const bool colwise = codes_col != nullptr;
    if (!args_ok(M, K, dtype, block, rounding, residual, gamax_mode, err_mode, scale_bound, colwise))
        return 1;

    /* y = x, or x + residual under error feedback [fp4-train, Method] */
    std::vector<float> y(static_cast<size_t>(M * K));
    parallel_for(M * K, [&](int64_t i0, int64_t i1) {
        for (int64_t i = i0; i < i1; ++i) {
            y[i] = widen(x, dtype, i);
            if (residual) y[i] = y[i] + residual[i];
        }
    });

    /* global amax and scales: per tensor or per row [4o6 PR, What] */
    std::vector<GScale> gs(static_cast<size_t>(M > 0 ? M : 1));
    if (gamax_mode == ORC_GAMAX_TENSOR) orc_amax(y.data(), M, K, ORC_F32, nullptr, ORC_GAMAX_TENSOR, gamax);
    if (gamax_mode == ORC_GAMAX_ROW) orc_amax(y.data(), M, K, ORC_F32, nullptr, ORC_GAMAX_ROW, gamax);
    for (int64_t r = 0; r < M; ++r) {
        GScale g{0.0f, 1.0f, 1.0f};
        if (gamax_mode == ORC_GAMAX_TENSOR || gamax_mode == ORC_GAMAX_TENSOR_GIVEN) g.A = gamax[0];
        if (gamax_mode == ORC_GAMAX_ROW || gamax_mode == ORC_GAMAX_ROW_GIVEN) g.A = gamax[r];
        if (gamax_mode != ORC_GAMAX_NONE) orc_global_scales(g.A, scale_bound, &g.S_enc, &g.S_dec);
        gs[r] = g;
    }

    std::vector<float> dq;
    if (residual) dq.resize(static_cast<size_t>(M * K));

    PlaneArgs P{y.data(), M, K, false, block, rounding, err_mode, scale_bound, gs.data(),
                seed, step, row_offset, codes, scales, residual ? dq.data() : nullptr};
    quantize_plane(P);

    /* error feedback: carry y - dequant(quantize(y)) [fp4-train, Method] */
    if (residual)
        parallel_for(M * K, [&](int64_t i0, int64_t i1) {
            for (int64_t i = i0; i < i1; ++i) residual[i] = y[i] - dq[i];
        });

    /* columnwise output = the rowwise quantization of x^T with the same
     * per-tensor scale [4o6 PR, Validation; Follow-up fusions] */
    if (colwise) {
        std::vector<float> yt(static_cast<size_t>(M * K));
        parallel_for(K, [&](int64_t c0, int64_t c1) {
            for (int64_t c = c0; c < c1; ++c)
                for (int64_t r = 0; r < M; ++r) yt[c * M + r] = y[r * K + c];
        });
        std::vector<GScale> gt(static_cast<size_t>(K > 0 ? K : 1), M > 0 ? gs[0] : GScale{0.0f, 1.0f, 1.0f});
        PlaneArgs T{yt.data(), K, M, true, block, rounding, err_mode, scale_bound, gt.data(),
                    seed, step, row_offset, codes_col, scales_col, nullptr};
        quantize_plane(T);
    }
    return 0;
}

/* ---- scale layout for the block-scaled matrix multiply ---------------- */
void orc_scales_to_mma(const uint8_t* scales, int64_t rows, int64_t cols, uint8_t* out) {
    const int64_t R = (rows + 127) / 128 * 128, C = (cols + 3) / 4 * 4;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c) {
            const uint8_t v = (r < rows && c < cols) ? scales[r * cols + c] : 0;
            const int64_t tile = (r / 128) * (C / 4) + c / 4;
            const int64_t rr = r % 128, cc = c % 4;
            out[tile * 512 + (rr % 32) * 16 + (rr / 32) * 4 + cc] = v;
        }
}

/* ---- dequantize ------------------------------------------------------- */
int orc_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t M, int64_t K,
                   int gamax_mode, const float* gamax, float scale_bound,
                   void* out, int out_dtype) {
    if (M < 0 || K < 0 || K % 16 != 0 || !valid_bound(scale_bound)) return 1;
    if (gamax_mode < ORC_GAMAX_NONE || gamax_mode > ORC_GAMAX_ROW_GIVEN) return 1;
    parallel_for(M, [&](int64_t r0, int64_t r1) {
        for (int64_t r = r0; r < r1; ++r) {
            float S_enc = 1.0f, S_dec = 1.0f;
            if (gamax_mode == ORC_GAMAX_TENSOR || gamax_mode == ORC_GAMAX_TENSOR_GIVEN)
                orc_global_scales(gamax[0], scale_bound, &S_enc, &S_dec);
            if (gamax_mode == ORC_GAMAX_ROW || gamax_mode == ORC_GAMAX_ROW_GIVEN)
                orc_global_scales(gamax[r], scale_bound, &S_enc, &S_dec);
            for (int64_t c = 0; c < K; ++c) {
                const uint8_t byte = codes[r * (K / 2) + c / 2];
                const uint8_t code = (c % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
                const float d = orc_e4m3_decode(scales[r * (K / 16) + c / 16]);
                /* the decoded value q * d is exact (a 2-bit grid value times a
                 * 4-bit E4M3 significand), so (q * d) * S_dec rounds once */
                const float v = (orc_e2m1_value(code) * d) * S_dec;
                if (out_dtype == ORC_BF16) static_cast<uint16_t*>(out)[r * K + c] = orc_f32_to_bf16(v);
                else static_cast<float*>(out)[r * K + c] = v;
            }
        }
    });
    return 0;
}

/* ---- qdq: quantize then dequantize [fp4-train, API qdq] --------------- */
int orc_qdq(const void* x, int64_t M, int64_t K, int dtype, int block, int rounding,
            float* residual, uint64_t seed, uint64_t step, int64_t row_offset,
            int gamax_mode, float* gamax, int err_mode, float scale_bound,
            uint8_t* codes, uint8_t* scales, uint16_t* out_bf16) {
    std::vector<uint8_t> c_tmp, s_tmp;
    if (!codes) { c_tmp.resize(static_cast<size_t>(M * K / 2)); codes = c_tmp.data(); }
    if (!scales) { s_tmp.resize(static_cast<size_t>(M * K / 16)); scales = s_tmp.data(); }
    const int rc = orc_quantize(x, M, K, dtype, block, rounding, residual, seed, step, row_offset,
                                gamax_mode, gamax, err_mode, scale_bound, codes, scales,
                                nullptr, nullptr);
    if (rc) return rc;
    return orc_dequantize(codes, scales, M, K, gamax_mode, gamax, scale_bound, out_bf16, ORC_BF16);
}

/* ---- batch forms of the scalar codecs (loops, for exhaustive checks) -- */
void orc_e4m3_encode_n(const float* s, int64_t n, uint8_t* out) {
    parallel_for(n, [&](int64_t i0, int64_t i1) {
        for (int64_t i = i0; i < i1; ++i) out[i] = orc_e4m3_encode(s[i]);
    });
}
void orc_e2m1_encode_rn_n(const float* v, int64_t n, uint8_t* out) {
    parallel_for(n, [&](int64_t i0, int64_t i1) {
        for (int64_t i = i0; i < i1; ++i) out[i] = orc_e2m1_encode_rn(v[i]);
    });
}
/* the same over consecutive fp32 bit patterns first, first + 1, ..., first + n - 1
 * (an exhaustive sweep needs no input array) */
void orc_e2m1_encode_rn_bits(uint32_t first, int64_t n, uint8_t* out) {
    parallel_for(n, [&](int64_t i0, int64_t i1) {
        for (int64_t i = i0; i < i1; ++i) {
            const uint32_t u = first + static_cast<uint32_t>(i);
            float f;
            std::memcpy(&f, &u, 4);
            out[i] = orc_e2m1_encode_rn(f);
        }
    });
}
void orc_e2m1_encode_sr_n(const float* v, const double* u, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e2m1_encode_sr(v[i], u[i]);
}
void orc_sr_uniform_n(uint64_t seed, uint64_t step, const uint64_t* idx, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_sr_uniform(seed, step, idx[i]);
}
void orc_f32_to_bf16_n(const float* f, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_bf16(f[i]);
}

int orc_set_threads(int n) {
    const int old = g_threads;
    if (n <= 0) n = static_cast<int>(std::thread::hardware_concurrency());
    g_threads = n > 0 ? n : 1;
    return old;
}

int orc_get_threads(void) { return g_threads; }

int orc_fp_env_ok(void) {
    volatile float t = 1.0e-38f;   /* below FLT_MIN: a subnormal */
    volatile float h = t * 0.5f;
    return (h != 0.0f && h < t) ? 1 : 0;
}

}  // extern "C"
