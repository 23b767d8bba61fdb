// nvfp4_params.h -- argument bundle passed from the C ABI to the kernels.
#pragma once

#include <cstdint>

#include "../../include/nvfp4.h"

namespace nvfp4 {

// Philox4x32-10 (Salmon et al., SC'11) keyed on the seed, with the step as the
// counter's upper words: the ten round keys and the first round's terms that
// depend only on (seed, step), filled on the host for each call so that the
// kernels read them as launch constants.  Counter (c0, c1, s0, s1) with
// (s0, s1) = step: round 0 gives (r0x ^ c1, r0y, hi(M0 c0) ^ r0z, lo(M0 c0)).
struct PhiloxKeys {
    uint32_t k0[10], k1[10];   // round r's key words
    uint32_t r0x;              // hi(M1 * s0) ^ k0[0]
    uint32_t r0y;              // lo(M1 * s0)
    uint32_t r0z;              // s1 ^ k1[0]
};

constexpr uint32_t kPhiloxM0 = 0xD2511F53u, kPhiloxM1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u, kPhiloxW1 = 0xBB67AE85u;

inline PhiloxKeys philox_keys(uint64_t seed, uint64_t step) {
    PhiloxKeys p;
    uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
    for (int r = 0; r < 10; ++r) {
        p.k0[r] = k0;
        p.k1[r] = k1;
        k0 += kPhiloxW0;
        k1 += kPhiloxW1;
    }
    const uint64_t m = static_cast<uint64_t>(kPhiloxM1) * static_cast<uint32_t>(step);
    p.r0x = static_cast<uint32_t>(m >> 32) ^ p.k0[0];
    p.r0y = static_cast<uint32_t>(m);
    p.r0z = static_cast<uint32_t>(step >> 32) ^ p.k1[0];
    return p;
}

struct QuantArgs {
    const void* x;
    int64_t M, K;
    int dtype, block, rounding;
    float* residual;          // null = no error feedback
    uint64_t seed, step;
    int64_t row_offset;
    int gamax_mode;           // after the amax step: NONE, TENSOR_GIVEN or ROW_GIVEN
    const float* gamax;
    int err_mode;
    float bound;
    uint8_t* codes;           // may be null for qdq
    uint8_t* scales;          // may be null for qdq
    uint8_t* codes_col;       // null = no columnwise output
    uint8_t* scales_col;
    uint16_t* dq_bf16;        // qdq output, null otherwise
    PhiloxKeys pk;            // philox_keys(seed, step), set by the entry point
};

struct DequantArgs {
    const uint8_t* codes;
    const uint8_t* scales;
    int64_t M, K;
    int gamax_mode;
    const float* gamax;
    float bound;
    void* out;
    int out_dtype;
};

// launchers (each returns cudaGetLastError() after its launches)
int launch_quantize_rows(const QuantArgs& a, void* stream);    // rowwise output only
int launch_quantize_tiles(const QuantArgs& a, void* stream);   // rowwise + columnwise
int launch_dequantize(const DequantArgs& a, void* stream);
int launch_scales_mma(const uint8_t* in, int64_t rows, int64_t cols, uint8_t* out, void* stream);
int launch_mm(const uint8_t* A, const uint8_t* SA, const uint8_t* B, const uint8_t* SB, int64_t M, int64_t N,
              int64_t K, const float* gamax_a, const float* gamax_b, float bound, void* out, int out_dtype,
              void* stream);
int launch_amax(const void* x, int64_t M, int64_t K, int dtype, const float* residual, int mode,
                float* out, void* stream);
int launch_probe_divide(const float* a, const float* b, float* out, int64_t n, void* stream);
int launch_probe_sub_f16(const uint32_t* q, const float* v, float* out, int64_t n, void* stream);
int launch_probe_e2m1(uint32_t first, int64_t n, uint8_t* out, void* stream);
int launch_global_scales(const float* gamax, int64_t n, float bound, float* s_enc, float* s_dec, void* stream);
int sm_count();

}  // namespace nvfp4
