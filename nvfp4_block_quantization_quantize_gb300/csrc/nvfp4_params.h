// nvfp4_params.h -- argument bundle passed from the C ABI to the kernels.
#pragma once

#include <cstdint>

#include "../../include/nvfp4.h"

namespace nvfp4 {

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
int launch_probe_e2m1(uint32_t first, int64_t n, uint8_t* out, void* stream);
int launch_global_scales(const float* gamax, int64_t n, float bound, float* s_enc, float* s_dec, void* stream);
int sm_count();

}  // namespace nvfp4
