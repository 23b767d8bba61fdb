// nvfp4_api.cu -- the C ABI declared in include/nvfp4.h.
//
// Host side only: argument checks (nothing is enqueued when one fails), the
// optional global-amax pass, and the choice of kernel.  No allocation, no
// synchronization; everything runs on the caller's stream.
#include <cstdarg>
#include <cstdio>
#include <cstdint>

#include <cuda_runtime.h>

#include "nvfp4_params.h"

namespace {

thread_local char g_msg[512] = "";

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(int err, const char* what) {
    return fail(NVFP4_ECUDA, "%s: %s", what, cudaGetErrorString(static_cast<cudaError_t>(err)));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_ptr(const void* p, const char* name, bool required, uintptr_t align = 16) {
    if (!p) return required ? fail(NVFP4_EINVAL, "%s must not be NULL", name) : NVFP4_OK;
    if (!aligned(p, align)) return fail(NVFP4_EINVAL, "%s must be %d-byte aligned", name, int(align));
    return NVFP4_OK;
}

int check_shape(int64_t M, int64_t K) {
    if (M < 0 || K < 0) return fail(NVFP4_EINVAL, "M and K must be >= 0 (got %lld, %lld)",
                                    (long long)M, (long long)K);
    if (K % 16 != 0) return fail(NVFP4_EINVAL, "K must be a multiple of 16 (got %lld)", (long long)K);
    if (K > 0 && M > INT64_MAX / 4 / K) return fail(NVFP4_EINVAL, "M*K is too large");
    if (M >= (int64_t{1} << 35) || K >= (int64_t{1} << 35))
        return fail(NVFP4_EINVAL, "M and K must each be below 2^35");
    return NVFP4_OK;
}

bool is_row_mode(int g) { return g == NVFP4_GAMAX_ROW || g == NVFP4_GAMAX_ROW_GIVEN; }

// Largest K with a columnwise output: 65535 CTA columns of 256 (1x16 row-owner
// kernel; the tile kernels cover 512 columns per CTA column).
constexpr int64_t kMaxColwiseK = 65535LL * 256;

// Checks shared by quantize and qdq.
int check_quant(const void* x, int64_t M, int64_t K, int dtype, int block, int rounding,
                const float* residual, int gamax_mode, const float* gamax, int err_mode,
                float bound, bool colwise) {
    int rc = check_shape(M, K);
    if (rc) return rc;
    if (dtype != NVFP4_F32 && dtype != NVFP4_BF16) return fail(NVFP4_EINVAL, "bad dtype %d", dtype);
    if (block != NVFP4_BLOCK_1X16 && block != NVFP4_BLOCK_16X16) return fail(NVFP4_EINVAL, "bad block %d", block);
    if (rounding != NVFP4_RTN && rounding != NVFP4_SR && rounding != NVFP4_RTN_STD)
        return fail(NVFP4_EINVAL, "bad rounding %d", rounding);
    if (gamax_mode < NVFP4_GAMAX_NONE || gamax_mode > NVFP4_GAMAX_ROW_GIVEN)
        return fail(NVFP4_EINVAL, "bad gamax_mode %d", gamax_mode);
    if (err_mode < NVFP4_ERR_NONE || err_mode > NVFP4_ERR_MSE) return fail(NVFP4_EINVAL, "bad err_mode %d", err_mode);
    if (!(bound > 0.0f && bound <= 448.0f)) return fail(NVFP4_EINVAL, "scale_bound must be in (0, 448]");
    if ((block == NVFP4_BLOCK_16X16 || colwise) && M % 16 != 0)
        return fail(NVFP4_EINVAL, "16x16 blocks and columnwise output need M %% 16 == 0");
    if (is_row_mode(gamax_mode) && (block == NVFP4_BLOCK_16X16 || colwise))
        return fail(NVFP4_EINVAL, "per-row global scales allow 1x16 rowwise output only");
    if (err_mode != NVFP4_ERR_NONE) {
        if (rounding != NVFP4_RTN)
            return fail(NVFP4_EINVAL, "four-over-six is round-to-nearest with its own scale association only");
        if (residual) return fail(NVFP4_EINVAL, "four-over-six takes no residual");
        if (gamax_mode == NVFP4_GAMAX_NONE) return fail(NVFP4_EINVAL, "four-over-six needs a global amax");
        if (bound != 256.0f && bound != 448.0f) return fail(NVFP4_EINVAL, "four-over-six bound must be 256 or 448");
    }
    if (colwise && residual) return fail(NVFP4_EINVAL, "columnwise output takes no residual");
    if (colwise && K > kMaxColwiseK)            // the columnwise kernels' grid spans K along y
        return fail(NVFP4_EINVAL, "columnwise output needs K <= %lld", static_cast<long long>(kMaxColwiseK));
    const bool any = M > 0 && K > 0;
    if ((rc = check_ptr(x, "x", any))) return rc;
    if ((rc = check_ptr(residual, "residual", false))) return rc;
    if ((rc = check_ptr(gamax, "gamax", gamax_mode != NVFP4_GAMAX_NONE && (any || gamax_mode == NVFP4_GAMAX_TENSOR ||
                                                                        (gamax_mode == NVFP4_GAMAX_ROW && M > 0)), 4)))
        return rc;
    return NVFP4_OK;
}

// The amax pass (TENSOR / ROW) then the quantize kernel with the amax given.
int run_quant(nvfp4::QuantArgs a, float* gamax, void* stream) {
    int err;
    a.pk = nvfp4::philox_keys(a.seed, a.step);
    if (a.gamax_mode == NVFP4_GAMAX_TENSOR || a.gamax_mode == NVFP4_GAMAX_ROW) {
        err = nvfp4::launch_amax(a.x, a.M, a.K, a.dtype, a.residual, a.gamax_mode, gamax, stream);
        if (err) return cuda_fail(err, "amax launch");
        a.gamax_mode = a.gamax_mode == NVFP4_GAMAX_TENSOR ? NVFP4_GAMAX_TENSOR_GIVEN : NVFP4_GAMAX_ROW_GIVEN;
    }
    if (a.M == 0 || a.K == 0) return NVFP4_OK;
    err = a.codes_col ? nvfp4::launch_quantize_tiles(a, stream) : nvfp4::launch_quantize_rows(a, stream);
    if (err) return cuda_fail(err, "quantize launch");
    return NVFP4_OK;
}

}  // namespace

extern "C" {

int nvfp4_quantize(const void* x, int64_t M, int64_t K, int dtype, int block, int rounding,
                   float* residual, uint64_t seed, uint64_t step, int64_t row_offset,
                   int gamax_mode, float* gamax, int err_mode, float scale_bound,
                   uint8_t* codes, uint8_t* scales, uint8_t* codes_col, uint8_t* scales_col,
                   cudaStream_t stream) {
    g_msg[0] = '\0';
    if ((codes_col == nullptr) != (scales_col == nullptr))
        return fail(NVFP4_EINVAL, "give both codes_col and scales_col, or neither");
    const bool colwise = codes_col != nullptr;
    int rc = check_quant(x, M, K, dtype, block, rounding, residual, gamax_mode, gamax, err_mode,
                         scale_bound, colwise);
    if (rc) return rc;
    const bool any = M > 0 && K > 0;
    if ((rc = check_ptr(codes, "codes", any))) return rc;
    if ((rc = check_ptr(scales, "scales", any))) return rc;
    if ((rc = check_ptr(codes_col, "codes_col", false))) return rc;
    if ((rc = check_ptr(scales_col, "scales_col", false))) return rc;
    nvfp4::QuantArgs a{x, M, K, dtype, block, rounding, residual, seed, step, row_offset,
                       gamax_mode, gamax, err_mode, scale_bound, codes, scales, codes_col,
                       scales_col, nullptr};
    return run_quant(a, gamax, stream);
}

int nvfp4_qdq(const void* x, int64_t M, int64_t K, int dtype, int block, int rounding,
              float* residual, uint64_t seed, uint64_t step, int64_t row_offset,
              int gamax_mode, float* gamax, int err_mode, float scale_bound,
              uint8_t* codes, uint8_t* scales, void* out_bf16, cudaStream_t stream) {
    g_msg[0] = '\0';
    int rc = check_quant(x, M, K, dtype, block, rounding, residual, gamax_mode, gamax, err_mode,
                         scale_bound, false);
    if (rc) return rc;
    const bool any = M > 0 && K > 0;
    if ((rc = check_ptr(codes, "codes", false))) return rc;
    if ((rc = check_ptr(scales, "scales", false))) return rc;
    if ((rc = check_ptr(out_bf16, "out_bf16", any))) return rc;
    nvfp4::QuantArgs a{x, M, K, dtype, block, rounding, residual, seed, step, row_offset,
                       gamax_mode, gamax, err_mode, scale_bound, codes, scales, nullptr, nullptr,
                       static_cast<uint16_t*>(out_bf16)};
    return run_quant(a, gamax, stream);
}

int nvfp4_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t M, int64_t K,
                     int gamax_mode, const float* gamax, float scale_bound, void* out,
                     int out_dtype, cudaStream_t stream) {
    g_msg[0] = '\0';
    int rc = check_shape(M, K);
    if (rc) return rc;
    if (gamax_mode < NVFP4_GAMAX_NONE || gamax_mode > NVFP4_GAMAX_ROW_GIVEN)
        return fail(NVFP4_EINVAL, "bad gamax_mode %d", gamax_mode);
    if (out_dtype != NVFP4_F32 && out_dtype != NVFP4_BF16) return fail(NVFP4_EINVAL, "bad out_dtype %d", out_dtype);
    if (!(scale_bound > 0.0f && scale_bound <= 448.0f)) return fail(NVFP4_EINVAL, "scale_bound must be in (0, 448]");
    const bool any = M > 0 && K > 0;
    if ((rc = check_ptr(codes, "codes", any))) return rc;
    if ((rc = check_ptr(scales, "scales", any))) return rc;
    if ((rc = check_ptr(out, "out", any))) return rc;
    if ((rc = check_ptr(gamax, "gamax", any && gamax_mode != NVFP4_GAMAX_NONE, 4))) return rc;
    nvfp4::DequantArgs a{codes, scales, M, K, gamax_mode, gamax, scale_bound, out, out_dtype};
    const int err = nvfp4::launch_dequantize(a, stream);
    if (err) return cuda_fail(err, "dequantize launch");
    return NVFP4_OK;
}

int nvfp4_amax(const void* x, int64_t M, int64_t K, int dtype, const float* residual, int mode,
               float* out, cudaStream_t stream) {
    g_msg[0] = '\0';
    int rc = check_shape(M, K);
    if (rc) return rc;
    if (dtype != NVFP4_F32 && dtype != NVFP4_BF16) return fail(NVFP4_EINVAL, "bad dtype %d", dtype);
    if (mode != NVFP4_GAMAX_TENSOR && mode != NVFP4_GAMAX_ROW)
        return fail(NVFP4_EINVAL, "amax mode must be NVFP4_GAMAX_TENSOR or NVFP4_GAMAX_ROW");
    const bool any = M > 0 && K > 0;
    if ((rc = check_ptr(x, "x", any))) return rc;
    if ((rc = check_ptr(residual, "residual", false))) return rc;
    if ((rc = check_ptr(out, "out", mode == NVFP4_GAMAX_TENSOR || M > 0, 4))) return rc;
    const int err = nvfp4::launch_amax(x, M, K, dtype, residual, mode, out, stream);
    if (err) return cuda_fail(err, "amax launch");
    return NVFP4_OK;
}

int nvfp4_scales_to_mma(const uint8_t* scales, int64_t rows, int64_t cols, uint8_t* out, cudaStream_t stream) {
    g_msg[0] = '\0';
    if (rows < 0 || cols < 0) return fail(NVFP4_EINVAL, "rows and cols must be >= 0");
    const bool any = rows > 0 && cols > 0;
    int rc;
    if ((rc = check_ptr(scales, "scales", any, 1))) return rc;
    if ((rc = check_ptr(out, "out", any, 4))) return rc;
    if (!any) return NVFP4_OK;
    const int err = nvfp4::launch_scales_mma(scales, rows, cols, out, stream);
    if (err) return cuda_fail(err, "scale layout launch");
    return NVFP4_OK;
}

int nvfp4_mm(const uint8_t* codes_a, const uint8_t* scales_a, const uint8_t* codes_b, const uint8_t* scales_b,
             int64_t M, int64_t N, int64_t K, const float* gamax_a, const float* gamax_b, float scale_bound,
             void* out, int out_dtype, cudaStream_t stream) {
    g_msg[0] = '\0';
    if (M < 0 || N < 0 || K < 0) return fail(NVFP4_EINVAL, "M, N and K must be >= 0");
    if (M % 128 || N % 128 || K % 64)
        return fail(NVFP4_EINVAL, "nvfp4_mm needs M %% 128 == 0, N %% 128 == 0 and K %% 64 == 0");
    if (out_dtype != NVFP4_F32 && out_dtype != NVFP4_BF16) return fail(NVFP4_EINVAL, "bad out_dtype %d", out_dtype);
    if (!(scale_bound > 0.0f && scale_bound <= 448.0f)) return fail(NVFP4_EINVAL, "scale_bound must be in (0, 448]");
    const bool any = M > 0 && N > 0;
    const bool anyk = any && K > 0;
    int rc;
    if ((rc = check_ptr(codes_a, "codes_a", anyk))) return rc;
    if ((rc = check_ptr(scales_a, "scales_a", anyk))) return rc;
    if ((rc = check_ptr(codes_b, "codes_b", anyk))) return rc;
    if ((rc = check_ptr(scales_b, "scales_b", anyk))) return rc;
    if ((rc = check_ptr(gamax_a, "gamax_a", false, 4))) return rc;
    if ((rc = check_ptr(gamax_b, "gamax_b", false, 4))) return rc;
    if ((rc = check_ptr(out, "out", any))) return rc;
    if (!any) return NVFP4_OK;
    if (K == 0) {
        const size_t bytes = static_cast<size_t>(M) * static_cast<size_t>(N) * (out_dtype == NVFP4_F32 ? 4 : 2);
        const int err = static_cast<int>(cudaMemsetAsync(out, 0, bytes, static_cast<cudaStream_t>(stream)));
        return err ? cuda_fail(err, "mm zero fill") : NVFP4_OK;
    }
    const int err = nvfp4::launch_mm(codes_a, scales_a, codes_b, scales_b, M, N, K, gamax_a, gamax_b, scale_bound,
                                     out, out_dtype, stream);
    if (err) return cuda_fail(err, "mm launch");
    return NVFP4_OK;
}

int nvfp4_global_scales(const float* gamax, int64_t n, float scale_bound, float* s_enc, float* s_dec,
                        cudaStream_t stream) {
    g_msg[0] = '\0';
    if (n < 0) return fail(NVFP4_EINVAL, "n must be >= 0");
    if (!(scale_bound > 0.0f && scale_bound <= 448.0f)) return fail(NVFP4_EINVAL, "scale_bound must be in (0, 448]");
    int rc;
    if ((rc = check_ptr(gamax, "gamax", n > 0, 4))) return rc;
    if ((rc = check_ptr(s_enc, "s_enc", false, 4))) return rc;
    if ((rc = check_ptr(s_dec, "s_dec", false, 4))) return rc;
    if (n > 0 && !s_enc && !s_dec) return fail(NVFP4_EINVAL, "give s_enc, s_dec or both");
    const int err = nvfp4::launch_global_scales(gamax, n, scale_bound, s_enc, s_dec, stream);
    if (err) return cuda_fail(err, "global scales launch");
    return NVFP4_OK;
}

int nvfp4_probe_divide(const float* a, const float* b, float* out, int64_t n, cudaStream_t stream) {
    g_msg[0] = '\0';
    if (n < 0) return fail(NVFP4_EINVAL, "n must be >= 0");
    int rc;
    if ((rc = check_ptr(a, "a", n > 0, 4))) return rc;
    if ((rc = check_ptr(b, "b", n > 0, 4))) return rc;
    if ((rc = check_ptr(out, "out", n > 0, 4))) return rc;
    const int err = nvfp4::launch_probe_divide(a, b, out, n, stream);
    if (err) return cuda_fail(err, "probe launch");
    return NVFP4_OK;
}

int nvfp4_probe_sub_f16(const uint32_t* q, const float* v, float* out, int64_t n, cudaStream_t stream) {
    g_msg[0] = '\0';
    if (n < 0) return fail(NVFP4_EINVAL, "n must be >= 0");
    int rc;
    if ((rc = check_ptr(q, "q", n > 0, 4))) return rc;
    if ((rc = check_ptr(v, "v", n > 0, 4))) return rc;
    if ((rc = check_ptr(out, "out", n > 0, 4))) return rc;
    const int err = nvfp4::launch_probe_sub_f16(q, v, out, n, stream);
    if (err) return cuda_fail(err, "probe launch");
    return NVFP4_OK;
}

int nvfp4_probe_e2m1(uint32_t first, int64_t n, uint8_t* out, cudaStream_t stream) {
    g_msg[0] = '\0';
    if (n < 0 || n > (int64_t{1} << 32)) return fail(NVFP4_EINVAL, "n must be in [0, 2^32]");
    if (static_cast<uint64_t>(first) + static_cast<uint64_t>(n) > (uint64_t{1} << 32))
        return fail(NVFP4_EINVAL, "first + n must not pass 2^32");
    int rc;
    if ((rc = check_ptr(out, "out", n > 0, 4))) return rc;
    const int err = nvfp4::launch_probe_e2m1(first, n, out, stream);
    if (err) return cuda_fail(err, "probe launch");
    return NVFP4_OK;
}

const char* nvfp4_last_error(void) { return g_msg; }

int nvfp4_abi_version(void) { return 100; }

}  // extern "C"
