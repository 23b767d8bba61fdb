/*
 * nvfp4_oracle.h -- plain, slow CPU oracle for NVFP4 block quantization.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this code; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no source with the CUDA path.
 *
 * Every routine is a literal restatement of the method described on three
 * pages, cited as:
 *   [fp4-train]  the page "fp4-train" (sections Usage, API, Method,
 *                Correctness, Requirements and limits);
 *   [4o6 PR]     the page "Add NVFP4 four-over-six (row-wise) quantization to
 *                the training prototype" (sections What, Two load-bearing
 *                numeric details, Validation, CuTe DSL kernel (SM100) / Design,
 *                Bitwise validation, Bench, Follow-up fusions);
 *   [TIBQ]       the abstract of "Stable FP4 Training via Transposition-
 *                Invariant Block Quantization".
 *
 * Arithmetic: IEEE binary32, round-to-nearest-even, no FMA contraction, no
 * flush-to-zero (the pages pin fp32 div.rn / mul.rn / add.rn, [4o6 PR] Design).
 * Decisions that only need exact comparisons are made in binary64, where every
 * quantity involved is exact.
 *
 * All pointers are host pointers.  Layouts match the product library:
 *   x         [M,K] row-major, fp32 or bf16 (raw uint16 bits)
 *   residual  [M,K] fp32, read and overwritten (error feedback)
 *   codes     [M,K/2]  uint8, element 2j in the low nibble, 2j+1 in the high
 *   scales    [M,K/16] uint8 e4m3 (16x16 mode: the tile's byte on each row)
 *   codes_col [K,M/2], scales_col [K,M/16]: the rowwise result for x^T
 */
#ifndef NVFP4_ORACLE_H
#define NVFP4_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* enum values are the same numbers the product header uses, restated here so
 * the two sides share no file */
enum { ORC_F32 = 0, ORC_BF16 = 1 };
enum { ORC_BLOCK_1X16 = 0, ORC_BLOCK_16X16 = 1 };
/* RTN_STD: round to nearest with the standard NVFP4 block-scale association
 * b * (S_enc * (1/6)) instead of (b / 6) * S_enc */
enum { ORC_RTN = 0, ORC_SR = 1, ORC_RTN_STD = 2 };
enum { ORC_GAMAX_NONE = 0, ORC_GAMAX_TENSOR = 1, ORC_GAMAX_ROW = 2,
       ORC_GAMAX_TENSOR_GIVEN = 3, ORC_GAMAX_ROW_GIVEN = 4 };
enum { ORC_ERR_NONE = 0, ORC_ERR_MAE = 1, ORC_ERR_MSE = 2 };

/* ---- scalar codecs ---------------------------------------------------- */
float   orc_e4m3_decode(uint8_t b);              /* exact value of an E4M3FN byte   */
uint8_t orc_e4m3_encode(float s);                /* RN-even, satfinite (max 448)     */
float   orc_e2m1_value(uint8_t code);            /* signed grid value of a 4-bit code */
uint8_t orc_e2m1_encode_rn(float v);             /* nearest grid point, ties to even */
uint8_t orc_e2m1_encode_sr(float v, double u);   /* stochastic, u in [0,1)           */
float   orc_bf16_to_f32(uint16_t h);
uint16_t orc_f32_to_bf16(float f);               /* RN-even                          */

/* ---- counter-based generator ------------------------------------------ */
/* Philox4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, SC'11). */
void  orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);
/* the uniform one element draws: key = seed, counter = (idx/4, step), word idx%4,
 * top 24 bits, scaled by 2^-24 */
double orc_sr_uniform(uint64_t seed, uint64_t step, uint64_t idx);

/* ---- global scale ------------------------------------------------------ */
void  orc_global_scales(float A, float bound, float* S_enc, float* S_dec);

/* amax of |x (+ residual)| over the tensor (mode TENSOR, 1 value) or per row
 * (mode ROW, M values); NaN dropped, empty/all-NaN gives +0 */
void  orc_amax(const void* x, int64_t M, int64_t K, int dtype, const float* residual,
               int mode, float* out);

/* ---- the three calls ---------------------------------------------------- */
/* returns 0 on success, 1 on an argument the method does not define */
int orc_quantize(const void* x, int64_t M, int64_t K, int dtype, int block, int rounding,
                 float* residual, uint64_t seed, uint64_t step, int64_t row_offset,
                 int gamax_mode, float* gamax, int err_mode, float scale_bound,
                 uint8_t* codes, uint8_t* scales, uint8_t* codes_col, uint8_t* scales_col);

int orc_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t M, int64_t K,
                   int gamax_mode, const float* gamax, float scale_bound,
                   void* out, int out_dtype);

/* quantize, then write dequant(quantize(x)) as bf16; codes/scales may be null */
int orc_qdq(const void* x, int64_t M, int64_t K, int dtype, int block, int rounding,
            float* residual, uint64_t seed, uint64_t step, int64_t row_offset,
            int gamax_mode, float* gamax, int err_mode, float scale_bound,
            uint8_t* codes, uint8_t* scales, uint16_t* out_bf16);

/* scale bytes [rows, cols] -> the block-scaled matrix-multiply layout:
 * rows padded to 128, cols to 4 (zero bytes), 128 x 4 tiles of 512 bytes in
 * row-major tile order, byte (r, c) of a tile at (r % 32) * 16 + (r / 32) * 4 + c
 * ("fp4-train", API: to_fp4_operands, the layout NVFP4 tensor cores read) */
void orc_scales_to_mma(const uint8_t* scales, int64_t rows, int64_t cols, uint8_t* out);

/* batch forms of the scalar codecs */
void orc_e4m3_encode_n(const float* s, int64_t n, uint8_t* out);
void orc_e2m1_encode_rn_n(const float* v, int64_t n, uint8_t* out);
void orc_e2m1_encode_sr_n(const float* v, const double* u, int64_t n, uint8_t* out);
void orc_sr_uniform_n(uint64_t seed, uint64_t step, const uint64_t* idx, int64_t n, double* out);
void orc_f32_to_bf16_n(const float* f, int64_t n, uint16_t* out);

/* codes of the consecutive fp32 bit patterns first .. first + n - 1 */
void orc_e2m1_encode_rn_bits(uint32_t first, int64_t n, uint8_t* out);

/* Worker threads for loops over independent rows, bands, tiles and elements
 * (n <= 0: one per hardware thread); returns the previous count.  The result
 * bytes do not depend on it.  Default 1. */
int orc_set_threads(int n);
int orc_get_threads(void);

/* 1 when subnormal fp32 arithmetic is honoured (no FTZ/DAZ) on this host */
int orc_fp_env_ok(void);

#ifdef __cplusplus
}
#endif
#endif
