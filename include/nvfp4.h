/*
 * nvfp4.h -- C ABI of the GB300 (sm_103a) NVFP4 block quantization library.
 *
 * Sources cited below:
 *   [fp4-train]  the page "fp4-train": sections API (quantize, dequantize, qdq),
 *                Method, Correctness, Requirements and limits.
 *   [4o6 PR]     the page "Add NVFP4 four-over-six (row-wise) quantization to
 *                the training prototype": sections What, Two load-bearing
 *                numeric details, Validation, CuTe DSL kernel (SM100) / Design,
 *                Follow-up fusions.
 *
 * Conventions shared by every call
 *   - Data pointers are DEVICE pointers owned by the caller; the library never
 *     allocates, frees or synchronizes.  Work is enqueued on `stream` (a
 *     cudaStream_t; NULL = the legacy default stream) on the current CUDA
 *     device.
 *   - Layouts are row-major:
 *       x          [M,K]     fp32 or bf16
 *       residual   [M,K]     fp32, read and overwritten in place
 *       codes      [M,K/2]   uint8: element 2j in the low nibble, 2j+1 in the high;
 *                            a code is sign<<3 | k, k indexing {0,.5,1,1.5,2,3,4,6}
 *       scales     [M,K/16]  uint8 E4M3 block scales; in 16x16 mode the tile's
 *                            one scale byte is written on each of its 16 rows
 *       codes_col  [K,M/2], scales_col [K,M/16]: the rowwise quantization of x^T
 *       gamax      1 fp32 (per tensor) or M fp32 (per row)
 *   - Every data pointer must be 16-byte aligned (gamax: 4-byte aligned).
 *     Inputs are never written, except
 *     `residual`.  Outputs must not overlap inputs or each other.
 *   - Return value: NVFP4_OK, NVFP4_EINVAL (bad arguments: checked on the host
 *     before anything is enqueued; outputs untouched) or NVFP4_ECUDA (a CUDA
 *     launch error; outputs undefined).  nvfp4_last_error() returns a message
 *     for the calling thread's last non-OK status.
 *   - M == 0 or K == 0 is a valid empty call (a per-tensor amax of an empty
 *     tensor is +0).  K must be a multiple of 16 [fp4-train, Requirements and
 *     limits]; 16x16 blocks and columnwise outputs also need M % 16 == 0.
 *     M and K are each below 2^35; a columnwise output needs K <= 16776960.
 *
 * Arithmetic: fp32, round-to-nearest-even, correctly rounded division, no
 * fused multiply-add and no flush-to-zero on the pinned steps [4o6 PR, Design].
 */
#ifndef NVFP4_H
#define NVFP4_H

#include <stdint.h>

/* cudaStream_t without the CUDA headers: the same opaque handle type the CUDA
 * runtime declares (a repeated identical typedef is valid C11 and C++). */
#ifndef CUDART_VERSION
typedef struct CUstream_st* cudaStream_t;
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* element type of x (and of dequantize's output) */
enum nvfp4_dtype { NVFP4_F32 = 0, NVFP4_BF16 = 1 };

/* block shape sharing one scale: 1x16 [fp4-train, Method], or a 16x16 tile
 * whose scale is the same for x and x^T [4o6 PR, What; Design] */
enum nvfp4_block { NVFP4_BLOCK_1X16 = 0, NVFP4_BLOCK_16X16 = 1 };

/* element rounding: nearest (ties to even) or stochastic [fp4-train, Method];
 * NVFP4_RTN_STD is nearest rounding with the standard NVFP4 block-scale
 * association b * (S_enc * (1/6)) ("Add NVFP4 four-over-six (row-wise)
 * quantization to the training prototype", Two load-bearing numeric details:
 * the recipe's gradient-side quantizer) instead of (b / 6) * S_enc. */
enum nvfp4_round { NVFP4_RTN = 0, NVFP4_SR = 1, NVFP4_RTN_STD = 2 };

/* global (second-level) scale [4o6 PR, What]:
 *   NONE          S_enc = S_dec = 1 (the fp4-train recipe); gamax unused
 *   TENSOR        A = max |y| over the tensor is computed and written to gamax[0]
 *   ROW           A_r = max |y| over row r is computed and written to gamax[r]
 *   TENSOR_GIVEN  A is read from gamax[0] (the caller's amax)
 *   ROW_GIVEN     A_r is read from gamax[r]
 * Then S_enc = min(6*bound / A, FLT_MAX), or 1 if A is not a positive finite
 * number; S_dec = 1 / S_enc.  NaN is dropped from every amax. */
enum nvfp4_gamax {
    NVFP4_GAMAX_NONE = 0,
    NVFP4_GAMAX_TENSOR = 1,
    NVFP4_GAMAX_ROW = 2,
    NVFP4_GAMAX_TENSOR_GIVEN = 3,
    NVFP4_GAMAX_ROW_GIVEN = 4
};

/* NONE: the plain quantizer (map-to-6 only).  MAE / MSE: four-over-six, keeping
 * per block whichever of map-to-6 and map-to-4 has the lower error [4o6 PR, What] */
enum nvfp4_err { NVFP4_ERR_NONE = 0, NVFP4_ERR_MAE = 1, NVFP4_ERR_MSE = 2 };

enum nvfp4_status { NVFP4_OK = 0, NVFP4_EINVAL = 1, NVFP4_ECUDA = 2 };

/*
 * nvfp4_quantize -- [fp4-train, API] quantize(x, stochastic, residual, seed,
 * step) and [4o6 PR, What] four_over_six_quantize(x, global_amax, block,
 * err_mode, e4m3_scale_bound), as one call.
 *
 * Per block of y = x (+ residual when residual != NULL):
 *   b    = max |y| over the block (NaN dropped)
 *   s6f  = (b / 6) * S_enc;  sf6 = E4M3(min(s6f, 448))              [fp4-train, Method]
 *        (NVFP4_RTN_STD: s6f = b * (S_enc * (1/6)), 1/6 the nearest fp32)
 *   plain (err_mode NONE): code = round(y / (dec(sf6) * S_dec)), nearest or
 *        stochastic with the Philox4x32-10 draw keyed on (seed, step, global
 *        index (row_offset + r) * K + c) of the element in x -- for the
 *        columnwise output too, so x and x^T round each element alike
 *        ("Stable FP4 Training via Transposition-Invariant Block
 *        Quantization", abstract); a zero scale gives zero codes.
 *   four-over-six (MAE/MSE): also sf4 = E4M3(min(1.5 * s6f, 448)); each
 *        candidate encodes y * min(1/(dec(sf)*S_dec), FLT_MAX) and is scored by
 *        the error of ((q*dec(sf))*A)/(6*bound) against y, summed in element
 *        order (16x16: the fixed width-16 tree over row sums); map-to-4 wins
 *        only when strictly better [4o6 PR, What; Design].
 *   residual: overwritten with y - (q*dec(sf))*S_dec                   [fp4-train, Method]
 *
 * Arguments
 *   x            device [M,K], dtype F32 or BF16
 *   block        NVFP4_BLOCK_1X16 or NVFP4_BLOCK_16X16
 *   rounding     NVFP4_RTN, NVFP4_SR or NVFP4_RTN_STD
 *   residual     NULL or device [M,K] fp32 (error feedback, in place)
 *   seed, step   SR key and step (unused by RTN)
 *   row_offset   global row index of x's row 0 (SR counter base; 0 for a
 *                whole tensor, the shard's first row for a row shard)
 *   gamax_mode   an nvfp4_gamax value; gamax is device fp32 [1] or [M]
 *                (written for TENSOR / ROW, read for *_GIVEN, unused for NONE)
 *   err_mode     an nvfp4_err value
 *   scale_bound  (0, 448] for the plain path; 256 or 448 for four-over-six
 *   codes/scales device outputs [M,K/2] / [M,K/16] (both required)
 *   codes_col/scales_col  NULL, or device outputs [K,M/2] / [K,M/16]: the
 *                quantization of x^T from the same read of x
 *
 * EINVAL when: M < 0, K < 0 or K % 16 != 0; M % 16 != 0 with 16x16 or a
 * columnwise output; a required pointer is NULL or a pointer is not 16-byte
 * aligned; an enum is out of range; ROW modes with 16x16 or columnwise
 * (a row-scaled tensor has no columnwise form [4o6 PR, What]); four-over-six
 * with SR or RTN_STD, a residual, gamax NONE or a bound other than 256/448
 * (the recipe is nearest-rounding only [4o6 PR, What]); columnwise with a
 * residual (one residual cannot serve two quantizations); a bound outside
 * (0, 448]; only one of codes_col / scales_col given; a columnwise output
 * with K > 16776960.
 */
int nvfp4_quantize(const void* x, int64_t M, int64_t K, int dtype, int block, int rounding,
                   float* residual, uint64_t seed, uint64_t step, int64_t row_offset,
                   int gamax_mode, float* gamax, int err_mode, float scale_bound,
                   uint8_t* codes, uint8_t* scales, uint8_t* codes_col, uint8_t* scales_col,
                   cudaStream_t stream);

/*
 * nvfp4_dequantize -- [fp4-train, API] dequantize(packed, scale, M, K):
 * out[r,c] = (q * dec(scale)) * S_dec, with S_dec from gamax as above
 * (TENSOR and TENSOR_GIVEN read gamax[0]; ROW and ROW_GIVEN read gamax[r];
 * NONE uses 1).  out is device [M,K], out_dtype BF16 (nearest-even) or F32.
 * EINVAL on bad shapes, NULL or misaligned pointers, bad enums or bound.
 */
int nvfp4_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t M, int64_t K,
                     int gamax_mode, const float* gamax, float scale_bound,
                     void* out, int out_dtype, cudaStream_t stream);

/*
 * nvfp4_qdq -- [fp4-train, API] qdq(x, stochastic, residual, seed, step):
 * quantize, then write the dequantized value as bf16 to out_bf16 [M,K], in one
 * pass.  Arguments as nvfp4_quantize (rowwise only); codes and scales may be
 * NULL when only the dequantized tensor is wanted.
 */
int nvfp4_qdq(const void* x, int64_t M, int64_t K, int dtype, int block, int rounding,
              float* residual, uint64_t seed, uint64_t step, int64_t row_offset,
              int gamax_mode, float* gamax, int err_mode, float scale_bound,
              uint8_t* codes, uint8_t* scales, void* out_bf16, cudaStream_t stream);

/*
 * nvfp4_amax -- the global amax step on its own [4o6 PR, What; Design]:
 * max |x (+ residual)| with NaN dropped, over the tensor (mode
 * NVFP4_GAMAX_TENSOR, writes out[0]) or per row (NVFP4_GAMAX_ROW, out[M]).
 * residual may be NULL.
 */
int nvfp4_amax(const void* x, int64_t M, int64_t K, int dtype, const float* residual,
               int mode, float* out, cudaStream_t stream);

/*
 * nvfp4_global_scales -- the global encode / decode scales of n global amaxes
 * ("Add NVFP4 four-over-six (row-wise) quantization to the training
 * prototype", What and Design): S_enc[i] = min(6*bound / gamax[i], FLT_MAX),
 * or 1 when gamax[i] is not a positive finite number, and S_dec[i] = 1 /
 * S_enc[i] (IEEE divisions) -- the values every quantize and dequantize call
 * uses, for consumers that apply the decode scale themselves (a block-scaled
 * matrix multiply multiplies its result by S_dec(A) * S_dec(B)).
 * gamax, s_enc, s_dec: device fp32 [n] (4-byte aligned); s_enc or s_dec may be
 * NULL (not both when n > 0).  EINVAL on n < 0, a bound outside (0, 448] or
 * bad pointers.
 */
int nvfp4_global_scales(const float* gamax, int64_t n, float scale_bound, float* s_enc, float* s_dec,
                        cudaStream_t stream);

/*
 * nvfp4_scales_to_mma -- re-lay a row-major scale matrix [rows, cols] (one
 * E4M3 byte per 16 elements along K: cols = K/16) out in the layout the
 * block-scaled tensor-core matrix multiply reads ("fp4-train", API:
 * to_fp4_operands returns "the layout NVFP4 tensor cores read"; the format is
 * the block-scaling-factor layout of NVIDIA's public cuBLAS documentation):
 *   rows padded to R = 128 * ceil(rows/128), cols to C = 4 * ceil(cols/4),
 *   padding bytes 0; 128 x 4 tiles of 512 bytes, tile (rt, ct) at byte
 *   (rt * C/4 + ct) * 512; inside a tile, byte (r, c) at
 *   (r % 32) * 16 + (r / 32) * 4 + c.
 * scales  device [rows, cols] bytes;  out  device [R * C] bytes (caller-owned).
 * EINVAL when rows < 0, cols < 0, or a pointer is NULL (with rows, cols > 0).
 */
int nvfp4_scales_to_mma(const uint8_t* scales, int64_t rows, int64_t cols, uint8_t* out, cudaStream_t stream);

/*
 * nvfp4_mm -- out = (A B^T) * S_dec(A) * S_dec(B) on the block-scaled FP4
 * tensor cores ("fp4-train", API: fp4_mm, a @ b^T on the NVFP4 tensor cores;
 * Correctness: the tensor-core result agrees with the dequantize path).
 *   codes_a [M, K/2], codes_b [N, K/2]: rowwise 1x16 codes from nvfp4_quantize
 *   scales_a, scales_b: their scale bytes in the nvfp4_scales_to_mma layout
 *   gamax_a, gamax_b: NULL (no global scale) or the per-tensor amax the codes
 *     were made with (device fp32 [1]); scale_bound the bound they used
 *   out: device [M, N], NVFP4_F32 or NVFP4_BF16 (RNE), row-major
 * Products are exact and accumulate in fp32 in tensor memory, 64 K-elements
 * per step.  EINVAL when M % 128, N % 128 or K % 64 is not 0, M, N or K is
 * negative, a pointer is NULL or misaligned (16 bytes; gamax 4), or the bound
 * is outside (0, 448].  A CTA that stops waiting for its tensor-core work
 * writes NaN to its 128 x 128 tile of out.
 */
int nvfp4_mm(const uint8_t* codes_a, const uint8_t* scales_a, const uint8_t* codes_b, const uint8_t* scales_b,
             int64_t M, int64_t N, int64_t K, const float* gamax_a, const float* gamax_b, float scale_bound,
             void* out, int out_dtype, cudaStream_t stream);

/*
 * nvfp4_probe_divide -- diagnostic.  out[i] = a[i] / b[i] computed by the
 * device routine the plain quantizer uses for "every element is divided by the
 * decoded scale" [fp4-train, Method] (its stochastic-rounding form, which must
 * equal IEEE round-to-nearest division for every input; a divisor that is an
 * E4M3 value takes the shorter form used without a global scale).  Device pointers,
 * n >= 0 elements, 4-byte aligned; EINVAL on bad arguments.  It exists so the
 * routine can be checked exhaustively against IEEE division.
 */
int nvfp4_probe_divide(const float* a, const float* b, float* out, int64_t n, cudaStream_t stream);

/*
 * nvfp4_probe_sub_f16 -- diagnostic.  For i < n, out[2i] and out[2i+1] are the
 * low and high f16 halves of q[i] minus v[2i] and v[2i+1], each rounded once to
 * fp32 by the mixed-precision subtract the certified four-over-six error sums
 * use (the grid value of a code, decoded to f16, minus the scaled value the
 * encode rounded; "Add NVFP4 four-over-six (row-wise) quantization to the
 * training prototype", Design: the candidates' errors).  Device pointers: q
 * n words, v and out 2n floats, 4-byte aligned; EINVAL on bad arguments.  It
 * exists so the rounding the sums' error bound assumes can be checked.
 */
int nvfp4_probe_sub_f16(const uint32_t* q, const float* v, float* out, int64_t n, cudaStream_t stream);

/*
 * nvfp4_probe_e2m1 -- diagnostic.  The e2m1 codes that the quantizers' element
 * encode ("fp4-train", Method: each value rounded to the signed grid
 * {0,.5,1,1.5,2,3,4,6}; "Add NVFP4 four-over-six (row-wise) quantization to
 * the training prototype", Design: NaN encodes to +6) gives the n fp32 values
 * whose bit patterns are first, first + 1, ..., first + n - 1, packed two per
 * byte like quantized codes (pattern 2j in the low nibble of byte j; for odd n
 * the last byte's high nibble is 0).  out is
 * device memory of (n + 1) / 2 bytes, 4-byte aligned.  EINVAL when n < 0 or
 * first + n > 2^32.  It exists so the conversion can be checked against the
 * oracle over every fp32 value.
 */
int nvfp4_probe_e2m1(uint32_t first, int64_t n, uint8_t* out, cudaStream_t stream);

/* message for the calling thread's last non-OK status ("" if none) */
const char* nvfp4_last_error(void);

/* ABI version of this header (major * 100 + minor) */
int nvfp4_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4_H */
