// nvfp4_quantize.cu -- NVFP4 block quantization kernels for sm_103a.
//
// Two kernels cover every quantize / qdq configuration:
//   k_quant_rows   1x16 blocks, rowwise output only.  A block is 16 consecutive
//                  elements of the row-major tensor (K % 16 == 0), so the
//                  tensor is one flat stream of blocks; each thread owns one
//                  block per grid-stride step.
//   k_quant_tiles  a 16-row band x 256 columns per CTA: 16x16 blocks (the
//                  tile amax and the four-over-six error tree reduce over the
//                  16 lanes that hold the tile's 16 rows), and/or the
//                  columnwise output (x^T's 1x16 or 16x16 blocks) computed
//                  from the same read of x through shared memory.
//
// Method: "fp4-train" (Method: block_absmax/6 e4m3 scale, e2m1 grid, SR with a
// counter-based draw, error feedback) and "Add NVFP4 four-over-six (row-wise)
// quantization to the training prototype" (What; CuTe DSL kernel (SM100),
// Design: the (b/6)*S_enc association, encode reciprocals, the 6*bound error
// denominator, sequential per-group error sums, the width-16 tree, strict
// err4 < err6 selection).
#include "nvfp4_device.cuh"

namespace nvfp4 {
namespace {

constexpr int kThreads = 256;
constexpr unsigned kFull = 0xFFFFFFFFu;

// map-to-6 scale: s6f = (b / 6) * S_enc, sf6 = E4M3(min(s6f, 448))
__device__ __forceinline__ void map6_scale(float b, float Senc, float& s6f, uint32_t& sf6,
                                           float& d6) {
    s6f = mul_rn(div_rn(b, 6.0f), Senc);
    sf6 = e4m3_encode(min_nd(s6f, 448.0f));
    d6 = e4m3_decode(sf6);
}

// map-to-4 scale: the pre-rounding scale expanded by exactly 1.5x
__device__ __forceinline__ void map4_scale(float s6f, uint32_t& sf4, float& d4) {
    sf4 = e4m3_encode(min_nd(mul_rn(s6f, 1.5f), 448.0f));
    d4 = e4m3_decode(sf4);
}

// Plain path: v = y / D per element, RN or SR; a zero divisor zeroes the block.
template <int RND>
__device__ __forceinline__ void encode_plain16(const float* y, float D, uint64_t idx0,
                                               uint64_t seed, uint64_t step, uint32_t& w0,
                                               uint32_t& w1) {
    if (RND == NVFP4_RTN) {
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = div_rn(y[i], D);
        w0 = e2m1_encode8(v);
        w1 = e2m1_encode8(v + 8);
    } else {
        uint32_t wd[16];
        sr_words16(idx0, seed, step, wd);
        w0 = 0;
        w1 = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            w0 |= e2m1_encode_sr(div_rn(y[i], D), wd[i]) << (4 * i);
            w1 |= e2m1_encode_sr(div_rn(y[8 + i], D), wd[8 + i]) << (4 * i);
        }
    }
    if (D == 0.0f) {
        w0 = 0;
        w1 = 0;
    }
}

// One four-over-six candidate over 16 values: codes of y * enc and the error
// sum of ((q*d)*A)/C against y, added in element order from 0.
template <int ERR>
__device__ __forceinline__ float candidate16(const float* y, float d, float Sdec, float A,
                                             float C, uint32_t& w0, uint32_t& w1) {
    const float enc = min_nd(div_rn(1.0f, mul_rn(d, Sdec)), FLT_MAX);
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = mul_rn(y[i], enc);
    w0 = e2m1_encode8(v);
    w1 = e2m1_encode8(v + 8);
    float q[16];
    e2m1_decode8(w0, q);
    e2m1_decode8(w1, q + 8);
    float E = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float dq = div_rn(mul_rn(mul_rn(q[i], d), A), C);
        const float diff = sub_rn(dq, y[i]);
        const float e = (ERR == NVFP4_ERR_MAE) ? fabsf(diff) : mul_rn(diff, diff);
        E = add_rn(E, e);
    }
    return E;
}

// Width-16 tree over the 16 lanes of a half warp, broadcast to all of them:
// (((e0+e8)+(e4+e12))+((e2+e10)+(e6+e14))) + (((e1+e9)+(e5+e13))+((e3+e11)+(e7+e15))).
// The xor butterfly forms exactly these pairs (in commuted order on some lanes).
__device__ __forceinline__ float tree16(float E) {
    E = add_rn(E, __shfl_xor_sync(kFull, E, 8));
    E = add_rn(E, __shfl_xor_sync(kFull, E, 4));
    E = add_rn(E, __shfl_xor_sync(kFull, E, 2));
    E = add_rn(E, __shfl_xor_sync(kFull, E, 1));
    return E;
}

__device__ __forceinline__ float max16(float m) {
    m = max_nd(m, __shfl_xor_sync(kFull, m, 8));
    m = max_nd(m, __shfl_xor_sync(kFull, m, 4));
    m = max_nd(m, __shfl_xor_sync(kFull, m, 2));
    m = max_nd(m, __shfl_xor_sync(kFull, m, 1));
    return m;
}

// dequantized value (q * d) * S_dec
__device__ __forceinline__ void dequant16(uint32_t w0, uint32_t w1, float d, float Sdec, float* dq) {
    float q[16];
    e2m1_decode8(w0, q);
    e2m1_decode8(w1, q + 8);
#pragma unroll
    for (int i = 0; i < 16; ++i) dq[i] = mul_rn(mul_rn(q[i], d), Sdec);
}

// Quantize one 16-value group whose block amax is b.  TREE: reduce the
// candidate errors over the half warp (16x16 blocks).
template <int ERR, int RND, bool TREE>
__device__ __forceinline__ void quantize_group(const float* y, float b, float A, float Senc,
                                               float Sdec, float C, uint64_t idx0, uint64_t seed,
                                               uint64_t step, uint32_t& w0, uint32_t& w1,
                                               uint32_t& sf, float& d) {
    float s6f, d6;
    uint32_t sf6;
    map6_scale(b, Senc, s6f, sf6, d6);
    if (ERR == NVFP4_ERR_NONE) {
        encode_plain16<RND>(y, mul_rn(d6, Sdec), idx0, seed, step, w0, w1);
        sf = sf6;
        d = d6;
    } else {
        uint32_t sf4;
        float d4;
        map4_scale(s6f, sf4, d4);
        uint32_t a0, a1, c0, c1;
        float E6 = candidate16<ERR>(y, d6, Sdec, A, C, a0, a1);
        float E4 = candidate16<ERR>(y, d4, Sdec, A, C, c0, c1);
        if (TREE) {
            E6 = tree16(E6);
            E4 = tree16(E4);
        }
        const bool pick4 = E4 < E6;   // ties and NaN keep map-to-6
        w0 = pick4 ? c0 : a0;
        w1 = pick4 ? c1 : a1;
        sf = pick4 ? sf4 : sf6;
        d = pick4 ? d4 : d6;
    }
}

// ---------------------------------------------------------------------------------------------
template <int DT, int ERR, int RND, bool EF>
__global__ void __launch_bounds__(kThreads) k_quant_rows(const QuantArgs a) {
    const int64_t bpr = a.K / 16;
    const int64_t nblk = a.M * bpr;
    float A = 0.0f, Senc = 1.0f, Sdec = 1.0f;
    if (a.gamax_mode == NVFP4_GAMAX_TENSOR_GIVEN) {
        A = a.gamax[0];
        global_scales(A, a.bound, Senc, Sdec);
    }
    const float C = mul_rn(6.0f, a.bound);
    const uint64_t idx_base = static_cast<uint64_t>(a.row_offset) * static_cast<uint64_t>(a.K);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t blk = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; blk < nblk;
         blk += stride) {
        const int64_t e0 = blk * 16;
        float y[16];
        load16<DT>(a.x, e0, y);
        if (EF) {
            float r[16];
            load16_f32(a.residual, e0, r);
#pragma unroll
            for (int i = 0; i < 16; ++i) y[i] = add_rn(y[i], r[i]);
        }
        float Ab = A, Se = Senc, Sd = Sdec;
        if (a.gamax_mode == NVFP4_GAMAX_ROW_GIVEN) {
            Ab = a.gamax[blk / bpr];
            global_scales(Ab, a.bound, Se, Sd);
        }
        float b = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) b = max_nd(b, fabsf(y[i]));
        uint32_t w0, w1, sf;
        float d;
        quantize_group<ERR, RND, false>(y, b, Ab, Se, Sd, C, idx_base + static_cast<uint64_t>(e0),
                                        a.seed, a.step, w0, w1, sf, d);
        if (a.codes) reinterpret_cast<uint2*>(a.codes)[blk] = make_uint2(w0, w1);
        if (a.scales) a.scales[blk] = static_cast<uint8_t>(sf);
        if (EF || a.dq_bf16) {
            float dq[16];
            dequant16(w0, w1, d, Sd, dq);
            if (EF) {
                float r[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) r[i] = sub_rn(y[i], dq[i]);
                store16_f32(a.residual, e0, r);
            }
            if (a.dq_bf16) store16_bf16(a.dq_bf16, e0, dq);
        }
    }
}

// ---------------------------------------------------------------------------------------------
// CTA = rows [16*band, 16*band+16) x 16-column blocks [16*chunk, 16*chunk+16).
// Thread (warp w, lane l): tile t = 2w + l/16 (its 16-column block), row l%16.
constexpr int kTileCols = 256;
constexpr int kYsStride = kTileCols + 4;

template <int DT, int BLK, int ERR, int RND, bool EF, bool COLW>
__global__ void __launch_bounds__(kThreads) k_quant_tiles(const QuantArgs a) {
    __shared__ float ys[COLW ? 16 * kYsStride : 1];
    const int64_t band = blockIdx.x;
    const int64_t chunk = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = 2 * warp + (lane >> 4);
    const int rr = lane & 15;
    const int64_t nb = a.K / 16;
    const int64_t cb = chunk * 16 + t;
    const bool valid = cb < nb;
    const int64_t row = band * 16 + rr;

    float A = 0.0f, Senc = 1.0f, Sdec = 1.0f;
    if (a.gamax_mode == NVFP4_GAMAX_TENSOR_GIVEN) {
        A = a.gamax[0];
        global_scales(A, a.bound, Senc, Sdec);
    }
    const float C = mul_rn(6.0f, a.bound);

    // ---- rowwise ----
    const int64_t e0 = row * a.K + cb * 16;
    float y[16];
    if (valid) {
        load16<DT>(a.x, e0, y);
        if (EF) {
            float r[16];
            load16_f32(a.residual, e0, r);
#pragma unroll
            for (int i = 0; i < 16; ++i) y[i] = add_rn(y[i], r[i]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) y[i] = 0.0f;
    }
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) m = max_nd(m, fabsf(y[i]));
    if (BLK == NVFP4_BLOCK_16X16) m = max16(m);

    if (BLK == NVFP4_BLOCK_16X16 || !COLW) {
        uint32_t w0, w1, sf;
        float d;
        const uint64_t idx0 =
            (static_cast<uint64_t>(a.row_offset) + static_cast<uint64_t>(row)) *
                static_cast<uint64_t>(a.K) + static_cast<uint64_t>(cb * 16);
        quantize_group<ERR, RND, BLK == NVFP4_BLOCK_16X16>(y, m, A, Senc, Sdec, C, idx0, a.seed,
                                                           a.step, w0, w1, sf, d);
        if (valid) {
            if (a.codes) reinterpret_cast<uint2*>(a.codes)[(row * a.K + cb * 16) / 16] = make_uint2(w0, w1);
            if (a.scales) a.scales[row * nb + cb] = static_cast<uint8_t>(sf);
            if (EF || a.dq_bf16) {
                float dq[16];
                dequant16(w0, w1, d, Sdec, dq);
                if (EF) {
                    float r[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) r[i] = sub_rn(y[i], dq[i]);
                    store16_f32(a.residual, e0, r);
                }
                if (a.dq_bf16) store16_bf16(a.dq_bf16, e0, dq);
            }
        }
    } else {
        // 1x16 rowwise next to a columnwise output
        uint32_t w0, w1, sf;
        float d;
        quantize_group<ERR, NVFP4_RTN, false>(y, m, A, Senc, Sdec, C, 0, 0, 0, w0, w1, sf, d);
        if (valid) {
            if (a.codes) reinterpret_cast<uint2*>(a.codes)[(row * a.K + cb * 16) / 16] = make_uint2(w0, w1);
            if (a.scales) a.scales[row * nb + cb] = static_cast<uint8_t>(sf);
        }
    }

    if (!COLW) return;

    // ---- columnwise: the rowwise quantization of x^T, from the staged tile ----
#pragma unroll
    for (int i = 0; i < 16; ++i) ys[rr * kYsStride + t * 16 + i] = y[i];
    __syncthreads();
    const int j = threadIdx.x;               // column within the chunk; its tile is t again
    const int64_t col = chunk * kTileCols + j;
    float c[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) c[r] = ys[r * kYsStride + j];
    float mc = 0.0f;
#pragma unroll
    for (int r = 0; r < 16; ++r) mc = max_nd(mc, fabsf(c[r]));
    if (BLK == NVFP4_BLOCK_16X16) mc = max16(mc);
    uint32_t w0, w1, sf;
    float d;
    quantize_group<ERR, NVFP4_RTN, BLK == NVFP4_BLOCK_16X16>(c, mc, A, Senc, Sdec, C, 0, 0, 0, w0,
                                                              w1, sf, d);
    if (col < a.K) {
        const int64_t M = a.M;
        reinterpret_cast<uint2*>(a.codes_col)[(col * M + band * 16) / 16] = make_uint2(w0, w1);
        a.scales_col[col * (M / 16) + band] = static_cast<uint8_t>(sf);
    }
}

// ---------------------------------------------------------------------------------------------
template <typename KernelT>
int launch_grid_stride(KernelT kernel, const QuantArgs& a, int64_t nblk, cudaStream_t s) {
    const int64_t want = (nblk + kThreads - 1) / kThreads;
    const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
    const int grid = static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
    kernel<<<grid, kThreads, 0, s>>>(a);
    return static_cast<int>(cudaGetLastError());
}

template <int DT>
int rows_dispatch(const QuantArgs& a, cudaStream_t s) {
    const int64_t nblk = a.M * (a.K / 16);
    const bool ef = a.residual != nullptr;
    if (a.err_mode == NVFP4_ERR_MAE) return launch_grid_stride(k_quant_rows<DT, NVFP4_ERR_MAE, NVFP4_RTN, false>, a, nblk, s);
    if (a.err_mode == NVFP4_ERR_MSE) return launch_grid_stride(k_quant_rows<DT, NVFP4_ERR_MSE, NVFP4_RTN, false>, a, nblk, s);
    if (a.rounding == NVFP4_RTN) {
        return ef ? launch_grid_stride(k_quant_rows<DT, NVFP4_ERR_NONE, NVFP4_RTN, true>, a, nblk, s)
                  : launch_grid_stride(k_quant_rows<DT, NVFP4_ERR_NONE, NVFP4_RTN, false>, a, nblk, s);
    }
    return ef ? launch_grid_stride(k_quant_rows<DT, NVFP4_ERR_NONE, NVFP4_SR, true>, a, nblk, s)
              : launch_grid_stride(k_quant_rows<DT, NVFP4_ERR_NONE, NVFP4_SR, false>, a, nblk, s);
}

template <typename KernelT>
int launch_tiles(KernelT kernel, const QuantArgs& a, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>(a.M / 16),
                    static_cast<unsigned>((a.K / 16 + 15) / 16));
    kernel<<<grid, kThreads, 0, s>>>(a);
    return static_cast<int>(cudaGetLastError());
}

template <int DT, int BLK, bool COLW>
int tiles_dispatch_err(const QuantArgs& a, cudaStream_t s) {
    if (a.err_mode == NVFP4_ERR_MAE) return launch_tiles(k_quant_tiles<DT, BLK, NVFP4_ERR_MAE, NVFP4_RTN, false, COLW>, a, s);
    if (a.err_mode == NVFP4_ERR_MSE) return launch_tiles(k_quant_tiles<DT, BLK, NVFP4_ERR_MSE, NVFP4_RTN, false, COLW>, a, s);
    if (COLW) return launch_tiles(k_quant_tiles<DT, BLK, NVFP4_ERR_NONE, NVFP4_RTN, false, COLW>, a, s);
    const bool ef = a.residual != nullptr;
    if (a.rounding == NVFP4_RTN) {
        return ef ? launch_tiles(k_quant_tiles<DT, BLK, NVFP4_ERR_NONE, NVFP4_RTN, true, false>, a, s)
                  : launch_tiles(k_quant_tiles<DT, BLK, NVFP4_ERR_NONE, NVFP4_RTN, false, false>, a, s);
    }
    return ef ? launch_tiles(k_quant_tiles<DT, BLK, NVFP4_ERR_NONE, NVFP4_SR, true, false>, a, s)
              : launch_tiles(k_quant_tiles<DT, BLK, NVFP4_ERR_NONE, NVFP4_SR, false, false>, a, s);
}

template <int DT>
int tiles_dispatch(const QuantArgs& a, cudaStream_t s) {
    const bool colw = a.codes_col != nullptr;
    if (a.block == NVFP4_BLOCK_16X16) {
        return colw ? tiles_dispatch_err<DT, NVFP4_BLOCK_16X16, true>(a, s)
                    : tiles_dispatch_err<DT, NVFP4_BLOCK_16X16, false>(a, s);
    }
    return tiles_dispatch_err<DT, NVFP4_BLOCK_1X16, true>(a, s);
}

}  // namespace

int launch_quantize_rows(const QuantArgs& a, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return a.dtype == NVFP4_BF16 ? rows_dispatch<NVFP4_BF16>(a, s) : rows_dispatch<NVFP4_F32>(a, s);
}

int launch_quantize_tiles(const QuantArgs& a, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return a.dtype == NVFP4_BF16 ? tiles_dispatch<NVFP4_BF16>(a, s) : tiles_dispatch<NVFP4_F32>(a, s);
}

}  // namespace nvfp4
