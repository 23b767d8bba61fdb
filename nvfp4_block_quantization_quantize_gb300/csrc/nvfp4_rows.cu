// nvfp4_rows.cu -- 1x16 rowwise quantization (and qdq) for sm_103a.
//
// K % 16 == 0, so the 1x16 blocks of a row-major [M,K] tensor are simply the
// consecutive 16-element groups of the flat array: the kernel streams them.
// Each thread owns one block per step, two steps per loop iteration (both
// blocks' loads are issued before either is computed, doubling the bytes in
// flight); one persistent wave of CTAs covers the tensor.  Per block:
// absmax -> (b/6)*S_enc -> E4M3 scale, then either the plain encode (division
// by the decoded scale through an exact reciprocal-and-correction sequence,
// nearest or Philox stochastic rounding) or four-over-six (two candidates,
// per-element error values from the per-tensor candidate table, sequential
// error sums), then codes, the scale byte and, when asked, the error-feedback
// residual and the bf16 dequantized value.
#include "nvfp4_block.cuh"

namespace nvfp4 {
namespace {

constexpr int kThreads = 256;

template <int DT, int ERR, int RND, bool EF, bool GS>
__device__ __forceinline__ void rows_block(const QuantArgs& a, int64_t blk, float* y,
                                           const GScale& g, float C, const Cand* tab,
                                           uint64_t idx_base, int64_t bpr) {
    GScale gb = g;
    if (a.gamax_mode == NVFP4_GAMAX_ROW_GIVEN) {
        gb.A = a.gamax[blk / bpr];
        global_scales(gb.A, a.bound, gb.Senc, gb.Sdec);
    }
    const float b = absmax16(y);
    uint32_t w0, w1, sf;
    float d;
    if (ERR == NVFP4_ERR_NONE) {
        const float s6f = block_s6f<GS>(b, gb.Senc);
        sf = e4m3_encode(min_nd(s6f, 448.0f));
        d = e4m3_decode(sf);
        const float D = GS ? mul_rn(d, gb.Sdec) : d;
        encode_plain16<RND>(y, D, b, idx_base + static_cast<uint64_t>(blk) * 16u, a.seed, a.step,
                            w0, w1);
    } else {
        four_over_six16<ERR, false>(y, b, gb, C, tab, w0, w1, sf, d);
    }
    if (a.codes) reinterpret_cast<uint2*>(a.codes)[blk] = make_uint2(w0, w1);
    if (a.scales) a.scales[blk] = static_cast<uint8_t>(sf);
    if (EF || a.dq_bf16) {
        float dq[16];
        dequant16<GS || ERR != NVFP4_ERR_NONE>(w0, w1, d, gb.Sdec, dq);
        if (EF) {
            float r[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) r[i] = sub_rn(y[i], dq[i]);
            store16_f32(a.residual, blk * 16, r);
        }
        if (a.dq_bf16) store16_bf16(a.dq_bf16, blk * 16, dq);
    }
}

template <int DT, bool EF>
__device__ __forceinline__ void rows_load(const QuantArgs& a, int64_t blk, float* y) {
    load16<DT>(a.x, blk * 16, y);
    if (EF) {
        float r[16];
        load16_f32(a.residual, blk * 16, r);
#pragma unroll
        for (int i = 0; i < 16; ++i) y[i] = add_rn(y[i], r[i]);
    }
}

template <int DT, int ERR, int RND, bool EF, bool GS>
__global__ void __launch_bounds__(kThreads) k_rows(const QuantArgs a) {
    __shared__ Cand tab[ERR != NVFP4_ERR_NONE ? 128 : 1];
    const int64_t bpr = a.K / 16;
    const int64_t nblk = a.M * bpr;
    GScale g{0.0f, 1.0f, 1.0f};
    if (a.gamax_mode == NVFP4_GAMAX_TENSOR_GIVEN) {
        g.A = a.gamax[0];
        global_scales(g.A, a.bound, g.Senc, g.Sdec);
    }
    const float C = mul_rn(6.0f, a.bound);
    const Cand* tp = nullptr;
    if (ERR != NVFP4_ERR_NONE && a.gamax_mode == NVFP4_GAMAX_TENSOR_GIVEN) {
        fill_cand_table(tab, g.Sdec, g.A, C);
        tp = tab;
    }
    const uint64_t idx_base = static_cast<uint64_t>(a.row_offset) * static_cast<uint64_t>(a.K);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t blk = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; blk < nblk;
         blk += 2 * stride) {
        const int64_t blk2 = blk + stride;
        float y[16], y2[16];
        rows_load<DT, EF>(a, blk, y);
        if (blk2 < nblk) rows_load<DT, EF>(a, blk2, y2);
        rows_block<DT, ERR, RND, EF, GS>(a, blk, y, g, C, tp, idx_base, bpr);
        if (blk2 < nblk) rows_block<DT, ERR, RND, EF, GS>(a, blk2, y2, g, C, tp, idx_base, bpr);
    }
}

template <typename KernelT>
int launch_wave(KernelT kernel, const QuantArgs& a, int64_t nblk, cudaStream_t s) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    const int64_t want = (nblk + 2 * kThreads - 1) / (2 * kThreads);
    const int64_t cap = static_cast<int64_t>(sm_count()) * per_sm;
    const int grid = static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
    kernel<<<grid, kThreads, 0, s>>>(a);
    return static_cast<int>(cudaGetLastError());
}

template <int DT, bool GS>
int rows_plain(const QuantArgs& a, int64_t nblk, cudaStream_t s) {
    const bool ef = a.residual != nullptr;
    if (a.rounding == NVFP4_RTN)
        return ef ? launch_wave(k_rows<DT, NVFP4_ERR_NONE, NVFP4_RTN, true, GS>, a, nblk, s)
                  : launch_wave(k_rows<DT, NVFP4_ERR_NONE, NVFP4_RTN, false, GS>, a, nblk, s);
    return ef ? launch_wave(k_rows<DT, NVFP4_ERR_NONE, NVFP4_SR, true, GS>, a, nblk, s)
              : launch_wave(k_rows<DT, NVFP4_ERR_NONE, NVFP4_SR, false, GS>, a, nblk, s);
}

template <int DT>
int rows_dispatch(const QuantArgs& a, cudaStream_t s) {
    const int64_t nblk = a.M * (a.K / 16);
    if (a.err_mode == NVFP4_ERR_MAE)
        return launch_wave(k_rows<DT, NVFP4_ERR_MAE, NVFP4_RTN, false, true>, a, nblk, s);
    if (a.err_mode == NVFP4_ERR_MSE)
        return launch_wave(k_rows<DT, NVFP4_ERR_MSE, NVFP4_RTN, false, true>, a, nblk, s);
    return a.gamax_mode == NVFP4_GAMAX_NONE ? rows_plain<DT, false>(a, nblk, s)
                                            : rows_plain<DT, true>(a, nblk, s);
}

}  // namespace

int launch_quantize_rows(const QuantArgs& a, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return a.dtype == NVFP4_BF16 ? rows_dispatch<NVFP4_BF16>(a, s) : rows_dispatch<NVFP4_F32>(a, s);
}

}  // namespace nvfp4
