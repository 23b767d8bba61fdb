// nvfp4_rows.cu -- 1x16 rowwise quantization (and qdq) for sm_103a.
//
// K % 16 == 0, so the 1x16 blocks of a row-major [M,K] tensor are simply the
// consecutive 16-element groups of the flat array: the kernel streams them.
// Each thread owns one block per grid-stride step and keeps the next three
// steps' bytes in flight with its own asynchronous global->shared copies (a
// per-thread four-stage pipeline: no registers held, no barrier); one
// persistent wave of CTAs covers the tensor.  Per block:
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
                                           const float* rt, uint64_t idx_base, int64_t bpr) {
    GScale gb = g;
    if (a.gamax_mode == NVFP4_GAMAX_ROW_GIVEN) {
        gb.A = a.gamax[blk / bpr];
        global_scales(gb.A, a.bound, gb.Senc, gb.Sdec);
    }
    const float b = absmax16(y);
    uint32_t w0, w1, sf;
    float d, q[16];
    const bool wq = EF || a.dq_bf16;
    constexpr bool QV = ERR == NVFP4_ERR_NONE && RND == NVFP4_SR;   // grid values kept
    if (ERR == NVFP4_ERR_NONE) {
        const float s6f = block_s6f<GS>(b, gb.Senc);
        sf = e4m3_encode(min_nd(s6f, 448.0f));
        d = e4m3_decode(sf);
        const float D = GS ? mul_rn(d, gb.Sdec) : d;
        encode_plain16<RND>(y, D, b, idx_base + static_cast<uint64_t>(blk) * 16u, a.seed, a.step,
                            w0, w1, GS ? nullptr : rt, sf, q, wq);
    } else {
        four_over_six16<ERR, false>(y, b, gb, C, tab, w0, w1, sf, d);
    }
    if (a.codes) reinterpret_cast<uint2*>(a.codes)[blk] = make_uint2(w0, w1);
    if (a.scales) a.scales[blk] = static_cast<uint8_t>(sf);
    if (wq) {
        float dq[16];
        if (QV) dequant_q16<GS>(q, d, gb.Sdec, dq);
        else dequant16<GS || ERR != NVFP4_ERR_NONE>(w0, w1, d, gb.Sdec, dq);
        if (EF) {
            float r[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) r[i] = sub_rn(y[i], dq[i]);
            store16_f32(a.residual, blk * 16, r);
        }
        if (a.dq_bf16) store16_bf16(a.dq_bf16, blk * 16, dq);
    }
}

// Per-thread copy pipeline: stage s holds, for each thread, its block's x
// bytes (and residual bytes under error feedback) for one grid-stride step.
// With a residual a block moves 96-128 bytes, so one step ahead at a higher
// occupancy keeps enough in flight; without, three steps ahead (the stage count is per variant).
template <int DT, bool EF>
struct RowsStage {
    static constexpr int STAGES = EF ? 2 : 4;
    static constexpr int XB = DT == NVFP4_BF16 ? 32 : 64;   // x bytes per block
    static constexpr int RB = EF ? 64 : 0;                    // residual bytes per block
    static constexpr int BYTES = kThreads * (XB + RB);
    static constexpr int TOTAL = STAGES * BYTES;
};

template <int DT, int ERR, int RND, bool EF, bool GS>
__global__ void __launch_bounds__(kThreads) k_rows(const QuantArgs a) {
    using St = RowsStage<DT, EF>;
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ Cand tab[ERR != NVFP4_ERR_NONE ? 128 : 1];
    __shared__ float rtab[(ERR == NVFP4_ERR_NONE && !GS) ? 128 : 1];
    if (ERR == NVFP4_ERR_NONE && !GS) fill_recip_table(rtab);
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
    const int tid = threadIdx.x;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t first = static_cast<int64_t>(blockIdx.x) * blockDim.x + tid;
    unsigned char* xs = smem + tid * St::XB;
    unsigned char* rs = smem + kThreads * St::XB + tid * St::RB;

    auto issue = [&](int64_t blk, int stage) {
        if (blk < nblk) {
            const unsigned char* gx = static_cast<const unsigned char*>(a.x) + blk * St::XB;
#pragma unroll
            for (int c = 0; c < St::XB / 16; ++c) cp_async16(xs + stage * St::BYTES + 16 * c, gx + 16 * c);
            if (EF) {
                const unsigned char* gr = reinterpret_cast<const unsigned char*>(a.residual) + blk * 64;
#pragma unroll
                for (int c = 0; c < 4; ++c) cp_async16(rs + stage * St::BYTES + 16 * c, gr + 16 * c);
            }
        }
        cp_async_commit();
    };

    constexpr int S = St::STAGES;
#pragma unroll
    for (int k = 0; k < S - 1; ++k) issue(first + k * stride, k);
    int stage = 0;
    for (int64_t blk = first; blk < nblk; blk += stride) {
        issue(blk + (S - 1) * stride, stage == 0 ? S - 1 : stage - 1);
        cp_async_wait<S - 1>();
        float y[16];
        lds16<DT>(xs + stage * St::BYTES, y);
        if (EF) {
            float r[16];
            lds16<NVFP4_F32>(rs + stage * St::BYTES, r);
#pragma unroll
            for (int i = 0; i < 16; ++i) y[i] = add_rn(y[i], r[i]);
        }
        rows_block<DT, ERR, RND, EF, GS>(a, blk, y, g, C, tp, rtab, idx_base, bpr);
        stage = stage == S - 1 ? 0 : stage + 1;
    }
    cp_async_wait<0>();
}

template <int DT, int ERR, int RND, bool EF, bool GS>
int launch_rows(const QuantArgs& a, int64_t nblk, cudaStream_t s) {
    auto kernel = k_rows<DT, ERR, RND, EF, GS>;
    constexpr int smem = RowsStage<DT, EF>::TOTAL;
    static thread_local int configured_dev = -1, per_sm = 1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_dev != dev) {
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem) != cudaSuccess ||
            per_sm < 1)
            per_sm = 1;
        configured_dev = dev;
    }
    const int64_t want = (nblk + kThreads - 1) / kThreads;
    const int64_t cap = static_cast<int64_t>(sm_count()) * per_sm;
    const int grid = static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
    kernel<<<grid, kThreads, smem, s>>>(a);
    return static_cast<int>(cudaGetLastError());
}

template <int DT, bool GS>
int rows_plain(const QuantArgs& a, int64_t nblk, cudaStream_t s) {
    const bool ef = a.residual != nullptr;
    if (a.rounding == NVFP4_RTN)
        return ef ? launch_rows<DT, NVFP4_ERR_NONE, NVFP4_RTN, true, GS>(a, nblk, s)
                  : launch_rows<DT, NVFP4_ERR_NONE, NVFP4_RTN, false, GS>(a, nblk, s);
    return ef ? launch_rows<DT, NVFP4_ERR_NONE, NVFP4_SR, true, GS>(a, nblk, s)
              : launch_rows<DT, NVFP4_ERR_NONE, NVFP4_SR, false, GS>(a, nblk, s);
}

template <int DT>
int rows_dispatch(const QuantArgs& a, cudaStream_t s) {
    const int64_t nblk = a.M * (a.K / 16);
    if (a.err_mode == NVFP4_ERR_MAE) return launch_rows<DT, NVFP4_ERR_MAE, NVFP4_RTN, false, true>(a, nblk, s);
    if (a.err_mode == NVFP4_ERR_MSE) return launch_rows<DT, NVFP4_ERR_MSE, NVFP4_RTN, false, true>(a, nblk, s);
    return a.gamax_mode == NVFP4_GAMAX_NONE ? rows_plain<DT, false>(a, nblk, s)
                                            : rows_plain<DT, true>(a, nblk, s);
}

}  // namespace

int launch_quantize_rows(const QuantArgs& a, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return a.dtype == NVFP4_BF16 ? rows_dispatch<NVFP4_BF16>(a, s) : rows_dispatch<NVFP4_F32>(a, s);
}

}  // namespace nvfp4
