// nvfp4_rows.cu -- rowwise quantization (and qdq) for sm_103a: 1x16 blocks
// (k_rows) and 16x16 blocks (k_band16).
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

// The block amax of a 1x16 group is its own absmax.
struct OwnAmax {
    static constexpr bool kSplit = false;
    static constexpr bool failed = false;
    float v;
    __device__ void post(float b) { v = b; }
    __device__ float get() const { return v; }
};

// One 1x16 group y of block-row blk: tile_amax.post(the group's absmax) then
// tile_amax.get() gives its block amax (after_amax() runs right after it),
// and its four-over-six error sums go through tile_sums (identities for 1x16
// blocks; the 16x16 tile's reductions otherwise).  With a split tile amax
// (kSplit) the stochastic-rounding draws, which do not depend on the scale,
// are made between post and get.  Nothing is stored when !live (a group past
// the tensor's last column block).  When the tile amax reports a failed wait
// the block's scale byte is the E4M3 NaN 0x7F (its bf16 output NaN) and
// nothing else is written.
template <int DT, int ERR, int RND, bool EF, bool GS, class TileAmax, class TileSums, class AfterAmax>
__device__ __forceinline__ void rows_block(const QuantArgs& a, int64_t blk, bool live, float* y,
                                           const GScale& g, float C, const O6Tab* tab,
                                           const float* rt, uint64_t idx_base, int64_t bpr,
                                           TileAmax& tile_amax, TileSums tile_sums, AfterAmax after_amax) {
    GScale gb = g;
    if (a.gamax_mode == NVFP4_GAMAX_ROW_GIVEN) {
        gb.A = a.gamax[blk / bpr];
        global_scales(gb.A, a.bound, gb.Senc, gb.Sdec);
    }
    constexpr bool EARLY = TileAmax::kSplit && ERR == NVFP4_ERR_NONE && RND == NVFP4_SR;
    const uint64_t idx0 = idx_base + static_cast<uint64_t>(blk) * 16u;
    tile_amax.post(absmax16(y));
    uint32_t wd[16];
    if constexpr (EARLY) sr_words16(idx0, a.pk, wd);
    const float b = tile_amax.get();
    after_amax();
    uint32_t w0, w1, sf;
    float d, q[16];
    const bool wq = EF || a.dq_bf16;
    constexpr bool QV = ERR == NVFP4_ERR_NONE && RND == NVFP4_SR;   // grid values kept
    if (ERR == NVFP4_ERR_NONE) {
        const float s6f = block_scale<GS>(b, gb.Senc, RND == NVFP4_RTN_STD);
        sf = e4m3_encode(min_nd(s6f, 448.0f));
        d = e4m3_decode(sf);
        const float D = GS ? mul_rn(d, gb.Sdec) : d;
        constexpr bool BF16_E4 = DT == NVFP4_BF16 && !EF && !GS;   // y a bf16 input, D an E4M3 scale
        if constexpr (EARLY)
            encode_plain16_words<RND, BF16_E4>(y, D, b, wd, w0, w1, GS ? nullptr : rt, sf, q, wq);
        else
            encode_plain16<RND, BF16_E4>(y, D, b, idx0, a.pk, w0, w1, GS ? nullptr : rt, sf, q, wq);
    } else {
        four_over_six16<ERR, std::is_same<TileAmax, OwnAmax>::value>(y, b, gb, C, tab, w0, w1, sf, d, tile_sums);
    }
    if (!live) return;
    if (tile_amax.failed) {
        if (a.scales) a.scales[blk] = 0x7F;
        if (a.dq_bf16) {
            float nan16[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) nan16[i] = __int_as_float(0x7FC00000);
            store16_bf16(a.dq_bf16, blk * 16, nan16);
        }
        return;
    }
    if (a.codes) reinterpret_cast<uint2*>(a.codes)[blk] = make_uint2(w0, w1);
    if (a.scales) a.scales[blk] = static_cast<uint8_t>(sf);
    if (wq) {
        // stochastic rounding without a global scale: the residual straight from the grid values
        constexpr bool FUSED = EF && QV && !GS;
        if (FUSED) {
            float r[16];
            residual_q16(y, q, d, r);
            store16_f32(a.residual, blk * 16, r);
        }
        if (!FUSED || a.dq_bf16) {
            float dq[16];
            if (QV) dequant_q16<GS>(q, d, gb.Sdec, dq);
            else dequant16<GS || ERR != NVFP4_ERR_NONE>(w0, w1, d, gb.Sdec, dq);
            if (EF && !FUSED) {
                float r[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) r[i] = sub_rn(y[i], dq[i]);
                store16_f32(a.residual, blk * 16, r);
            }
            if (a.dq_bf16) store16_bf16(a.dq_bf16, blk * 16, dq);
        }
    }
}

// Per-thread copy pipeline: stage s holds, for each thread, its block's x
// bytes (and residual bytes under error feedback) for one grid-stride step,
// each in a slot of its own with the 16-byte pieces swizzled (piece_swizzle).
// With a residual a block moves 96-128 bytes, so one step ahead at a higher
// occupancy keeps enough in flight; without, three steps ahead (the stage count is per variant).
template <int DT, bool EF, int NT = kThreads, int EF_STAGES = 2>
struct RowsStage {
    static constexpr int STAGES = EF ? EF_STAGES : 4;
    static constexpr int XB = DT == NVFP4_BF16 ? 32 : 64;   // x bytes per block
    static constexpr int RB = EF ? 64 : 0;                    // residual bytes per block
    static constexpr int BYTES = NT * (XB + RB);
    static constexpr int TOTAL = STAGES * BYTES;
};

template <int DT, int ERR, int RND, bool EF, bool GS>
__global__ void __launch_bounds__(kThreads) k_rows(const QuantArgs a) {
    using St = RowsStage<DT, EF>;
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ O6TabOf<ERR> tab;
    __shared__ float rtab[(ERR == NVFP4_ERR_NONE && !GS) ? 128 : 1];
    if (ERR == NVFP4_ERR_NONE && !GS) fill_recip_table(rtab);
    pdl_wait();
    const int64_t bpr = a.K / 16;
    const int64_t nblk = a.M * bpr;
    GScale g{0.0f, 1.0f, 1.0f};
    if (a.gamax_mode == NVFP4_GAMAX_TENSOR_GIVEN) {
        g.A = a.gamax[0];
        global_scales(g.A, a.bound, g.Senc, g.Sdec);
    }
    const float C = mul_rn(6.0f, a.bound);
    const O6Tab* tp = nullptr;
    if constexpr (ERR != NVFP4_ERR_NONE) {
        if (a.gamax_mode == NVFP4_GAMAX_TENSOR_GIVEN) {
            fill_o6_table(&tab, g.Sdec, g.A, C);
            tp = &tab;
        }
    }
    const uint64_t idx_base = static_cast<uint64_t>(a.row_offset) * static_cast<uint64_t>(a.K);
    const int tid = threadIdx.x;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t first = static_cast<int64_t>(blockIdx.x) * blockDim.x + tid;
    unsigned char* xs = smem + tid * St::XB;
    unsigned char* rs = smem + kThreads * St::XB + tid * St::RB;
    const uint32_t swx = piece_swizzle<St::XB / 16>(tid), swr = piece_swizzle<4>(tid);

    auto issue = [&](int64_t blk, int stage) {
        if (blk < nblk) {
            const unsigned char* gx = static_cast<const unsigned char*>(a.x) + blk * St::XB;
#pragma unroll
            for (int c = 0; c < St::XB / 16; ++c) cp_async16(xs + stage * St::BYTES + ((c ^ swx) << 4), gx + 16 * c);
            if (EF) {
                const unsigned char* gr = reinterpret_cast<const unsigned char*>(a.residual) + blk * 64;
#pragma unroll
                for (int c = 0; c < 4; ++c) cp_async16(rs + stage * St::BYTES + ((c ^ swr) << 4), gr + 16 * c);
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
        lds16_swz<DT>(xs + stage * St::BYTES, swx, y);
        if (EF) {
            float r[16];
            lds16_swz<NVFP4_F32>(rs + stage * St::BYTES, swr, r);
            add16(y, r);
        }
        OwnAmax own;
        rows_block<DT, ERR, RND, EF, GS>(a, blk, true, y, g, C, tp, rtab, idx_base, bpr, own,
                                         [](float&, float&) {}, [] {});
        stage = stage == S - 1 ? 0 : stage + 1;
    }
    pdl_trigger();
    cp_async_wait<0>();
}

// 16x16 blocks, rowwise output.  One CTA step quantizes a 16-row band x T
// tiles (BandGeom: T = 16 for 256 threads): warp w holds RPW consecutive rows
// of the band (2 for 256 threads: lanes 0-15 and 16-31), lane l % T the tile,
// so a warp's loads and stores run along its rows like the 1x16 walk's.  The
// tile amax is reduced over the warp's rows with shuffles and then over the
// warps through shared memory; four-over-six's row error sums are
// combined with the width-16 tree in the same way.  The CTAs walk the steps
// (band-major) persistently, each thread fetching its group one step ahead
// (the per-thread copy pipeline of k_rows); the reductions' shared buffers
// alternate between steps, so one barrier per reduction suffices.  (Staging
// whole bands with bulk copies several steps ahead, and publishing each
// step's tile maxima one step early, were both measured slower: fewer CTAs
// fit per SM and the extra shared-memory traffic outweighed the shorter
// waits.)
//
// Band geometry for a CTA of NT threads: a step covers 16 rows x T tiles
// (T = NT / 16); warp w holds rows w*RPW .. w*RPW + RPW - 1 (RPW = 32 / T),
// lane l row w*RPW + l / T and tile l % T, so a warp's loads run along RPW
// rows, T * 32 bytes (bf16) each.
template <int NT>
struct BandGeom {
    static constexpr int T = NT / 16;            // tiles per step
    static constexpr int RPW = 32 / T;           // rows per warp
    static constexpr int NW = NT / 32;           // warps
};

// The tile amax of k_band16: post() reduces the group maxima over the warp's
// rows with shuffles and publishes the warp's value; get() passes the CTA
// barrier (a hardware barrier: waiting warps issue nothing) and reduces over
// the warps.  The stochastic-rounding draws are made between the two.  The
// partial maxima alternate between two buffers by step parity: a thread
// writes a step's buffer only after it passed the previous step's barrier,
// which every thread reaches after reading the buffer two steps back.  Every
// thread runs the same CTA-uniform steps, so every barrier completes.
template <int NT>
struct BandAmax {
    using Gm = BandGeom<NT>;
    static constexpr bool kSplit = true;
    static constexpr bool failed = false;
    float (*red)[Gm::NW][Gm::T];
    int warp, lane, t;
    uint32_t step;                               // this thread's step count
    __device__ void post(float b) {
#pragma unroll
        for (int o = Gm::T; o < 32; o <<= 1) b = max_nd(b, __shfl_xor_sync(kFullMask, b, o));
        if (lane < Gm::T) red[step & 1][warp][t] = b;
    }
    __device__ float get() {
        __syncthreads();
        float m = red[step & 1][0][t];
#pragma unroll
        for (int w = 1; w < Gm::NW; ++w) m = max_nd(m, red[step & 1][w][t]);
        ++step;
        return m;
    }
};

// CTA-uniform step (band, column chunk) and this thread's 1x16 block in it.
// The band and chunk counters are 32-bit; the block index (64-bit) is kept
// up to date by additions only: a chunk is T blocks along the row, a band 16
// rows of nb blocks.
struct BandCursor {
    int32_t band, chunk, nch, dband, dchunk;
    int64_t blk;                                 // block index of (band*16 + rr, chunk*T + t)
    int64_t dblk_band, dblk_step;                // blk increments: one band, one regular step
    __device__ void init(int64_t u, int32_t nch_, int64_t stride, int64_t nb, int rr, int t, int T) {
        nch = nch_;
        band = static_cast<int32_t>(u / nch);
        chunk = static_cast<int32_t>(u - static_cast<int64_t>(band) * nch);
        dband = static_cast<int32_t>(stride / nch);
        dchunk = static_cast<int32_t>(stride - static_cast<int64_t>(dband) * nch);
        dblk_band = 16 * nb;
        dblk_step = dband * dblk_band + static_cast<int64_t>(dchunk) * T;
        blk = (static_cast<int64_t>(band) * 16 + rr) * nb + static_cast<int64_t>(chunk) * T + t;
        wrap = dblk_band - static_cast<int64_t>(nch) * T;
    }
    int64_t wrap;                                // blk correction when the chunk wraps to the next band
    __device__ void advance() {
        band += dband;
        chunk += dchunk;
        blk += dblk_step;
        if (chunk >= nch) {
            chunk -= nch;
            ++band;
            blk += wrap;
        }
    }
};

#ifndef NVFP4_BAND_THREADS
#define NVFP4_BAND_THREADS 128
#endif
#ifndef NVFP4_BAND_EF_STAGES
#define NVFP4_BAND_EF_STAGES 2
#endif
constexpr int kBandThreads = NVFP4_BAND_THREADS;
constexpr int kBandEfStages = NVFP4_BAND_EF_STAGES;

template <int DT, int ERR, int RND, bool EF, bool GS>
__global__ void __launch_bounds__(kBandThreads) k_band16(const QuantArgs a) {
    constexpr int NT = kBandThreads;
    using Gm = BandGeom<NT>;
    using St = RowsStage<DT, EF, NT, kBandEfStages>;
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ O6TabOf<ERR> tab;
    __shared__ float rtab[(ERR == NVFP4_ERR_NONE && !GS) ? 128 : 1];
    __shared__ float red[2][Gm::NW][Gm::T];                           // [step parity][warp][tile]
    __shared__ float esum[ERR != NVFP4_ERR_NONE ? 2 : 1][2][16][Gm::T];  // [parity][cand][row][tile]
    if (ERR == NVFP4_ERR_NONE && !GS) fill_recip_table(rtab);
    pdl_wait();
    const int64_t nb = a.K / 16;
    const int64_t nch = (nb + Gm::T - 1) / Gm::T;
    const int64_t nbands = a.M / 16;
    GScale g{0.0f, 1.0f, 1.0f};
    if (a.gamax_mode == NVFP4_GAMAX_TENSOR_GIVEN) {
        g.A = a.gamax[0];
        global_scales(g.A, a.bound, g.Senc, g.Sdec);
    }
    const float C = mul_rn(6.0f, a.bound);
    const O6Tab* tp = nullptr;
    if constexpr (ERR != NVFP4_ERR_NONE) {
        fill_o6_table(&tab, g.Sdec, g.A, C);
        tp = &tab;
    }
    const uint64_t idx_base = static_cast<uint64_t>(a.row_offset) * static_cast<uint64_t>(a.K);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rr = warp * Gm::RPW + lane / Gm::T;   // row within the band
    const int t = lane % Gm::T;                  // tile within the chunk
    unsigned char* xs = smem + tid * St::XB;
    unsigned char* rs = smem + NT * St::XB + tid * St::RB;
    const uint32_t swx = piece_swizzle<St::XB / 16>(tid), swr = piece_swizzle<4>(tid);

    const int32_t nbands32 = static_cast<int32_t>(nbands), nb32 = static_cast<int32_t>(nb);
    const bool whole = nb32 % Gm::T == 0;        // every chunk full: a column is never past the row
    auto group = [&](const BandCursor& c, bool& live) {   // this thread's 1x16 block
        live = c.band < nbands32 && (whole || c.chunk * Gm::T + t < nb32);
        return c.blk;
    };
    auto issue = [&](const BandCursor& c, int stage) {   // returns the group's liveness
        bool live;
        const int64_t blk = group(c, live);
        if (live) {
            const unsigned char* gx = static_cast<const unsigned char*>(a.x) + blk * St::XB;
#pragma unroll
            for (int k = 0; k < St::XB / 16; ++k) cp_async16(xs + stage * St::BYTES + ((k ^ swx) << 4), gx + 16 * k);
            if (EF) {
                const unsigned char* gr = reinterpret_cast<const unsigned char*>(a.residual) + blk * 64;
#pragma unroll
                for (int k = 0; k < 4; ++k) cp_async16(rs + stage * St::BYTES + ((k ^ swr) << 4), gr + 16 * k);
            }
        }
        cp_async_commit();
        return live;
    };

    constexpr int S = St::STAGES;
    BandCursor cur, ahead;
    cur.init(blockIdx.x, static_cast<int32_t>(nch), gridDim.x, nb, rr, t, Gm::T);
    ahead = cur;
    bool live_cur = false;                       // S == 2: the current group's liveness, from its issue
#pragma unroll
    for (int k = 0; k < S - 1; ++k) {
        live_cur = issue(ahead, k);
        ahead.advance();
    }
    int stage = 0, par = 0;
    BandAmax<NT> tile_amax{red, warp, lane, t, 0u};
    while (cur.band < nbands32) {
        // with two stages the next step is the one just issued: copied, not advanced
        const BandCursor next = ahead;
        const bool live_next = issue(ahead, stage == 0 ? S - 1 : stage - 1);
        ahead.advance();
        cp_async_wait<S - 1>();
        bool live = live_cur;
        const int64_t blk = S == 2 ? cur.blk : group(cur, live);
        float y[16];
        if (live) {
            lds16_swz<DT>(xs + stage * St::BYTES, swx, y);
            if (EF) {
                float r[16];
                lds16_swz<NVFP4_F32>(rs + stage * St::BYTES, swr, r);
                add16(y, r);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) y[i] = 0.0f;
        }
        auto tile_sums = [&](float& E6, float& E4) {
            if constexpr (ERR != NVFP4_ERR_NONE) {
                esum[par][0][rr][t] = E6;
                esum[par][1][rr][t] = E4;
                __syncthreads();
                float e[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) e[r] = esum[par][0][r][t];
                E6 = tree16_regs(e);
#pragma unroll
                for (int r = 0; r < 16; ++r) e[r] = esum[par][1][r][t];
                E4 = tree16_regs(e);
            }
        };
        rows_block<DT, ERR, RND, EF, GS>(a, blk, live, y, g, C, tp, rtab, idx_base, nb, tile_amax, tile_sums,
                                         [] {});
        stage = stage == S - 1 ? 0 : stage + 1;
        par ^= 1;
        if (S == 2) {
            cur = next;
            live_cur = live_next;
        } else {
            cur.advance();
        }
    }
    pdl_trigger();
    cp_async_wait<0>();
}

template <class KernelT>
int launch_persistent(KernelT kernel, int smem, int64_t units_per_cta_step, int64_t units, const QuantArgs& a,
                      cudaStream_t s, int& configured_dev, int& per_sm, int threads = kThreads) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_dev != dev) {
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess ||
            per_sm < 1)
            per_sm = 1;
        configured_dev = dev;
    }
    const int64_t want = (units + units_per_cta_step - 1) / units_per_cta_step;
    const int64_t cap = static_cast<int64_t>(sm_count()) * per_sm;
    const int grid = static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
    launch_pdl(kernel, grid, threads, smem, s, a);
    return static_cast<int>(cudaGetLastError());
}

// BLK 1x16: k_rows over blocks; 16x16: k_band16 over (band, chunk) steps
template <int DT, int BLK, int ERR, int RND, bool EF, bool GS>
int launch_rows(const QuantArgs& a, int64_t nblk, cudaStream_t s) {
    static thread_local int configured_dev = -1, per_sm = 1;
    if (BLK == NVFP4_BLOCK_16X16) {
        constexpr int T = BandGeom<kBandThreads>::T;
        const int64_t steps = (a.M / 16) * ((a.K / 16 + T - 1) / T);
        return launch_persistent(k_band16<DT, ERR, RND, EF, GS>,
                                 RowsStage<DT, EF, kBandThreads, kBandEfStages>::TOTAL, 1, steps, a, s,
                                 configured_dev, per_sm, kBandThreads);
    }
    return launch_persistent(k_rows<DT, ERR, RND, EF, GS>, RowsStage<DT, EF>::TOTAL, kThreads, nblk, a, s,
                             configured_dev, per_sm);
}

template <int DT, int BLK, bool GS>
int rows_plain(const QuantArgs& a, int64_t nblk, cudaStream_t s) {
    const bool ef = a.residual != nullptr;
    if (a.rounding == NVFP4_RTN)
        return ef ? launch_rows<DT, BLK, NVFP4_ERR_NONE, NVFP4_RTN, true, GS>(a, nblk, s)
                  : launch_rows<DT, BLK, NVFP4_ERR_NONE, NVFP4_RTN, false, GS>(a, nblk, s);
    if (a.rounding == NVFP4_RTN_STD)
        return ef ? launch_rows<DT, BLK, NVFP4_ERR_NONE, NVFP4_RTN_STD, true, GS>(a, nblk, s)
                  : launch_rows<DT, BLK, NVFP4_ERR_NONE, NVFP4_RTN_STD, false, GS>(a, nblk, s);
    return ef ? launch_rows<DT, BLK, NVFP4_ERR_NONE, NVFP4_SR, true, GS>(a, nblk, s)
              : launch_rows<DT, BLK, NVFP4_ERR_NONE, NVFP4_SR, false, GS>(a, nblk, s);
}

template <int DT, int BLK>
int rows_dispatch_blk(const QuantArgs& a, cudaStream_t s) {
    const int64_t nblk = a.M * (a.K / 16);
    if (a.err_mode == NVFP4_ERR_MAE) return launch_rows<DT, BLK, NVFP4_ERR_MAE, NVFP4_RTN, false, true>(a, nblk, s);
    if (a.err_mode == NVFP4_ERR_MSE) return launch_rows<DT, BLK, NVFP4_ERR_MSE, NVFP4_RTN, false, true>(a, nblk, s);
    return a.gamax_mode == NVFP4_GAMAX_NONE ? rows_plain<DT, BLK, false>(a, nblk, s)
                                            : rows_plain<DT, BLK, true>(a, nblk, s);
}

template <int DT>
int rows_dispatch(const QuantArgs& a, cudaStream_t s) {
    return a.block == NVFP4_BLOCK_16X16 ? rows_dispatch_blk<DT, NVFP4_BLOCK_16X16>(a, s)
                                        : rows_dispatch_blk<DT, NVFP4_BLOCK_1X16>(a, s);
}

}  // namespace

int launch_quantize_rows(const QuantArgs& a, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return a.dtype == NVFP4_BF16 ? rows_dispatch<NVFP4_BF16>(a, s) : rows_dispatch<NVFP4_F32>(a, s);
}

}  // namespace nvfp4
