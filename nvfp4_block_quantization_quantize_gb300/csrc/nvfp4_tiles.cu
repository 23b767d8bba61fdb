// nvfp4_tiles.cu -- 16x16 blocks and columnwise outputs for sm_103a.
//
// k_tiles_rows  rowwise + columnwise output (no residual): one CTA = 256
//               columns of 4 consecutive 16-row bands, walked in turn; lane
//               l of warp w holds row l%16 of the 16x16 tile 2w + l/16.
//               16x16 blocks reduce their amax (and, for four-over-six, their
//               row error sums with the fixed width-16 tree) over the half
//               warp.  The band is then staged in shared memory and each
//               thread owns one column (x^T's row) of it for the columnwise
//               pass; the 4 bands' columnwise codes wait in shared memory and
//               leave as one 32-byte run per column.  It serves the 1x16
//               row+col calls with stochastic rounding, with four-over-six
//               and with fp32 input.
// k_tile_r1     1x16 row+col, nearest rounding, bf16: one thread per 16x16
//               tile staged in shared memory, its rows and columns encoded
//               as independent blocks.
// k_tile_p      plain 16x16 row+col (nearest or stochastic): one thread per
//               tile, the tile's one scale serving both outputs, the
//               columnwise codes the rowwise ones transposed.
// k_tile_ts     four-over-six 16x16 with rowwise AND columnwise output, bf16
//               input: one thread owns a whole 16x16 tile, copies its 16 rows
//               into shared memory up front, and walks them twice (amax; both
//               candidates' codes and approximate errors, the column sums
//               accumulated in row order).  One approximate sum per candidate
//               certifies both the row and the column choice; where it does
//               not, the exact row sums and x^T's element-order column sums
//               are taken from the error-value table.  The columnwise codes
//               are transposed in registers.  A CTA is 4 bands (one per warp)
//               x 32 tiles: a warp's copies of a row cover 32 consecutive
//               tiles (fully coalesced), and the columnwise output, staged in
//               shared memory, leaves as one 32-byte run per column (4 bands
//               x 8 bytes) instead of 8-byte pieces 32 to a warp store.
// k_tile_ts4    the same for fp32 input with four threads per tile (lanes
//               4t .. 4t+3: columns 0-3, 4-7, 8-11, 12-15), so that a
//               thread's share, 16 rows x 4 fp32, is staged whole too; the
//               quad exchanges the tile amax and the column sums by shuffles
//               and on the exact path runs each row's sum along its lanes.
//               A CTA is 4 bands x 8 tiles.
//
// Method: "Add NVFP4 four-over-six (row-wise) quantization to the training
// prototype" (What: 16x16 blocks, rowwise / columnwise; CuTe DSL kernel
// (SM100), Design: width-16 tree, element-order sums; Follow-up fusions: a
// fused row + col kernel) and "Stable FP4 Training via Transposition-Invariant
// Block Quantization" (abstract: one 2D block scale for x and x^T).
#include "nvfp4_block.cuh"

namespace nvfp4 {
namespace {

constexpr int kThreads = 256;
constexpr int kTileCols = 256;
constexpr int kYsStride = kTileCols + 4;

constexpr int kRowBands = 4;                    // bands per CTA of k_tiles_rows

template <int DT, int BLK, int ERR, int RND, bool GS>
__global__ void __launch_bounds__(kThreads) k_tiles_rows(const QuantArgs a) {
    __shared__ float ys[16 * kYsStride];
    // stochastic rounding: the row pass's draws, keyed on x's index, reused by
    // the column pass
    __shared__ uint32_t ws[RND == NVFP4_SR ? 16 * kYsStride : 1];
    __shared__ O6TabOf<ERR> tab;
    __shared__ float rtab[(ERR == NVFP4_ERR_NONE && !GS) ? 128 : 1];
    // columnwise codes and scale bytes of the CTA's bands, [band][column]
    __shared__ uint2 ccs[kRowBands][kTileCols];
    __shared__ uint8_t scs[kRowBands][kTileCols];
    // the thread's block of the current and the next band, copied ahead
    // asynchronously (each thread reads only its own slot)
    constexpr int XB = DT == NVFP4_BF16 ? 32 : 64;
    __shared__ __align__(16) unsigned char xb[2][kThreads * XB];
    if (ERR == NVFP4_ERR_NONE && !GS) fill_recip_table(rtab);
    pdl_wait();
    const int64_t chunk = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = 2 * warp + (lane >> 4);
    const int rr = lane & 15;
    const int64_t nb = a.K / 16;
    const int64_t nbands = a.M / 16;
    const int64_t band0 = static_cast<int64_t>(blockIdx.x) * kRowBands;
    const int64_t cb = chunk * 16 + t;
    const bool valid = cb < nb;

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

    const int j = threadIdx.x;                  // column within the chunk (its tile is t)
    auto fetch = [&](int bi) {
        const int64_t band = band0 + bi;
        if (valid && bi < kRowBands && band < nbands) {
            const unsigned char* src = static_cast<const unsigned char*>(a.x) +
                                       ((band * 16 + rr) * a.K + cb * 16) * (XB / 16);
#pragma unroll
            for (int c = 0; c < XB / 16; ++c) cp_async16(&xb[bi & 1][threadIdx.x * XB + 16 * c], src + 16 * c);
        }
        cp_async_commit();
    };
    fetch(0);
    for (int bi = 0; bi < kRowBands; ++bi) {
        const int64_t band = band0 + bi;
        if (band >= nbands) break;              // CTA-uniform
        const int64_t row = band * 16 + rr;
        const int64_t e0 = row * a.K + cb * 16;
        fetch(bi + 1);
        cp_async_wait<1>();
        float y[16];
        if (valid) {
            lds16<DT>(&xb[bi & 1][threadIdx.x * XB], y);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) y[i] = 0.0f;
        }
        float b = absmax16(y);
        if (BLK == NVFP4_BLOCK_16X16) b = max16_lanes(b);

        // ---- rowwise ----
        {
            uint32_t w0, w1, sf;
            float d;
            if (ERR == NVFP4_ERR_NONE) {
                const float s6f = block_scale<GS>(b, g.Senc, RND == NVFP4_RTN_STD);
                sf = e4m3_encode(min_nd(s6f, 448.0f));
                d = e4m3_decode(sf);
                const float D = GS ? mul_rn(d, g.Sdec) : d;
                float q[16];
                uint32_t wd[16];
                if (RND == NVFP4_SR) {
                    const uint64_t idx0 = (static_cast<uint64_t>(a.row_offset) + static_cast<uint64_t>(row)) *
                                              static_cast<uint64_t>(a.K) + static_cast<uint64_t>(cb * 16);
                    sr_words16(idx0, a.pk, wd);
#pragma unroll
                    for (int i = 0; i < 16; ++i) ws[rr * kYsStride + t * 16 + i] = wd[i];
                }
                encode_plain16_words<RND>(y, D, b, wd, w0, w1, GS ? nullptr : rtab, sf, q, false);
            } else {
                four_over_six16<ERR, BLK == NVFP4_BLOCK_16X16>(y, b, g, C, tp, w0, w1, sf, d);
            }
            if (valid) {
                if (a.codes) reinterpret_cast<uint2*>(a.codes)[e0 / 16] = make_uint2(w0, w1);
                if (a.scales) a.scales[row * nb + cb] = static_cast<uint8_t>(sf);
            }
        }
        // ---- columnwise: the rowwise quantization of x^T, from the staged band ----
#pragma unroll
        for (int i = 0; i < 16; ++i) ys[rr * kYsStride + t * 16 + i] = y[i];
        __syncthreads();
        float c[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) c[r] = ys[r * kYsStride + j];
        float bc = absmax16(c);
        if (BLK == NVFP4_BLOCK_16X16) bc = max16_lanes(bc);
        uint32_t w0, w1, sf;
        float d;
        if (ERR == NVFP4_ERR_NONE) {
            const float s6f = block_scale<GS>(bc, g.Senc, RND == NVFP4_RTN_STD);
            sf = e4m3_encode(min_nd(s6f, 448.0f));
            d = e4m3_decode(sf);
            const float D = GS ? mul_rn(d, g.Sdec) : d;
            float qc[16];
            uint32_t wd[16];
            if (RND == NVFP4_SR) {
#pragma unroll
                for (int r = 0; r < 16; ++r) wd[r] = ws[r * kYsStride + j];
            }
            encode_plain16_words<RND>(c, D, bc, wd, w0, w1, GS ? nullptr : rtab, sf, qc, false);
        } else {
            four_over_six16<ERR, BLK == NVFP4_BLOCK_16X16>(c, bc, g, C, tp, w0, w1, sf, d);
        }
        ccs[bi][j] = make_uint2(w0, w1);
        scs[bi][j] = static_cast<uint8_t>(sf);
        __syncthreads();                        // ys and ws are rewritten by the next band
    }
    cp_async_wait<0>();
    // x^T's row col holds 8 code bytes and one scale byte per band: the CTA's
    // bands give each of its columns one run of consecutive bytes, written
    // by consecutive threads
    const int64_t nbc = nbands - band0 < kRowBands ? nbands - band0 : kRowBands;
    uint2* cc = reinterpret_cast<uint2*>(a.codes_col);
    for (int q = threadIdx.x; q < kRowBands * kTileCols; q += kThreads) {
        const int jj = q / kRowBands, bb = q % kRowBands;
        const int64_t cj = chunk * kTileCols + jj;
        if (bb < nbc && cj < a.K) {
            cc[cj * nbands + band0 + bb] = ccs[bb][jj];
            a.scales_col[cj * nbands + band0 + bb] = scs[bb][jj];
        }
    }
    pdl_trigger();
}

// ---------------------------------------------------------------------------------------------
constexpr int kTileThreads = 128;

// Ring of tile rows per thread of k_tile_p: 4 slots of bf16 rows, 3 of fp32
// rows (the same bytes in flight).
template <int DT>
struct TilePRing {
    static constexpr int XB = DT == NVFP4_BF16 ? 32 : 64;    // bytes of one tile row
    static constexpr int SLOTS = DT == NVFP4_BF16 ? 4 : 3;
    static constexpr int BYTES = SLOTS * kTileThreads * XB;
};

// The width-16 tree's upper levels over the first level's eight pair sums
// s[i] = R[i] + R[i + 8] of the row sums R.
__device__ __forceinline__ float tree16_upper(const float* s) {
    return add_rn(add_rn(add_rn(s[0], s[4]), add_rn(s[2], s[6])),
                  add_rn(add_rn(s[1], s[5]), add_rn(s[3], s[7])));
}

constexpr int kBands = kTileThreads / 32;       // 16-row bands per CTA, one per warp

// Staging slot of (band b of the CTA, column j of the CTA's 512) for the
// columnwise words: band-major, the column's low four bits XORed with its
// tile's (j / 16) and with 8 for odd bands, so that a warp's writes (one
// column of each of 32 tiles) and its reads (8 columns x 4 bands) both take
// the minimum of two shared-memory wavefronts.
__device__ __forceinline__ int stage_index(int b, int j) {
    return b * 512 + (j ^ ((j >> 4) & 15) ^ ((b & 1) << 3));
}

// Four-over-six 16x16 with rowwise and columnwise output, bf16 input, the
// whole tile staged: one thread per tile computes both candidates' codes and
// errors from one walk, certifies both choices with one approximate sum per
// candidate and falls back to the exact sums where that fails.  Each thread
// copies its tile's 16 rows (512 bytes) into shared memory with
// asynchronous copies as soon as it starts, so the error pass reads shared
// memory instead of waiting on L2 one row ahead.  The
// 64 KB of a CTA's tiles leaves room for three CTAs per SM, so the other
// CTAs' error passes cover a CTA's copies.  A thread's slot of row r (32
// bytes, its 16-byte pieces swizzled by piece_swizzle<2>) is reused once row
// r has been read: its first piece takes the row's code words of both
// candidates (map-to-6 then map-to-4), the second piece of rows 0-7 the row
// sums (the width-16 tree's first level), and the exact fallback's error
// values wait in the second piece of rows 8-15 (the fallback reads x again
// from global memory).  The columnwise output is staged in the same buffer
// once every thread is done with its slots.
constexpr int kStagedTileBytes = 16 * kTileThreads * 32;

template <int ERR>
__global__ void __launch_bounds__(kTileThreads) k_tile_ts(const QuantArgs a) {
    extern __shared__ __align__(16) unsigned char tile_s[];   // [row][thread][32 bytes]
    __shared__ float tenc[128];                 // encode reciprocal of every scale byte
    __shared__ uint8_t scol[kBands][32];        // columnwise scale byte of each tile
    pdl_wait();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t M = a.M, K = a.K;
    const int64_t band0 = static_cast<int64_t>(blockIdx.x) * kBands, band = band0 + warp;
    const int64_t tile0 = static_cast<int64_t>(blockIdx.y) * 32, tile = tile0 + lane;
    const int64_t nb = K / 16, nbands = M / 16;
    const bool own = band < nbands && tile < nb;
    const int64_t base = band * 16 * K + tile * 16;
    const uint32_t swz = piece_swizzle<2>(tid);
    auto slot = [&](int r) { return tile_s + (r * kTileThreads + tid) * 32; };
    auto piece = [&](int r, uint32_t c) { return slot(r) + ((c ^ swz) << 4); };
    if (own) {                                  // the tile's rows, four per copy group
        const unsigned char* gx = static_cast<const unsigned char*>(a.x) + base * 2;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            cp_async16(piece(r, 0), gx + static_cast<int64_t>(r) * K * 2);
            cp_async16(piece(r, 1), gx + static_cast<int64_t>(r) * K * 2 + 16);
            if ((r & 3) == 3) cp_async_commit();
        }
    }
    GScale g{0.0f, 1.0f, 1.0f};
    if (a.gamax_mode == NVFP4_GAMAX_TENSOR_GIVEN) {
        g.A = a.gamax[0];
        global_scales(g.A, a.bound, g.Senc, g.Sdec);
    }
    const float C = mul_rn(6.0f, a.bound);
    for (int i = tid; i < 128; i += blockDim.x)
        tenc[i] = min_nd(div_rn(1.0f, mul_rn(e4m3_decode(static_cast<uint32_t>(i)), g.Sdec)), FLT_MAX);
    __syncthreads();

    uint32_t lo[16], hi[16];                    // columnwise code words, transposed
    uint32_t sf_c = 0;
    if (own) {
        // pass 0: tile amax on the packed pairs, each copy group as it lands
        uint32_t m2 = 0u;
        auto amax4 = [&](int r0) {
#pragma unroll
            for (int r = r0; r < r0 + 4; ++r) {
                const uint4 u = *reinterpret_cast<const uint4*>(piece(r, 0));
                const uint4 v = *reinterpret_cast<const uint4*>(piece(r, 1));
                m2 = absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(m2, u.x), u.y), u.z), u.w);
                m2 = absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(m2, v.x), v.y), v.z), v.w);
            }
        };
        cp_async_wait<3>();
        amax4(0);
        cp_async_wait<2>();
        amax4(4);
        cp_async_wait<1>();
        amax4(8);
        cp_async_wait<0>();
        amax4(12);
        const float b = max_nd(__uint_as_float(m2 << 16), __uint_as_float(m2 & 0xFFFF0000u));
        const float s6f = block_s6f<true>(b, g.Senc);
        const uint32_t sf6 = e4m3_encode(min_nd(s6f, 448.0f));
        const uint32_t sf4 = e4m3_encode(min_nd(mul_rn(s6f, 1.5f), 448.0f));
        const float enc6 = tenc[sf6], enc4 = tenc[sf4];
        const float d6 = e4m3_decode(sf6), d4 = e4m3_decode(sf4);
        // K: the error value of grid value 1, ((1 * d) * A) / (6 * bound)
        const float K6 = div_rn(mul_rn(d6, g.A), C), K4 = div_rn(mul_rn(d4, g.A), C);

        // pass 1: both candidates' codes, and approximate per-element errors
        // in the scaled domain, |q - v| with v = y * enc (squared for MSE; q
        // the code's signed grid value) from one mixed f16/f32 subtract; the
        // column sums in row order, from the staged rows
        float F6[16], F4[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) F6[i] = F4[i] = 0.0f;
        const uint64_t ENC6 = pack2(enc6, enc6), ENC4 = pack2(enc4, enc4);
        auto candidate = [&](const float* y, uint64_t enc2, uint32_t& w0, uint32_t& w1, float* e) {
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; i += 2) unpack2(mul2(pack2(y[i], y[i + 1]), enc2), v[i], v[i + 1]);
            uint32_t h[8];
            w0 = e2m1_encode8_dec(v, h);
            w1 = e2m1_encode8_dec(v + 8, h + 4);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                sub_f16x2_f32(h[j], v[2 * j], v[2 * j + 1], e[2 * j], e[2 * j + 1]);
                if (ERR != NVFP4_ERR_MAE) {
                    const uint64_t D = pack2(e[2 * j], e[2 * j + 1]);
                    unpack2(mul2(D, D), e[2 * j], e[2 * j + 1]);
                }
            }
            if (ERR == NVFP4_ERR_MAE) {
#pragma unroll
                for (int i = 0; i < 16; ++i) e[i] = fabsf(e[i]);
            }
        };
        auto col_sums = [&](float* F, const float* e) { add16(F, e); };
        // row sums: rows 0-7 stored, row r >= 8 added to row r - 8's
        auto row_sums = [&](int r, float R6, float R4) {
            float2* p = reinterpret_cast<float2*>(piece(r & 7, 1));
            if (r >= 8) {
                const float2 s = *p;
                R6 = add_rn(s.x, R6);
                R4 = add_rn(s.y, R4);
            }
            *p = make_float2(R6, R4);
        };
        float y[16];
#pragma unroll 4
        for (int r = 0; r < 16; ++r) {
            lds16_swz<NVFP4_BF16>(slot(r), swz, y);
            float e[16];
            uint32_t a0, a1, b0, b1;
            candidate(y, ENC6, a0, a1, e);
            col_sums(F6, e);
            candidate(y, ENC4, b0, b1, e);
            col_sums(F4, e);
            *reinterpret_cast<uint4*>(piece(r, 0)) = make_uint4(a0, a1, b0, b1);
        }
        float E6r, E4r, E6c, E4c;
        auto tree_sums = [&]() {
            float S6[8], S4[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float2 s = *reinterpret_cast<const float2*>(piece(i, 1));
                S6[i] = s.x;
                S4[i] = s.y;
            }
            E6r = tree16_upper(S6);
            E4r = tree16_upper(S4);
            E6c = tree16_regs(F6);
            E4c = tree16_regs(F4);
        };
        {   // back from the scaled domain, one sum per candidate for both choices
            const float k6 = ERR == NVFP4_ERR_MAE ? K6 : mul_rn(K6, K6);
            const float k4 = ERR == NVFP4_ERR_MAE ? K4 : mul_rn(K4, K4);
            E6r = E6c = mul_rn(k6, tree16_regs(F6));
            E4r = E4c = mul_rn(k4, tree16_regs(F4));
        }
        if (!tile_sums_decide<ERR>(E6c, E4c, K6, K4, b)) {
            // the exact sums: error values |dq| = ((G[k] * d) * A) / (6 *
            // bound) of each grid magnitude (a code of index k stands for
            // +-|dq| with the sign of its y, so |dq - y| = | |dq| - |y| |
            // exactly, and likewise the square) in row 8 + k's second piece
            // (map-to-6, map-to-4), the codes kept in the first pieces, x
            // read again; row sums in element order and x^T's column sums
            const float G[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
#pragma unroll
            for (int k = 0; k < 8; ++k)
                *reinterpret_cast<float2*>(piece(8 + k, 1)) =
                    make_float2(div_rn(mul_rn(mul_rn(G[k], d6), g.A), C), div_rn(mul_rn(mul_rn(G[k], d4), g.A), C));
            auto exact = [&](const float* y, uint32_t w0, uint32_t w1, int c, float* e) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const uint32_t k = ((i < 8 ? w0 : w1) >> (4 * (i & 7))) & 7u;
                    const float dq = reinterpret_cast<const float*>(piece(8 + k, 1))[c];
                    const float diff = sub_rn(dq, fabsf(y[i]));
                    e[i] = (ERR == NVFP4_ERR_MAE) ? fabsf(diff) : mul_rn(diff, diff);
                }
            };
#pragma unroll
            for (int i = 0; i < 16; ++i) F6[i] = F4[i] = 0.0f;
#pragma unroll 1
            for (int r = 0; r < 16; ++r) {
                load16<NVFP4_BF16>(a.x, base + static_cast<int64_t>(r) * K, y);
                const uint4 w = *reinterpret_cast<const uint4*>(piece(r, 0));
                float e[16];
                exact(y, w.x, w.y, 0, e);
                const float R6 = seq_sum16(e);
#pragma unroll
                for (int i = 0; i < 16; ++i) F6[i] = add_rn(F6[i], e[i]);
                exact(y, w.z, w.w, 1, e);
                const float R4 = seq_sum16(e);
#pragma unroll
                for (int i = 0; i < 16; ++i) F4[i] = add_rn(F4[i], e[i]);
                row_sums(r, R6, R4);
            }
            tree_sums();
        }
        const bool row4 = E4r < E6r, col4 = E4c < E6c;       // ties and NaN keep map-to-6
        const uint8_t sf_r = static_cast<uint8_t>(row4 ? sf4 : sf6);

        // store the rowwise codes of the chosen candidate; gather the columnwise one's
        const int64_t nbr = K / 16;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const uint4 w = *reinterpret_cast<const uint4*>(piece(r, 0));
            const int64_t rowg = band * 16 + r;
            reinterpret_cast<uint2*>(a.codes)[(rowg * K + tile * 16) / 16] =
                row4 ? make_uint2(w.z, w.w) : make_uint2(w.x, w.y);
            a.scales[rowg * nbr + tile] = sf_r;
            lo[r] = col4 ? w.z : w.x;
            hi[r] = col4 ? w.w : w.y;
        }
        transpose8x8_nibbles(lo);          // rows 0-7,  cols 0-7
        transpose8x8_nibbles(lo + 8);      // rows 8-15, cols 0-7
        transpose8x8_nibbles(hi);          // rows 0-7,  cols 8-15
        transpose8x8_nibbles(hi + 8);      // rows 8-15, cols 8-15
        sf_c = col4 ? sf4 : sf6;
    }
    // columnwise output: x^T's row (tile0 * 16 + j) holds 8 code bytes of
    // each band, so the CTA's kBands bands give each of its 512 columns 32
    // consecutive bytes (one sector) and kBands consecutive scale bytes.  The
    // transposed words are staged in the tile buffer, once every thread is
    // done with its slots, and written column by column.
    __syncthreads();
    uint2* stg = reinterpret_cast<uint2*>(tile_s);
    if (own) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            stg[stage_index(warp, lane * 16 + c)] = make_uint2(lo[c], lo[8 + c]);
            stg[stage_index(warp, lane * 16 + 8 + c)] = make_uint2(hi[c], hi[8 + c]);
        }
    }
    scol[warp][lane] = static_cast<uint8_t>(sf_c);
    __syncthreads();
    uint2* cc = reinterpret_cast<uint2*>(a.codes_col);
#pragma unroll 4
    for (int q = tid; q < 512 * kBands; q += kTileThreads) {
        const int j = q / kBands, bb = q % kBands;          // column of the CTA, band of the CTA
        const int64_t col = tile0 * 16 + j, bnd = band0 + bb;
        if (col < K && bnd < nbands) {
            cc[col * nbands + bnd] = stg[stage_index(bb, j)];
            a.scales_col[col * nbands + bnd] = scol[bb][j >> 4];
        }
    }
    pdl_trigger();
}

// Plain 1x16 quantization with rowwise AND columnwise output, bf16 input,
// nearest rounding (either scale association): one thread per 16x16 tile,
// staged whole in shared memory as in k_tile_ts.  The tile's 16 rows are
// its rowwise blocks and its 16 columns its columnwise blocks (rows of x^T),
// each with its own scale; nothing is shared between them but the read of
// x, so no barrier is needed until the columnwise output is staged.  A row
// is read as its two 16-byte pieces; the columns are read as two half
// tiles (8 columns x 16 rows: piece h of every row, 64 words held in
// registers), each column's 16 values taken out of the words.  The
// columnwise codes and scale bytes leave as in k_tile_ts: one 32-byte run
// and four consecutive scale bytes per column of the CTA.
template <int RND, bool GS>
__global__ void __launch_bounds__(kTileThreads) k_tile_r1(const QuantArgs a) {
    extern __shared__ __align__(16) unsigned char tile_s[];   // [row][thread][32 bytes]
    __shared__ float rtab[GS ? 1 : 128];
    __shared__ uint8_t scol[kBands][512];       // columnwise scale bytes, [band][column of the CTA]
    if (!GS) fill_recip_table(rtab);
    pdl_wait();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t M = a.M, K = a.K;
    const int64_t band0 = static_cast<int64_t>(blockIdx.x) * kBands, band = band0 + warp;
    const int64_t tile0 = static_cast<int64_t>(blockIdx.y) * 32, tile = tile0 + lane;
    const int64_t nb = K / 16, nbands = M / 16;
    const bool own = band < nbands && tile < nb;
    const int64_t base = band * 16 * K + tile * 16;
    const uint32_t swz = piece_swizzle<2>(tid);
    auto slot = [&](int r) { return tile_s + (r * kTileThreads + tid) * 32; };
    auto piece = [&](int r, uint32_t c) { return slot(r) + ((c ^ swz) << 4); };
    if (own) {
        const unsigned char* gx = static_cast<const unsigned char*>(a.x) + base * 2;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            cp_async16(piece(r, 0), gx + static_cast<int64_t>(r) * K * 2);
            cp_async16(piece(r, 1), gx + static_cast<int64_t>(r) * K * 2 + 16);
            if ((r & 3) == 3) cp_async_commit();
        }
    }
    GScale g{0.0f, 1.0f, 1.0f};
    if (a.gamax_mode == NVFP4_GAMAX_TENSOR_GIVEN) {
        g.A = a.gamax[0];
        global_scales(g.A, a.bound, g.Senc, g.Sdec);
    }
    // one 1x16 block: codes and scale byte
    auto quant16 = [&](const float* y, uint32_t& w0, uint32_t& w1, uint32_t& sf) {
        const float b = absmax16(y);
        const float s6f = block_scale<GS>(b, g.Senc, RND == NVFP4_RTN_STD);
        sf = e4m3_encode(min_nd(s6f, 448.0f));
        const float d = e4m3_decode(sf);
        const float D = GS ? mul_rn(d, g.Sdec) : d;
        float q[16];
        encode_plain16<RND>(y, D, b, 0, a.pk, w0, w1, GS ? nullptr : rtab, sf, q, false);
    };
    uint32_t cw[16][2];                         // columnwise code words of the tile's columns
    if (own) {
        const int64_t nbr = K / 16;
        auto row_pass = [&](int r0) {           // rows r0 .. r0 + 3, rowwise blocks
#pragma unroll 2
            for (int r = r0; r < r0 + 4; ++r) {
                float y[16];
                lds16_swz<NVFP4_BF16>(slot(r), swz, y);
                uint32_t w0, w1, sf;
                quant16(y, w0, w1, sf);
                const int64_t rowg = band * 16 + r;
                reinterpret_cast<uint2*>(a.codes)[(rowg * K + tile * 16) / 16] = make_uint2(w0, w1);
                a.scales[rowg * nbr + tile] = static_cast<uint8_t>(sf);
            }
        };
        cp_async_wait<3>();
        row_pass(0);
        cp_async_wait<2>();
        row_pass(4);
        cp_async_wait<1>();
        row_pass(8);
        cp_async_wait<0>();
        row_pass(12);
#pragma unroll
        for (int h = 0; h < 2; ++h) {           // columns 8h .. 8h + 7
            uint32_t wv[16][4];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const uint4 u = *reinterpret_cast<const uint4*>(piece(r, h));
                wv[r][0] = u.x;
                wv[r][1] = u.y;
                wv[r][2] = u.z;
                wv[r][3] = u.w;
            }
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                float y[16];
#pragma unroll
                for (int r = 0; r < 16; ++r)
                    y[r] = __uint_as_float((c & 1) ? (wv[r][c >> 1] & 0xFFFF0000u) : (wv[r][c >> 1] << 16));
                uint32_t sf;
                quant16(y, cw[8 * h + c][0], cw[8 * h + c][1], sf);
                scol[warp][lane * 16 + 8 * h + c] = static_cast<uint8_t>(sf);
            }
        }
    }
    // columnwise output as in k_tile_ts, staged in the tile buffer once every
    // thread is done with its slots
    __syncthreads();
    uint2* stg = reinterpret_cast<uint2*>(tile_s);
    if (own) {
#pragma unroll
        for (int c = 0; c < 16; ++c) stg[stage_index(warp, lane * 16 + c)] = make_uint2(cw[c][0], cw[c][1]);
    }
    __syncthreads();
    uint2* cc = reinterpret_cast<uint2*>(a.codes_col);
#pragma unroll 4
    for (int q = tid; q < 512 * kBands; q += kTileThreads) {
        const int j = q / kBands, bb = q % kBands;          // column of the CTA, band of the CTA
        const int64_t col = tile0 * 16 + j, bnd = band0 + bb;
        if (col < K && bnd < nbands) {
            cc[col * nbands + bnd] = stg[stage_index(bb, j)];
            a.scales_col[col * nbands + bnd] = scol[bb][j];
        }
    }
    pdl_trigger();
}

// Four-over-six 16x16 with rowwise and columnwise output, fp32 input, four
// threads per tile: lanes 4t .. 4t+3 of a warp hold columns 0-3, 4-7, 8-11
// and 12-15 of tile t (8 tiles per warp, one band per warp, a CTA 4 bands x
// 8 tiles), so a thread's share, 16 rows x 4 fp32 (256 bytes), is staged in
// shared memory up front (32 KB per CTA, six CTAs per SM; with two threads
// per tile, 64 KB and three CTAs per SM, c4 ran 15 % slower).  The quad exchanges the tile amax and the column sums by
// shuffles: the width-16 tree's first level pairs lanes q and q^2 (columns j
// and j+8), its second level lanes q and q^1 (j and j+4), and the last two
// levels run in every lane alike.  On the exact path each row's element-
// order sum runs along the quad, each lane continuing its left neighbour's
// partial.  Row r's slot (16 bytes) takes, once read, the row's 4-code
// words of both candidates and 8 bytes of scratch.
constexpr int kTile4Bytes = 16 * kTileThreads * 16;

template <int ERR>
__global__ void __launch_bounds__(kTileThreads) k_tile_ts4(const QuantArgs a) {
    extern __shared__ __align__(16) unsigned char tile_s[];   // [row][thread][16 bytes]
    __shared__ float tenc[128];                 // encode reciprocal of every scale byte
    __shared__ uint8_t scol[kBands][8];         // columnwise scale byte of each tile
    pdl_wait();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, q = lane & 3;
    const int qbase = lane & 28;                // the quad's first lane
    const unsigned pm = 15u << qbase;           // the quad's lanes
    const int64_t M = a.M, K = a.K;
    const int64_t nb = K / 16, nbands = M / 16;
    const int64_t ntg = (nb + 7) / 8;           // CTA columns of 8 tiles (a 1D grid: K/128 may pass 65535)
    const int64_t cta = blockIdx.x;
    const int64_t band0 = (cta / ntg) * kBands, band = band0 + warp;
    const int64_t tile0 = (cta % ntg) * 8, tile = tile0 + (lane >> 2);
    const bool own = band < nbands && tile < nb;
    const int64_t base = band * 16 * K + tile * 16 + 4 * q;       // the thread's first element
    auto slot = [&](int r) { return tile_s + (r * kTileThreads + tid) * 16; };
    auto codes_at = [&](int r) { return reinterpret_cast<uint32_t*>(slot(r)); };   // 4-code words, both candidates
    auto scratch = [&](int r) { return reinterpret_cast<float2*>(slot(r) + 8); };
    if (own) {
        const unsigned char* gx = static_cast<const unsigned char*>(a.x) + base * 4;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            cp_async16(slot(r), gx + static_cast<int64_t>(r) * K * 4);
            if ((r & 3) == 3) cp_async_commit();
        }
    }
    GScale g{0.0f, 1.0f, 1.0f};
    if (a.gamax_mode == NVFP4_GAMAX_TENSOR_GIVEN) {
        g.A = a.gamax[0];
        global_scales(g.A, a.bound, g.Senc, g.Sdec);
    }
    const float C = mul_rn(6.0f, a.bound);
    for (int i = tid; i < 128; i += blockDim.x)
        tenc[i] = min_nd(div_rn(1.0f, mul_rn(e4m3_decode(static_cast<uint32_t>(i)), g.Sdec)), FLT_MAX);
    __syncthreads();

    auto load4 = [&](int r, float* y) {         // the thread's 4 elements of row r
        const float4 p = *reinterpret_cast<const float4*>(slot(r));
        y[0] = p.x; y[1] = p.y; y[2] = p.z; y[3] = p.w;
    };
    // the width-16 tree over the tile's 16 column sums, 4 per lane
    auto col_tree = [&](const float* F) {
        float t[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {           // level 1: column j + column j + 8
            const float o = __shfl_xor_sync(pm, F[i], 2);
            t[i] = q < 2 ? add_rn(F[i], o) : add_rn(o, F[i]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {           // level 2: (j, j + 8) + (j + 4, j + 12)
            const float o = __shfl_xor_sync(pm, t[i], 1);
            t[i] = (q & 1) == 0 ? add_rn(t[i], o) : add_rn(o, t[i]);
        }
        return add_rn(add_rn(t[0], t[2]), add_rn(t[1], t[3]));
    };
    uint32_t lo[4], hi[4];                      // columnwise code words of the thread's 4 columns
    uint32_t sf_c = 0;
    if (own) {
        // pass 0: tile amax, each copy group as it lands, then over the quad
        float b = 0.0f;
        auto amax4 = [&](int r0) {
#pragma unroll
            for (int r = r0; r < r0 + 4; ++r) {
                float y[4];
                load4(r, y);
#pragma unroll
                for (int i = 0; i < 4; ++i) b = max_nd(b, fabsf(y[i]));
            }
        };
        cp_async_wait<3>();
        amax4(0);
        cp_async_wait<2>();
        amax4(4);
        cp_async_wait<1>();
        amax4(8);
        cp_async_wait<0>();
        amax4(12);
        b = max_nd(b, __shfl_xor_sync(pm, b, 1));
        b = max_nd(b, __shfl_xor_sync(pm, b, 2));
        const float s6f = block_s6f<true>(b, g.Senc);
        const uint32_t sf6 = e4m3_encode(min_nd(s6f, 448.0f));
        const uint32_t sf4 = e4m3_encode(min_nd(mul_rn(s6f, 1.5f), 448.0f));
        const float enc6 = tenc[sf6], enc4 = tenc[sf4];
        const float d6 = e4m3_decode(sf6), d4 = e4m3_decode(sf4);
        const float K6 = div_rn(mul_rn(d6, g.A), C), K4 = div_rn(mul_rn(d4, g.A), C);

        // pass 1: both candidates' codes and scaled-domain approximate errors,
        // the 4 column sums in row order
        float F6[4], F4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) F6[i] = F4[i] = 0.0f;
        const uint64_t ENC6 = pack2(enc6, enc6), ENC4 = pack2(enc4, enc4);
        auto candidate = [&](const float* y, uint64_t enc2, uint32_t& w, float* e) {
            float v[4];
#pragma unroll
            for (int i = 0; i < 4; i += 2) unpack2(mul2(pack2(y[i], y[i + 1]), enc2), v[i], v[i + 1]);
            uint32_t h[2];
            w = e2m1_encode4_dec(v, h);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                sub_f16x2_f32(h[j], v[2 * j], v[2 * j + 1], e[2 * j], e[2 * j + 1]);
                if (ERR != NVFP4_ERR_MAE) {
                    const uint64_t D = pack2(e[2 * j], e[2 * j + 1]);
                    unpack2(mul2(D, D), e[2 * j], e[2 * j + 1]);
                }
            }
            if (ERR == NVFP4_ERR_MAE) {
#pragma unroll
                for (int i = 0; i < 4; ++i) e[i] = fabsf(e[i]);
            }
        };
        auto add4 = [&](float* F, const float* e) {
#pragma unroll
            for (int i = 0; i < 4; i += 2) unpack2(add2(pack2(F[i], F[i + 1]), pack2(e[i], e[i + 1])), F[i], F[i + 1]);
        };
#pragma unroll 4
        for (int r = 0; r < 16; ++r) {
            float y[4], e[4];
            load4(r, y);
            uint32_t w6, w4;
            candidate(y, ENC6, w6, e);
            add4(F6, e);
            candidate(y, ENC4, w4, e);
            add4(F4, e);
            *codes_at(r) = w6 | (w4 << 16);
        }
        float E6c = col_tree(F6), E4c = col_tree(F4);
        {   // back from the scaled domain: E^ = RN(K * S'), or RN(RN(K * K) * S')
            const float k6 = ERR == NVFP4_ERR_MAE ? K6 : mul_rn(K6, K6);
            const float k4 = ERR == NVFP4_ERR_MAE ? K4 : mul_rn(K4, K4);
            E6c = mul_rn(k6, E6c);
            E4c = mul_rn(k4, E4c);
        }
        float E6r = E6c, E4r = E4c;
        if (!tile_sums_decide<ERR>(E6c, E4c, K6, K4, b)) {     // all four lanes alike
            // the exact sums: error values |dq| of each grid magnitude (row
            // 8 + k's scratch: map-to-6, map-to-4), x read again
            const float G8[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
#pragma unroll
            for (int k = 0; k < 8; ++k)
                *scratch(8 + k) = make_float2(div_rn(mul_rn(mul_rn(G8[k], d6), g.A), C),
                                              div_rn(mul_rn(mul_rn(G8[k], d4), g.A), C));
            auto exact = [&](const float* y, uint32_t w, int c, float* e) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t k = (w >> (4 * i)) & 7u;
                    const float2 t = *scratch(8 + static_cast<int>(k));
                    const float diff = sub_rn(c ? t.y : t.x, fabsf(y[i]));
                    e[i] = (ERR == NVFP4_ERR_MAE) ? fabsf(diff) : mul_rn(diff, diff);
                }
            };
#pragma unroll
            for (int i = 0; i < 4; ++i) F6[i] = F4[i] = 0.0f;
#pragma unroll 1
            for (int r = 0; r < 16; ++r) {
                float y[4], e6[4], e4[4];
                const float4 p = __ldg(reinterpret_cast<const float4*>(
                    static_cast<const unsigned char*>(a.x) + (base + static_cast<int64_t>(r) * K) * 4));
                y[0] = p.x; y[1] = p.y; y[2] = p.z; y[3] = p.w;
                const uint32_t w = *codes_at(r);
                exact(y, w & 0xFFFFu, 0, e6);
                exact(y, w >> 16, 1, e4);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    F6[i] = add_rn(F6[i], e6[i]);
                    F4[i] = add_rn(F4[i], e4[i]);
                }
                // row r in element order along the quad: lane 0 from zero,
                // each next lane continuing its left neighbour's partial
                float s6 = 0.0f, s4 = 0.0f;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if (q == k) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            s6 = add_rn(s6, e6[i]);
                            s4 = add_rn(s4, e4[i]);
                        }
                    }
                    if (k < 3) {
                        const float t6 = __shfl_sync(pm, s6, qbase + k), t4 = __shfl_sync(pm, s4, qbase + k);
                        if (q == k + 1) {
                            s6 = t6;
                            s4 = t4;
                        }
                    }
                }
                if (q == 3) {                   // the width-16 tree's first level: row i + row i + 8
                    float2* p2 = scratch(r & 7);
                    if (r >= 8) {
                        const float2 t = *p2;
                        s6 = add_rn(t.x, s6);
                        s4 = add_rn(t.y, s4);
                    }
                    *p2 = make_float2(s6, s4);
                }
            }
            float R6 = 0.0f, R4 = 0.0f;
            if (q == 3) {
                float S6[8], S4[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float2 t = *scratch(i);
                    S6[i] = t.x;
                    S4[i] = t.y;
                }
                R6 = tree16_upper(S6);
                R4 = tree16_upper(S4);
            }
            E6r = __shfl_sync(pm, R6, qbase + 3);
            E4r = __shfl_sync(pm, R4, qbase + 3);
            E6c = col_tree(F6);
            E4c = col_tree(F4);
        }
        const bool row4 = E4r < E6r, col4 = E4c < E6c;       // ties and NaN keep map-to-6
        const uint8_t sf_r = static_cast<uint8_t>(row4 ? sf4 : sf6);

        // rowwise codes of the chosen candidate (the thread's 4 codes of each
        // row); the columnwise candidate's codes transposed (rows 0-7 and 8-15,
        // the 16-bit words padded to 8x8 nibble blocks)
        const int64_t nbr = K / 16;
        uint16_t* codes16 = reinterpret_cast<uint16_t*>(a.codes);
        uint32_t cl[8], ch[8];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const uint32_t w = *codes_at(r);
            const int64_t rowg = band * 16 + r;
            codes16[(rowg * K + tile * 16) / 4 + q] = static_cast<uint16_t>(row4 ? (w >> 16) : (w & 0xFFFFu));
            if (q == 0) a.scales[rowg * nbr + tile] = sf_r;
            const uint32_t c = col4 ? (w >> 16) : (w & 0xFFFFu);
            if (r < 8) cl[r] = c;
            else ch[r - 8] = c;
        }
        transpose8x8_nibbles(cl);          // rows 0-7: word c = column c
        transpose8x8_nibbles(ch);          // rows 8-15
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            lo[c] = cl[c];
            hi[c] = ch[c];
        }
        sf_c = col4 ? sf4 : sf6;
    }
    // columnwise output (the CTA's 128 columns), staged in the tile buffer once
    // every thread is done with its slots
    __syncthreads();
    uint2* stg = reinterpret_cast<uint2*>(tile_s);
    if (own) {
#pragma unroll
        for (int c = 0; c < 4; ++c) stg[stage_index(warp, (lane >> 2) * 16 + 4 * q + c)] = make_uint2(lo[c], hi[c]);
        if (q == 0) scol[warp][lane >> 2] = static_cast<uint8_t>(sf_c);
    }
    __syncthreads();
    uint2* cc = reinterpret_cast<uint2*>(a.codes_col);
#pragma unroll 4
    for (int qq = tid; qq < 128 * kBands; qq += kTileThreads) {
        const int j = qq / kBands, bb = qq % kBands;        // column of the CTA, band of the CTA
        const int64_t col = tile0 * 16 + j, bnd = band0 + bb;
        if (col < K && bnd < nbands) {
            cc[col * nbands + bnd] = stg[stage_index(bb, j)];
            a.scales_col[col * nbands + bnd] = scol[bb][j >> 4];
        }
    }
    pdl_trigger();
}

// Plain (map-to-6) 16x16 quantization with rowwise AND columnwise output:
// the tile's one scale serves both outputs and x^T's codes are x's codes
// transposed (stochastic rounding draws are keyed on x's index), so a thread
// owns a tile as in k_tile_ts, finds the tile amax in a first walk over its
// rows and encodes each row in a second (from L2), storing the row's codes
// and shifting its nibbles into the column words: rows come in pairs, whose
// nibbles are interleaved into one byte per column (low nibble the even row)
// and moved in at the top of that column's word, so after rows 0-7 (and
// again 8-15) word c holds column c with row r in nibble r % 8.  The
// columnwise output is staged and written as in k_tile_ts.
template <int DT, int RND, bool GS>
__global__ void __launch_bounds__(kTileThreads) k_tile_p(const QuantArgs a) {
    using Rg = TilePRing<DT>;
    __shared__ __align__(16) unsigned char ring[Rg::BYTES];
    __shared__ uint2 stg[kBands * 512];          // columnwise words, [stage_index]
    __shared__ uint8_t scol[kBands][32];
    __shared__ float rtab[GS ? 1 : 128];
    if (!GS) fill_recip_table(rtab);
    pdl_wait();
    GScale g{0.0f, 1.0f, 1.0f};
    if (a.gamax_mode == NVFP4_GAMAX_TENSOR_GIVEN) {
        g.A = a.gamax[0];
        global_scales(g.A, a.bound, g.Senc, g.Sdec);
    }
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t M = a.M, K = a.K;
    const int64_t band0 = static_cast<int64_t>(blockIdx.x) * kBands, band = band0 + warp;
    const int64_t tile0 = static_cast<int64_t>(blockIdx.y) * 32, tile = tile0 + lane;
    const int64_t nb = K / 16, nbands = M / 16;
    uint32_t colw[16], top[16];
    uint32_t sf = 0;
    if (band < nbands && tile < nb) {
        const int64_t base = band * 16 * K + tile * 16;
        const unsigned char* gx = static_cast<const unsigned char*>(a.x) + base * (Rg::XB / 16);
        const int64_t row_bytes = K * (Rg::XB / 16);
        unsigned char* slot0 = ring + tid * Rg::XB;
        auto issue = [&](int j) {                // row read j (0..31) is tile row j % 16
            if (j < 32) {
                const unsigned char* src = gx + static_cast<int64_t>(j & 15) * row_bytes;
                unsigned char* dst = slot0 + (j % Rg::SLOTS) * (kTileThreads * Rg::XB);
#pragma unroll
                for (int c = 0; c < Rg::XB / 16; ++c) cp_async16(dst + 16 * c, src + 16 * c);
            }
            cp_async_commit();
        };
        auto next_row = [&](int j, float* y) {
            issue(j + Rg::SLOTS - 1);
            cp_async_wait<Rg::SLOTS - 1>();
            lds16<DT>(slot0 + (j % Rg::SLOTS) * (kTileThreads * Rg::XB), y);
        };
#pragma unroll
        for (int j = 0; j < Rg::SLOTS - 1; ++j) issue(j);

        // pass 0: tile amax (bf16: on the packed pairs)
        float y[16];
        float b = 0.0f;
        if constexpr (DT == NVFP4_BF16) {
            uint32_t m2 = 0u;
#pragma unroll 1
            for (int r = 0; r < 16; ++r) {
                issue(r + Rg::SLOTS - 1);
                cp_async_wait<Rg::SLOTS - 1>();
                const uint4* p = reinterpret_cast<const uint4*>(slot0 + (r % Rg::SLOTS) * (kTileThreads * Rg::XB));
                const uint4 u = p[0], v = p[1];
                m2 = absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(m2, u.x), u.y), u.z), u.w);
                m2 = absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(m2, v.x), v.y), v.z), v.w);
            }
            b = max_nd(__uint_as_float(m2 << 16), __uint_as_float(m2 & 0xFFFF0000u));
        } else {
#pragma unroll 1
            for (int r = 0; r < 16; ++r) {
                next_row(r, y);
                b = max_nd(b, absmax16(y));
            }
        }
        const float s6f = block_scale<GS>(b, g.Senc, RND == NVFP4_RTN_STD);
        sf = e4m3_encode(min_nd(s6f, 448.0f));
        const float d = e4m3_decode(sf);
        const float D = GS ? mul_rn(d, g.Sdec) : d;

        // pass 1: encode each row; rowwise codes stored, columnwise gathered
#pragma unroll
        for (int c = 0; c < 16; ++c) colw[c] = top[c] = 0u;
        uint32_t pw0 = 0u, pw1 = 0u;             // the pair's even row
        const uint64_t idx_row0 = (static_cast<uint64_t>(a.row_offset) + static_cast<uint64_t>(band * 16)) *
                                      static_cast<uint64_t>(K) + static_cast<uint64_t>(tile * 16);
#pragma unroll 1
        for (int r = 0; r < 16; ++r) {
            next_row(16 + r, y);
            uint32_t wd[16];
            if (RND == NVFP4_SR) sr_words16(idx_row0 + static_cast<uint64_t>(r) * static_cast<uint64_t>(K),
                                            a.pk, wd);
            uint32_t w0, w1;
            float q[16];
            encode_plain16_words<RND>(y, D, b, wd, w0, w1, GS ? nullptr : rtab, sf, q, false);
            const int64_t rowg = band * 16 + r;
            reinterpret_cast<uint2*>(a.codes)[(rowg * K + tile * 16) / 16] = make_uint2(w0, w1);
            a.scales[rowg * nb + tile] = static_cast<uint8_t>(sf);
            if ((r & 1) == 0) {
                pw0 = w0;
                pw1 = w1;
            } else {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t e = h ? pw1 : pw0, o = h ? w1 : w0;
                    // byte k of ev: column 2k of both rows; of od: column 2k + 1
                    const uint32_t ev = (e & 0x0F0F0F0Fu) | ((o & 0x0F0F0F0Fu) << 4);
                    const uint32_t od = ((e >> 4) & 0x0F0F0F0Fu) | (o & 0xF0F0F0F0u);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        // word >> 8 with byte k of the pair's bytes on top
                        colw[8 * h + 2 * k] = __byte_perm(colw[8 * h + 2 * k], ev, 0x0321u | ((4u + k) << 12));
                        colw[8 * h + 2 * k + 1] = __byte_perm(colw[8 * h + 2 * k + 1], od, 0x0321u | ((4u + k) << 12));
                    }
                }
                if (r == 7) {
#pragma unroll
                    for (int c = 0; c < 16; ++c) top[c] = colw[c];
                }
            }
        }
        cp_async_wait<0>();
#pragma unroll
        for (int c = 0; c < 16; ++c) stg[stage_index(warp, lane * 16 + c)] = make_uint2(top[c], colw[c]);
    }
    scol[warp][lane] = static_cast<uint8_t>(sf);
    __syncthreads();
    uint2* cc = reinterpret_cast<uint2*>(a.codes_col);
#pragma unroll 4
    for (int q = tid; q < 512 * kBands; q += kTileThreads) {
        const int j = q / kBands, bb = q % kBands;          // column of the CTA, band of the CTA
        const int64_t col = tile0 * 16 + j, bnd = band0 + bb;
        if (col < K && bnd < nbands) {
            cc[col * nbands + bnd] = stg[stage_index(bb, j)];
            a.scales_col[col * nbands + bnd] = scol[bb][j >> 4];
        }
    }
    pdl_trigger();
}

// ---------------------------------------------------------------------------------------------
template <typename KernelT>
int launch_rowowner(KernelT kernel, const QuantArgs& a, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>((a.M / 16 + kRowBands - 1) / kRowBands),
                    static_cast<unsigned>((a.K / 16 + 15) / 16));
    launch_pdl(kernel, grid, kThreads, 0, s, a);
    return static_cast<int>(cudaGetLastError());
}

// the thread-per-tile kernels: CTA = kBands bands x 32 tiles
template <typename KernelT>
int launch_tile(KernelT kernel, const QuantArgs& a, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>((a.M / 16 + kBands - 1) / kBands),
                    static_cast<unsigned>((a.K / 16 + 31) / 32));
    launch_pdl(kernel, grid, kTileThreads, 0, s, a);
    return static_cast<int>(cudaGetLastError());
}

template <int ERR>
int launch_tile_ts4(const QuantArgs& a, cudaStream_t s) {
    static int configured_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_dev != dev) {
        cudaFuncSetAttribute(k_tile_ts4<ERR>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
        configured_dev = dev;
    }
    const int64_t ctas = ((a.M / 16 + kBands - 1) / kBands) * ((a.K / 16 + 7) / 8);
    launch_pdl(k_tile_ts4<ERR>, dim3(static_cast<unsigned>(ctas)), kTileThreads, kTile4Bytes, s, a);
    return static_cast<int>(cudaGetLastError());
}

template <int DT, int ERR>
int launch_tile_4o6(const QuantArgs& a, cudaStream_t s) {
    if constexpr (DT == NVFP4_F32) {
        return launch_tile_ts4<ERR>(a, s);
    } else {
        static int configured_dev = -1;
        int dev = 0;
        cudaGetDevice(&dev);
        if (configured_dev != dev) {
            cudaFuncSetAttribute(k_tile_ts<ERR>, cudaFuncAttributeMaxDynamicSharedMemorySize, kStagedTileBytes);
            cudaFuncSetAttribute(k_tile_ts<ERR>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
            configured_dev = dev;
        }
        const dim3 grid(static_cast<unsigned>((a.M / 16 + kBands - 1) / kBands),
                        static_cast<unsigned>((a.K / 16 + 31) / 32));
        launch_pdl(k_tile_ts<ERR>, grid, kTileThreads, kStagedTileBytes, s, a);
        return static_cast<int>(cudaGetLastError());
    }
}

// k_tile_r1: 64 KB of dynamic shared memory (set once per device)
template <int RND, bool GS>
int launch_tile_r1(const QuantArgs& a, cudaStream_t s) {
    static int configured_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_dev != dev) {
        cudaFuncSetAttribute(k_tile_r1<RND, GS>, cudaFuncAttributeMaxDynamicSharedMemorySize, kStagedTileBytes);
        cudaFuncSetAttribute(k_tile_r1<RND, GS>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
        configured_dev = dev;
    }
    const dim3 grid(static_cast<unsigned>((a.M / 16 + kBands - 1) / kBands),
                    static_cast<unsigned>((a.K / 16 + 31) / 32));
    launch_pdl(k_tile_r1<RND, GS>, grid, kTileThreads, kStagedTileBytes, s, a);
    return static_cast<int>(cudaGetLastError());
}

// rowwise + columnwise outputs (no residual)
template <int DT, int BLK>
int tiles_dispatch_blk(const QuantArgs& a, cudaStream_t s) {
    if (a.err_mode != NVFP4_ERR_NONE) {
        if (BLK == NVFP4_BLOCK_16X16)
            return a.err_mode == NVFP4_ERR_MAE ? launch_tile_4o6<DT, NVFP4_ERR_MAE>(a, s)
                                               : launch_tile_4o6<DT, NVFP4_ERR_MSE>(a, s);
        return a.err_mode == NVFP4_ERR_MAE ? launch_rowowner(k_tiles_rows<DT, BLK, NVFP4_ERR_MAE, NVFP4_RTN, true>, a, s)
                                           : launch_rowowner(k_tiles_rows<DT, BLK, NVFP4_ERR_MSE, NVFP4_RTN, true>, a, s);
    }
    const bool gs = a.gamax_mode != NVFP4_GAMAX_NONE;
    if (BLK == NVFP4_BLOCK_16X16) {
        if (a.rounding == NVFP4_SR)
            return gs ? launch_tile(k_tile_p<DT, NVFP4_SR, true>, a, s) : launch_tile(k_tile_p<DT, NVFP4_SR, false>, a, s);
        if (a.rounding == NVFP4_RTN_STD)
            return gs ? launch_tile(k_tile_p<DT, NVFP4_RTN_STD, true>, a, s)
                      : launch_tile(k_tile_p<DT, NVFP4_RTN_STD, false>, a, s);
        return gs ? launch_tile(k_tile_p<DT, NVFP4_RTN, true>, a, s) : launch_tile(k_tile_p<DT, NVFP4_RTN, false>, a, s);
    }
    if (a.rounding == NVFP4_SR)
        return gs ? launch_rowowner(k_tiles_rows<DT, BLK, NVFP4_ERR_NONE, NVFP4_SR, true>, a, s)
                  : launch_rowowner(k_tiles_rows<DT, BLK, NVFP4_ERR_NONE, NVFP4_SR, false>, a, s);
    if constexpr (DT == NVFP4_BF16) {           // nearest rounding, bf16: a thread per staged tile
        if (a.rounding == NVFP4_RTN_STD)
            return gs ? launch_tile_r1<NVFP4_RTN_STD, true>(a, s) : launch_tile_r1<NVFP4_RTN_STD, false>(a, s);
        return gs ? launch_tile_r1<NVFP4_RTN, true>(a, s) : launch_tile_r1<NVFP4_RTN, false>(a, s);
    }
    if (a.rounding == NVFP4_RTN_STD)
        return gs ? launch_rowowner(k_tiles_rows<DT, BLK, NVFP4_ERR_NONE, NVFP4_RTN_STD, true>, a, s)
                  : launch_rowowner(k_tiles_rows<DT, BLK, NVFP4_ERR_NONE, NVFP4_RTN_STD, false>, a, s);
    return gs ? launch_rowowner(k_tiles_rows<DT, BLK, NVFP4_ERR_NONE, NVFP4_RTN, true>, a, s)
              : launch_rowowner(k_tiles_rows<DT, BLK, NVFP4_ERR_NONE, NVFP4_RTN, false>, a, s);
}

template <int DT>
int tiles_dispatch(const QuantArgs& a, cudaStream_t s) {
    return a.block == NVFP4_BLOCK_16X16 ? tiles_dispatch_blk<DT, NVFP4_BLOCK_16X16>(a, s)
                                        : tiles_dispatch_blk<DT, NVFP4_BLOCK_1X16>(a, s);
}

}  // namespace

int launch_quantize_tiles(const QuantArgs& a, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return a.dtype == NVFP4_BF16 ? tiles_dispatch<NVFP4_BF16>(a, s) : tiles_dispatch<NVFP4_F32>(a, s);
}

}  // namespace nvfp4
