// nvfp4_aux.cu -- global amax and dequantize kernels for sm_103a.
//
// amax: max |x (+ residual)| with NaN dropped, per tensor or per row, the
// global scale's input ("Add NVFP4 four-over-six (row-wise) quantization to
// the training prototype", What: scalar vs (rows,) global_amax; CuTe DSL
// kernel (SM100), Design: NaN-dropping max).
// dequantize: (q * dec(scale)) * S_dec ("fp4-train", API: dequantize).
#include "nvfp4_block.cuh"

namespace nvfp4 {
namespace {

constexpr int kThreads = 256;
constexpr unsigned kFull = 0xFFFFFFFFu;

template <int DT, bool EF>
__device__ __forceinline__ float block_absmax(const void* x, const float* res, int64_t e0) {
    float y[16];
    load16<DT>(x, e0, y);
    if (EF) {
        float r[16];
        load16_f32(res, e0, r);
#pragma unroll
        for (int i = 0; i < 16; ++i) y[i] = add_rn(y[i], r[i]);
    }
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) m = max_nd(m, fabsf(y[i]));
    return m;
}

__device__ __forceinline__ float warp_max(float m) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max_nd(m, __shfl_xor_sync(kFull, m, o));
    return m;
}

// Max of |x (+ r)| over one 8-element vector: 16 (bf16) or 32 (fp32) bytes
// of x, 32 bytes of the residual.
template <int DT, bool EF>
struct AmaxVec {
    uint4 x[DT == NVFP4_BF16 ? 1 : 2];
    uint4 r[EF ? 2 : 1];
    __device__ void load(const void* xp, const float* rp, int64_t v) {
        const uint4* px = static_cast<const uint4*>(xp) + v * (DT == NVFP4_BF16 ? 1 : 2);
#pragma unroll
        for (int k = 0; k < (DT == NVFP4_BF16 ? 1 : 2); ++k) x[k] = __ldg(px + k);
        if (EF) {
            const uint4* pr = reinterpret_cast<const uint4*>(rp) + v * 2;
            r[0] = __ldg(pr);
            r[1] = __ldg(pr + 1);
        }
    }
    __device__ float absmax() const {
        float y[8];
        if (DT == NVFP4_BF16) {
            const uint32_t w[4] = {x[0].x, x[0].y, x[0].z, x[0].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                y[2 * i] = __uint_as_float(w[i] << 16);
                y[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
            }
        } else {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                y[4 * k] = __uint_as_float(x[k].x);
                y[4 * k + 1] = __uint_as_float(x[k].y);
                y[4 * k + 2] = __uint_as_float(x[k].z);
                y[4 * k + 3] = __uint_as_float(x[k].w);
            }
        }
        if (EF) {
            const uint32_t rw[8] = {r[0].x, r[0].y, r[0].z, r[0].w, r[1].x, r[1].y, r[1].z, r[1].w};
#pragma unroll
            for (int i = 0; i < 8; ++i) y[i] = add_rn(y[i], __uint_as_float(rw[i]));
        }
        float m = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) m = max_nd(m, fabsf(y[i]));
        return m;
    }
};

// Per-tensor amax; *out must hold +0 on entry.  The tensor is read as 8-element
// vectors, kAmaxUnroll per thread and step, all loads issued before the max
// (consecutive lanes on consecutive vectors).  The maximum of non-negative
// floats orders like their bit patterns, so an unsigned atomic max is exact.
constexpr int kAmaxUnroll = 4;

// bf16 without a residual keeps its running maximum as a packed pair of bf16
// magnitudes (absmax_bf16x2: exact, NaN-dropping) and widens it once at the end.
// The per-tensor amax's zero, as a kernel so that the stream keeps
// programmatic launch edges between kernels (a memset between two kernels
// ends the overlap of one's tail with the next's launch).  It waits for the
// previous kernel, which may still read the old amax.
__global__ void k_amax_zero(float* out) {
    pdl_wait();
    out[0] = 0.0f;
    pdl_trigger();
}

template <int DT, bool EF>
__global__ void __launch_bounds__(kThreads) k_amax_tensor(const void* x, const float* res,
                                                          int64_t nvec, float* out) {
    __shared__ float part[kThreads / 32];
    constexpr bool PACKED = DT == NVFP4_BF16 && !EF;
    pdl_wait();
    float m = 0.0f;
    uint32_t m2 = 0u;
    const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x * kAmaxUnroll;
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x * kAmaxUnroll + threadIdx.x; base < nvec;
         base += step) {
        AmaxVec<DT, EF> v[kAmaxUnroll];
#pragma unroll
        for (int k = 0; k < kAmaxUnroll; ++k)
            if (base + k * kThreads < nvec) v[k].load(x, res, base + k * kThreads);
#pragma unroll
        for (int k = 0; k < kAmaxUnroll; ++k) {
            if (base + k * kThreads < nvec) {
                if constexpr (PACKED) {
                    m2 = absmax_bf16x2(absmax_bf16x2(m2, v[k].x[0].x), v[k].x[0].y);
                    m2 = absmax_bf16x2(absmax_bf16x2(m2, v[k].x[0].z), v[k].x[0].w);
                } else {
                    m = max_nd(m, v[k].absmax());
                }
            }
        }
    }
    if constexpr (PACKED) m = max_nd(__uint_as_float(m2 << 16), __uint_as_float(m2 & 0xFFFF0000u));
    pdl_trigger();
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x < 32) {
        m = threadIdx.x < kThreads / 32 ? part[threadIdx.x] : 0.0f;
        m = warp_max(m);
        if (threadIdx.x == 0) atomicMax(reinterpret_cast<unsigned int*>(out), __float_as_uint(m));
    }
}

// Per-row amax: one warp per row.
template <int DT, bool EF>
__global__ void __launch_bounds__(kThreads) k_amax_rows(const void* x, const float* res, int64_t M,
                                                        int64_t K, float* out) {
    const int64_t row = static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5);
    pdl_wait();
    if (row >= M) return;
    const int lane = threadIdx.x & 31;
    float m = 0.0f;
    for (int64_t b = lane; b < K / 16; b += 32) m = max_nd(m, block_absmax<DT, EF>(x, res, row * K + b * 16));
    pdl_trigger();
    m = warp_max(m);
    if (lane == 0) out[row] = m;
}

// dequantized values (q * d) * S_dec of one block
__device__ __forceinline__ void dequant_values(const DequantArgs& a, int64_t blk, uint32_t w0, uint32_t w1,
                                               uint32_t sf, float Sdec, bool per_row, int64_t bpr, float* v) {
    float Sd = Sdec;
    if (per_row) {
        float se;
        global_scales(a.gamax[blk / bpr], a.bound, se, Sd);
    }
    const float d = e4m3_decode(sf);
    float q[16];
    e2m1_decode8(w0, q);
    e2m1_decode8(w1, q + 8);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = mul_rn(mul_rn(q[i], d), Sd);
}

// Four blocks per thread per step, interleaved across the warp (lane l takes
// blocks base + l, +32, +64, +96) so every load covers consecutive blocks;
// all four blocks' codes and scales are loaded first.  The 32 blocks of one
// group are contiguous in the output too: the warp passes them through a
// shared buffer (16-byte chunk c of lane l at CH*l + (c ^ swz(l)), which
// keeps both the writes and the reads at the minimum of shared-memory
// wavefronts) so that store instruction c of lane l writes chunk 32 c + l,
// 512 consecutive bytes per instruction.
template <int ODT>
__global__ void __launch_bounds__(kThreads) k_dequant(const DequantArgs a) {
    constexpr int CH = ODT == NVFP4_BF16 ? 2 : 4;          // 16-byte output chunks per block
    __shared__ uint4 wst[kThreads / 32][32 * CH];
    pdl_wait();
    const int64_t bpr = a.K / 16;
    const int64_t nblk = a.M * bpr;
    float Senc = 1.0f, Sdec = 1.0f;
    const bool per_tensor = a.gamax_mode == NVFP4_GAMAX_TENSOR || a.gamax_mode == NVFP4_GAMAX_TENSOR_GIVEN;
    const bool per_row = a.gamax_mode == NVFP4_GAMAX_ROW || a.gamax_mode == NVFP4_GAMAX_ROW_GIVEN;
    if (per_tensor) global_scales(a.gamax[0], a.bound, Senc, Sdec);
    const int lane = threadIdx.x & 31;
    uint4* buf = wst[threadIdx.x >> 5];
    auto pos = [](int l, int c) { return CH * l + (c ^ ((l / (8 / CH)) & (CH - 1))); };
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const uint2* codes = reinterpret_cast<const uint2*>(a.codes);
    uint4* out = static_cast<uint4*>(a.out);
    for (int64_t base = warp * 128; base < nblk; base += nwarps * 128) {   // warp-uniform
        uint2 w[4];
        uint32_t sf[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t blk = base + 32 * k + lane;
            if (blk < nblk) {
                w[k] = __ldg(codes + blk);
                sf[k] = __ldg(a.scales + blk);
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t blk0 = base + 32 * k;                 // the group's first block
            if (blk0 + lane < nblk) {
                float v[16];
                dequant_values(a, blk0 + lane, w[k].x, w[k].y, sf[k], Sdec, per_row, bpr, v);
                if (ODT == NVFP4_BF16) {
                    uint32_t h[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        h[i] = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v[2 * i]))) |
                               (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v[2 * i + 1]))) << 16);
                    buf[pos(lane, 0)] = make_uint4(h[0], h[1], h[2], h[3]);
                    buf[pos(lane, 1)] = make_uint4(h[4], h[5], h[6], h[7]);
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        buf[pos(lane, c)] = make_uint4(__float_as_uint(v[4 * c]), __float_as_uint(v[4 * c + 1]),
                                                       __float_as_uint(v[4 * c + 2]), __float_as_uint(v[4 * c + 3]));
                }
            }
            __syncwarp();
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                const int q = 32 * c + lane;
                if (blk0 + q / CH < nblk) out[blk0 * CH + q] = buf[pos(q / CH, q % CH)];
            }
            __syncwarp();
        }
    }
    pdl_trigger();
}

// out[i] = the plain path's division a[i] / b[i] (its exact, stochastic-
// rounding form), with the block amax taken as |a[i]|; an E4M3-valued divisor
// takes the one-step form the kernels use without a global scale.
// out[2i], out[2i+1] = the two f16 halves of q[i] minus v[2i], v[2i+1], as
// the certified four-over-six sums take them
__global__ void __launch_bounds__(kThreads) k_probe_sub_f16(const uint32_t* q, const float* v, float* out,
                                                            int64_t n) {
    pdl_wait();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
        float d0, d1;
        sub_f16x2_f32(q[i], v[2 * i], v[2 * i + 1], d0, d1);
        out[2 * i] = d0;
        out[2 * i + 1] = d1;
    }
    pdl_trigger();
}

__global__ void __launch_bounds__(kThreads) k_probe_divide(const float* a, const float* b,
                                                           float* out, int64_t n) {
    pdl_wait();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
        const float y = a[i], D = b[i];
        const bool fast = plain_fast(D, fabsf(y));
        const uint32_t sf = e4m3_encode(D);
        if (fast && D > 0.0f && D <= 448.0f && e4m3_decode(sf) == D) {
            out[i] = plain_quotient<true, true>(y, D, div_rn(1.0f, D), fast);   // E4M3 divisor form
        } else {
            const float r = fast ? div_rn(1.0f, D) : 0.0f;
            out[i] = plain_quotient<true>(y, D, r, fast);
        }
    }
}

// out holds the e2m1 codes of the fp32 bit patterns first, first + 1, ...,
// first + n - 1, packed like quantized codes (pattern 2j in the low nibble of
// byte j; for odd n the last high nibble is 0), encoded by the routine every
// quantize kernel uses.
__global__ void __launch_bounds__(kThreads) k_probe_e2m1(uint32_t first, int64_t n, uint8_t* out) {
    pdl_wait();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g * 8 < n; g += stride) {
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(first + static_cast<uint32_t>(g * 8 + i));
        const uint32_t w = e2m1_encode8(v);
        if (g * 8 + 8 <= n) {
            reinterpret_cast<uint32_t*>(out)[g] = w;
        } else {
            for (int64_t b = 0; 8 * g + 2 * b < n; ++b) {
                const uint32_t byte = (w >> (8 * b)) & 0xFFu;
                out[4 * g + b] = static_cast<uint8_t>(8 * g + 2 * b + 1 < n ? byte : byte & 0x0Fu);
            }
        }
    }
}

// S_enc[i], S_dec[i] of the global amaxes gamax[i] (the global_scales step
// every quantize and dequantize kernel runs), for consumers that apply the
// decode scales themselves.
__global__ void __launch_bounds__(kThreads) k_global_scales(const float* gamax, int64_t n, float bound,
                                                            float* s_enc, float* s_dec) {
    pdl_wait();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
        float enc, dec;
        global_scales(gamax[i], bound, enc, dec);
        if (s_enc) s_enc[i] = enc;
        if (s_dec) s_dec[i] = dec;
    }
}

int grid_for(int64_t nblk) {
    const int64_t want = (nblk + kThreads - 1) / kThreads;
    const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
    return static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
}

// Scale re-layout for the block-scaled matrix multiply: one thread per
// (row, group of 4 columns) of the padded matrix, i.e. one 4-byte word of the
// output: tile (r/128, c/4), word (r % 32) * 4 + (r % 128) / 32 of the tile.
__global__ void __launch_bounds__(kThreads) k_scales_mma(const uint8_t* __restrict__ in, int64_t rows,
                                                         int64_t cols, int64_t R, int64_t C4,
                                                         uint32_t* __restrict__ out) {
    pdl_wait();
    const int64_t n = R * C4;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / C4, cg = i - r * C4;
        uint32_t w = 0;
        if (r < rows) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int64_t c = 4 * cg + k;
                if (c < cols) w |= static_cast<uint32_t>(in[r * cols + c]) << (8 * k);
            }
        }
        const int64_t tile = (r / 128) * C4 + cg;
        out[tile * 128 + (r % 32) * 4 + (r % 128) / 32] = w;
    }
}

}  // namespace

int sm_count() {
    static thread_local int dev = -1, count = 0;
    int cur = 0;
    cudaGetDevice(&cur);
    if (cur != dev) {
        cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, cur);
        if (count <= 0) count = 1;
        dev = cur;
    }
    return count;
}

int launch_amax(const void* x, int64_t M, int64_t K, int dtype, const float* residual, int mode,
                float* out, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool ef = residual != nullptr;
    if (mode == NVFP4_GAMAX_TENSOR) {
        launch_pdl(k_amax_zero, 1, 1, 0, s, out);
        const int64_t nvec = M * (K / 8);
        if (nvec > 0) {
            const int g = grid_for((nvec + kAmaxUnroll - 1) / kAmaxUnroll);
            if (dtype == NVFP4_BF16) {
                if (ef) launch_pdl(k_amax_tensor<NVFP4_BF16, true>, g, kThreads, 0, s, x, residual, nvec, out);
                else launch_pdl(k_amax_tensor<NVFP4_BF16, false>, g, kThreads, 0, s, x, residual, nvec, out);
            } else {
                if (ef) launch_pdl(k_amax_tensor<NVFP4_F32, true>, g, kThreads, 0, s, x, residual, nvec, out);
                else launch_pdl(k_amax_tensor<NVFP4_F32, false>, g, kThreads, 0, s, x, residual, nvec, out);
            }
        }
    } else {
        if (M > 0) {
            const int g = static_cast<int>((M + kThreads / 32 - 1) / (kThreads / 32));
            if (dtype == NVFP4_BF16) {
                if (ef) launch_pdl(k_amax_rows<NVFP4_BF16, true>, g, kThreads, 0, s, x, residual, M, K, out);
                else launch_pdl(k_amax_rows<NVFP4_BF16, false>, g, kThreads, 0, s, x, residual, M, K, out);
            } else {
                if (ef) launch_pdl(k_amax_rows<NVFP4_F32, true>, g, kThreads, 0, s, x, residual, M, K, out);
                else launch_pdl(k_amax_rows<NVFP4_F32, false>, g, kThreads, 0, s, x, residual, M, K, out);
            }
        }
    }
    return static_cast<int>(cudaGetLastError());
}

int launch_scales_mma(const uint8_t* in, int64_t rows, int64_t cols, uint8_t* out, void* stream) {
    const int64_t R = (rows + 127) / 128 * 128, C4 = (cols + 3) / 4;
    const int64_t n = R * C4;
    if (n <= 0) return 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    launch_pdl(k_scales_mma, grid_for(n), kThreads, 0, s, in, rows, cols, R, C4, reinterpret_cast<uint32_t*>(out));
    return static_cast<int>(cudaGetLastError());
}

int launch_probe_sub_f16(const uint32_t* q, const float* v, float* out, int64_t n, void* stream) {
    if (n <= 0) return 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    launch_pdl(k_probe_sub_f16, grid_for(n), kThreads, 0, s, q, v, out, n);
    return static_cast<int>(cudaGetLastError());
}

int launch_probe_divide(const float* a, const float* b, float* out, int64_t n, void* stream) {
    if (n <= 0) return 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    launch_pdl(k_probe_divide, grid_for((n + 15) / 16), kThreads, 0, s, a, b, out, n);
    return static_cast<int>(cudaGetLastError());
}

int launch_probe_e2m1(uint32_t first, int64_t n, uint8_t* out, void* stream) {
    if (n <= 0) return 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    launch_pdl(k_probe_e2m1, grid_for((n + 7) / 8), kThreads, 0, s, first, n, out);
    return static_cast<int>(cudaGetLastError());
}

int launch_global_scales(const float* gamax, int64_t n, float bound, float* s_enc, float* s_dec, void* stream) {
    if (n <= 0) return 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    launch_pdl(k_global_scales, grid_for(n), kThreads, 0, s, gamax, n, bound, s_enc, s_dec);
    return static_cast<int>(cudaGetLastError());
}

int launch_dequantize(const DequantArgs& a, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t nblk = a.M * (a.K / 16);
    if (nblk == 0) return 0;
    const int g = grid_for((nblk + 3) / 4);   // 4 blocks per thread
    if (a.out_dtype == NVFP4_BF16) launch_pdl(k_dequant<NVFP4_BF16>, g, kThreads, 0, s, a);
    else launch_pdl(k_dequant<NVFP4_F32>, g, kThreads, 0, s, a);
    return static_cast<int>(cudaGetLastError());
}

}  // namespace nvfp4
