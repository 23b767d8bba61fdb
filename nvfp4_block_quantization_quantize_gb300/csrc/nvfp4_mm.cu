// nvfp4_mm.cu -- C = A B^T on NVFP4 operands with the sm_103a block-scaled
// tensor cores (tcgen05.mma .kind::mxf4nvf4, 16-element blocks, E4M3 scales).
//
// "fp4-train" (API: fp4_mm, "a @ b^T on the Blackwell NVFP4 tensor cores";
// Correctness: the tensor-core path agrees with the dequantize path).  A and B
// are the quantizer's rowwise outputs: codes [M, K/2] and [N, K/2] (two e2m1
// codes per byte, element 2j in the low nibble) and their scale bytes re-laid
// out by nvfp4_scales_to_mma (128 x 4 tiles).  One CTA of 128 threads owns a
// 128 x 128 tile of C; for each 64-element step of K it stages the A and B
// slices in shared memory in the no-swizzle K-major core-matrix layout (8 rows
// x 16 bytes per core matrix), copies the step's two 512-byte scale tiles into
// tensor memory (tcgen05.cp 32x128b.warpx4: each lane quadrant gets the 128 x
// 4 tile, a lane finds its row's four scales in the column of its quadrant),
// and one thread issues the MMA, accumulating in fp32 in tensor memory.
// Completion is tracked with an mbarrier whose waits are bounded; a CTA whose
// wait runs out writes NaN to its tile.  The epilogue reads the accumulator
// with tcgen05.ld and multiplies by both per-tensor decode scales.
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "nvfp4_params.h"

namespace nvfp4 {
namespace {

constexpr int kMmThreads = 128;
constexpr int kTileM = 128, kTileN = 128, kStepK = 64;   // K elements per MMA
constexpr int kOpBytes = kTileM * kStepK / 2;            // 4 KB per operand slice
constexpr uint32_t kTmemCols = 256;                       // accumulator 128 + scale columns
constexpr uint32_t kColSfa = 128, kColSfb = 132;
constexpr long kWaitLimit = 1L << 22;                     // try_wait rounds before giving up

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// shared-memory matrix descriptor: no swizzle, K-major core matrices of 8 rows
// x 16 bytes; lbo = byte step between core matrices along K, sbo = along M/N
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;                                      // descriptor version for sm_100 family
    return d;                                             // base offset 0, layout type 0 (no swizzle)
}

// instruction descriptor for .kind::mxf4nvf4: A and B e2m1 (format 1), both
// K-major, E4M3 scales, scale-factor ids 0, N >> 3 and M >> 4
__device__ __forceinline__ uint32_t instr_desc(int M, int N) {
    uint32_t d = 0;
    d |= 1u << 7;                                         // A format: e2m1
    d |= 1u << 10;                                        // B format: e2m1
    d |= static_cast<uint32_t>(N >> 3) << 17;
    d |= static_cast<uint32_t>(M >> 4) << 24;
    return d;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(bar)));
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    for (long it = 0; it < kWaitLimit; ++it) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(smem_addr(bar)), "r"(parity)
            : "memory");
        if (ok) return true;
    }
    return false;
}

__device__ __forceinline__ void cp16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}

// decode scale S_dec = 1 / min(6 * bound / A, FLT_MAX) of a per-tensor amax
// (1 without one, and when A is not a positive finite number)
__device__ __forceinline__ float decode_scale(const float* gamax, float bound) {
    if (!gamax) return 1.0f;
    const float A = *gamax;
    const float enc = (!(A > 0.0f) || isinf(A)) ? 1.0f : fminf(__fdiv_rn(__fmul_rn(6.0f, bound), A), 3.4028234663852886e+38f);
    return __fdiv_rn(1.0f, enc);
}

template <int ODT>
__global__ void __launch_bounds__(kMmThreads) k_mm(const uint8_t* __restrict__ A, const uint8_t* __restrict__ SA,
                                                   const uint8_t* __restrict__ B, const uint8_t* __restrict__ SB,
                                                   int64_t M, int64_t N, int64_t K, const float* gamax_a,
                                                   const float* gamax_b, float bound, void* out) {
    __shared__ __align__(128) uint8_t sA[kOpBytes];
    __shared__ __align__(128) uint8_t sB[kOpBytes];
    __shared__ __align__(128) uint8_t sSA[512];
    __shared__ __align__(128) uint8_t sSB[512];
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t tmem_base;
    __shared__ int timed_out;

    const int tid = threadIdx.x, warp = tid >> 5;
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * kTileM, n0 = static_cast<int64_t>(blockIdx.x) * kTileN;
    const int64_t row_bytes = K / 2;
    const int64_t ksteps = K / kStepK;
    const int64_t sf_tiles_k = K / kStepK;                // 4-column scale tiles along K (K / 16 / 4)

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(&tmem_base)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == 0) {
        mbar_init(&bar);
        timed_out = 0;
        asm volatile("fence.mbarrier_init.release.cluster;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;");
    const uint32_t tmem = tmem_base;
    const uint32_t idesc = instr_desc(kTileM, kTileN);
    const float alpha = __fmul_rn(decode_scale(gamax_a, bound), decode_scale(gamax_b, bound));
    uint32_t last_parity = 0;

    for (int64_t ks = 0; ks < ksteps; ++ks) {
        // stage the A and B slices: row r's 32 bytes are core matrices (r/8, 0) and
        // (r/8, 1), each 8 rows x 16 bytes; core (g, j) sits at (2 g + j) * 128
        for (int c = tid; c < 2 * kTileM * 2; c += kMmThreads) {
            const int op = c / (kTileM * 2), rc = c % (kTileM * 2);
            const int r = rc >> 1, j = rc & 1;
            const uint8_t* src = (op == 0 ? A + (m0 + r) * row_bytes : B + (n0 + r) * row_bytes) + ks * 32 + 16 * j;
            uint8_t* dst = (op == 0 ? sA : sB) + ((r >> 3) * 2 + j) * 128 + (r & 7) * 16;
            cp16(dst, src);
        }
        // the step's 128 x 4 scale tiles (512 contiguous bytes each)
        if (tid < 64) {
            const int op = tid >> 5, q = tid & 31;
            const uint8_t* src = (op == 0 ? SA + ((m0 / 128) * sf_tiles_k + ks) * 512
                                          : SB + ((n0 / 128) * sf_tiles_k + ks) * 512) + 16 * q;
            cp16((op == 0 ? sSA : sSB) + 16 * q, src);
        }
        asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // make the stores visible to the tensor core
        __syncthreads();
        if (tid == 0 && !timed_out) {
            asm volatile("tcgen05.fence::after_thread_sync;");
            const uint64_t dsa = smem_desc(smem_addr(sSA), 0, 128);
            const uint64_t dsb = smem_desc(smem_addr(sSB), 0, 128);
            asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(tmem + kColSfa), "l"(dsa));
            asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(tmem + kColSfb), "l"(dsb));
            const uint64_t da = smem_desc(smem_addr(sA), 128, 256);
            const uint64_t db = smem_desc(smem_addr(sB), 128, 256);
            const uint32_t acc = ks > 0 ? 1u : 0u;
            asm volatile(
                "{\n\t.reg .pred p;\n\t"
                "setp.ne.b32 p, %6, 0;\n\t"
                "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(tmem),
                "l"(da), "l"(db), "r"(idesc), "r"(tmem + kColSfa), "r"(tmem + kColSfb), "r"(acc));
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                smem_addr(&bar)));
        }
        // the MMA has read the staged slices before they are overwritten
        last_parity = static_cast<uint32_t>(ks & 1);
        if (!timed_out && !mbar_wait(&bar, last_parity)) timed_out = 1;
        __syncthreads();
        if (timed_out) break;
    }
    if (timed_out) mbar_wait(&bar, last_parity);        // once more (bounded) before tensor memory is freed
    asm volatile("tcgen05.fence::after_thread_sync;");

    // epilogue: warp w reads accumulator lanes 32w .. 32w+31 (rows m0 + 32w + lane)
    const int64_t row = m0 + 32 * warp + (tid & 31);
    for (int c0 = 0; c0 < kTileN; c0 += 16) {
        uint32_t v[16];
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
            : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
              "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
            : "r"(tmem + (static_cast<uint32_t>(32 * warp) << 16) + static_cast<uint32_t>(c0)));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        float f[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) f[i] = timed_out ? __int_as_float(0x7FC00000) : __fmul_rn(__uint_as_float(v[i]), alpha);
        if (ODT == NVFP4_F32) {
            float4* o = reinterpret_cast<float4*>(static_cast<float*>(out) + row * N + n0 + c0);
#pragma unroll
            for (int i = 0; i < 4; ++i) o[i] = make_float4(f[4 * i], f[4 * i + 1], f[4 * i + 2], f[4 * i + 3]);
        } else {
            uint32_t h[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const __nv_bfloat162 p = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
                h[i] = *reinterpret_cast<const uint32_t*>(&p);
            }
            uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + row * N + n0 + c0);
            o[0] = make_uint4(h[0], h[1], h[2], h[3]);
            o[1] = make_uint4(h[4], h[5], h[6], h[7]);
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

}  // namespace

int launch_mm(const uint8_t* A, const uint8_t* SA, const uint8_t* B, const uint8_t* SB, int64_t M, int64_t N,
              int64_t K, const float* gamax_a, const float* gamax_b, float bound, void* out, int out_dtype,
              void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const dim3 grid(static_cast<unsigned>(N / kTileN), static_cast<unsigned>(M / kTileM));
    if (out_dtype == NVFP4_F32)
        k_mm<NVFP4_F32><<<grid, kMmThreads, 0, s>>>(A, SA, B, SB, M, N, K, gamax_a, gamax_b, bound, out);
    else
        k_mm<NVFP4_BF16><<<grid, kMmThreads, 0, s>>>(A, SA, B, SB, M, N, K, gamax_a, gamax_b, bound, out);
    return static_cast<int>(cudaGetLastError());
}

}  // namespace nvfp4
