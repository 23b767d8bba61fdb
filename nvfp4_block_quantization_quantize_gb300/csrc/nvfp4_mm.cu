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
constexpr uint32_t kColSfa = 128;                         // first scale column
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

// Pipeline: a stage holds kStageK K-steps of both operands and their scale
// tiles; kStages stages rotate, the loads for stage t + kAhead are issued while
// stage t is multiplied, into the slot stage t + kAhead - kStages last used,
// whose MMAs were committed kStages - kAhead stages earlier.
constexpr int kStageK = 2;                                // MMA K-steps (64 elements each) per stage
constexpr int kStages = 6, kAhead = 4;
constexpr int kSlotA = kStageK * kOpBytes;               // 8 KB
constexpr int kSlotSf = kStageK * 512;                   // 1 KB
constexpr int kSlotBytes = 2 * kSlotA + 2 * kSlotSf;     // 18 KB
constexpr int kMmSmem = kStages * kSlotBytes;             // 108 KB
constexpr uint32_t kSfColsPerStage = 2 * 4 * kStageK;    // SFA and SFB, 4 columns per K-step each

template <int ODT>
__global__ void __launch_bounds__(kMmThreads) k_mm(const uint8_t* __restrict__ A, const uint8_t* __restrict__ SA,
                                                   const uint8_t* __restrict__ B, const uint8_t* __restrict__ SB,
                                                   int64_t M, int64_t N, int64_t K, const float* gamax_a,
                                                   const float* gamax_b, float bound, void* out) {
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ __align__(8) uint64_t done[kStages];       // MMAs of the stage in the slot have completed
    __shared__ uint32_t tmem_base;
    __shared__ int timed_out;

    const int tid = threadIdx.x, warp = tid >> 5;
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * kTileM, n0 = static_cast<int64_t>(blockIdx.x) * kTileN;
    const int64_t row_bytes = K / 2;
    const int64_t ksteps = K / kStepK;                    // 64-element steps
    const int64_t nstages = (ksteps + kStageK - 1) / kStageK;
    const int64_t sf_tiles_k = ksteps;                    // 128 x 4 scale tiles along K

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(&tmem_base)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) mbar_init(&done[i]);
        timed_out = 0;
        asm volatile("fence.mbarrier_init.release.cluster;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;");
    const uint32_t tmem = tmem_base;
    const uint32_t idesc = instr_desc(kTileM, kTileN);
    const float alpha = __fmul_rn(decode_scale(gamax_a, bound), decode_scale(gamax_b, bound));

    // copies of stage t into slot t % kStages: row r's 32 bytes of K-step kk are
    // core matrices (r/8, 0), (r/8, 1) of that K-step's 4 KB block; consecutive
    // threads read one row's contiguous bytes
    auto issue = [&](int64_t t) {
        if (t < nstages) {
            uint8_t* slot = smem + (t % kStages) * kSlotBytes;
            const int64_t k0 = t * kStageK;
            const int nk = static_cast<int>(ksteps - k0 < kStageK ? ksteps - k0 : kStageK);
            constexpr int kRowChunks = 2 * kStageK;        // 16-byte chunks of one row per stage
            for (int c = tid; c < 2 * kTileM * kRowChunks; c += kMmThreads) {
                const int op = c / (kTileM * kRowChunks), rc = c % (kTileM * kRowChunks);
                const int r = rc / kRowChunks, q = rc % kRowChunks, kk = q >> 1, j = q & 1;
                if (kk < nk) {
                    const uint8_t* src =
                        (op == 0 ? A + (m0 + r) * row_bytes : B + (n0 + r) * row_bytes) + (k0 + kk) * 32 + 16 * j;
                    uint8_t* dst = slot + op * kSlotA + kk * kOpBytes + ((r >> 3) * 2 + j) * 128 + (r & 7) * 16;
                    cp16(dst, src);
                }
            }
            for (int c = tid; c < 2 * kStageK * 32; c += kMmThreads) {
                const int op = c / (kStageK * 32), rc = c % (kStageK * 32), kk = rc >> 5, q = rc & 31;
                if (kk < nk) {
                    const uint8_t* src = (op == 0 ? SA + ((m0 / 128) * sf_tiles_k + k0 + kk) * 512
                                                  : SB + ((n0 / 128) * sf_tiles_k + k0 + kk) * 512) + 16 * q;
                    cp16(slot + 2 * kSlotA + op * kSlotSf + kk * 512 + 16 * q, src);
                }
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };

    int64_t committed = -1;                               // last stage whose MMAs were committed
    for (int64_t t = 0; t < kAhead; ++t) issue(t);
    for (int64_t t = 0; t < nstages; ++t) {
        // the slot of stage t + kAhead last held stage t + kAhead - kStages
        const int64_t prev = t + kAhead - kStages;
        if (prev >= 0 && !timed_out &&
            !mbar_wait(&done[prev % kStages], static_cast<uint32_t>((prev / kStages) & 1)))
            timed_out = 1;
        issue(t + kAhead);
        asm volatile("cp.async.wait_group %0;" ::"n"(kAhead) : "memory");   // stage t's own copies landed
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (timed_out) break;
        if (tid == 0) {
            asm volatile("tcgen05.fence::after_thread_sync;");
            const uint8_t* slot = smem + (t % kStages) * kSlotBytes;
            const uint32_t sfcol = kColSfa + static_cast<uint32_t>(t % kStages) * kSfColsPerStage;
            const int64_t k0 = t * kStageK;
            const int nk = static_cast<int>(ksteps - k0 < kStageK ? ksteps - k0 : kStageK);
            for (int kk = 0; kk < nk; ++kk) {
                const uint32_t ca = sfcol + 8 * kk, cb = ca + 4;
                const uint64_t dsa = smem_desc(smem_addr(slot + 2 * kSlotA + kk * 512), 0, 128);
                const uint64_t dsb = smem_desc(smem_addr(slot + 2 * kSlotA + kSlotSf + kk * 512), 0, 128);
                asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(tmem + ca), "l"(dsa));
                asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(tmem + cb), "l"(dsb));
                const uint64_t da = smem_desc(smem_addr(slot + kk * kOpBytes), 128, 256);
                const uint64_t db = smem_desc(smem_addr(slot + kSlotA + kk * kOpBytes), 128, 256);
                const uint32_t acc = (k0 + kk) > 0 ? 1u : 0u;
                asm volatile(
                    "{\n\t.reg .pred p;\n\t"
                    "setp.ne.b32 p, %6, 0;\n\t"
                    "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(tmem),
                    "l"(da), "l"(db), "r"(idesc), "r"(tmem + ca), "r"(tmem + cb), "r"(acc));
            }
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                smem_addr(&done[t % kStages])));
        }
        committed = t;
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    // every MMA has completed once the last commit has arrived (a commit tracks
    // all earlier tensor-core work of the issuing thread)
    if (committed >= 0 &&
        !mbar_wait(&done[committed % kStages], static_cast<uint32_t>((committed / kStages) & 1)))
        timed_out = 1;
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;");

    // epilogue: warp w reads accumulator lanes 32w .. 32w+31 (rows m0 + 32w + lane)
    const int64_t row = m0 + 32 * warp + (tid & 31);
    const bool bad = timed_out != 0;
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
        for (int i = 0; i < 16; ++i) f[i] = bad ? __int_as_float(0x7FC00000) : __fmul_rn(__uint_as_float(v[i]), alpha);
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
    static bool configured = false;
    if (!configured) {
        cudaFuncSetAttribute(k_mm<NVFP4_F32>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMmSmem);
        cudaFuncSetAttribute(k_mm<NVFP4_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMmSmem);
        configured = true;
    }
    if (out_dtype == NVFP4_F32)
        k_mm<NVFP4_F32><<<grid, kMmThreads, kMmSmem, s>>>(A, SA, B, SB, M, N, K, gamax_a, gamax_b, bound, out);
    else
        k_mm<NVFP4_BF16><<<grid, kMmThreads, kMmSmem, s>>>(A, SA, B, SB, M, N, K, gamax_a, gamax_b, bound, out);
    return static_cast<int>(cudaGetLastError());
}

}  // namespace nvfp4
