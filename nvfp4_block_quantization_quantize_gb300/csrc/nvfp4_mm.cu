// nvfp4_mm.cu -- C = A B^T on NVFP4 operands with the sm_103a block-scaled
// tensor cores (tcgen05.mma .kind::mxf4nvf4, 16-element blocks, E4M3 scales).
//
// "fp4-train" (API: fp4_mm, "a @ b^T on the Blackwell NVFP4 tensor cores";
// Correctness: the tensor-core path agrees with the dequantize path).  A and B
// are the quantizer's rowwise outputs: codes [M, K/2] and [N, K/2] (two e2m1
// codes per byte, element 2j in the low nibble) and their scale bytes re-laid
// out by nvfp4_scales_to_mma (128 x 4 tiles).  Each 512-byte scale tile goes
// to tensor memory with tcgen05.cp 32x128b.warpx4: every lane quadrant gets
// the 128 x 4 tile, and a lane finds its row's four scales in the column of
// its quadrant.  Products accumulate in fp32 in tensor memory.  Every wait on
// an mbarrier is bounded; a CTA whose wait runs out writes NaN to its tile.
// The epilogue reads the accumulator with tcgen05.ld and multiplies by both
// per-tensor decode scales.
#include <cstdint>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "nvfp4_params.h"

namespace nvfp4 {
namespace {

constexpr int kMmThreads = 128;
constexpr int kTileM = 128, kStepK = 64;                 // K elements per MMA
constexpr uint32_t kColSfa = 128;                         // first scale column (after the accumulator)
constexpr long kWaitLimit = 1L << 22;                     // try_wait rounds before giving up

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// shared-memory matrix descriptor, K-major: lbo = byte step between core
// matrices along K, sbo = between 8-row groups along M/N; layout 0 = no
// swizzle (core matrices of 8 rows x 16 bytes), 2 = 128-byte swizzle (rows
// of 128 bytes, 8-row atoms of 1 KB, 1 KB-aligned)
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout = 0) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;                                      // descriptor version for sm_100 family
    d |= static_cast<uint64_t>(layout & 7u) << 61;        // base offset 0
    return d;
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


// decode scale S_dec = 1 / min(6 * bound / A, FLT_MAX) of a per-tensor amax
// (1 without one, and when A is not a positive finite number)
__device__ __forceinline__ float decode_scale(const float* gamax, float bound) {
    if (!gamax) return 1.0f;
    const float A = *gamax;
    const float enc = (!(A > 0.0f) || isinf(A)) ? 1.0f : fminf(__fdiv_rn(__fmul_rn(6.0f, bound), A), 3.4028234663852886e+38f);
    return __fdiv_rn(1.0f, enc);
}

// Pipeline (warp-specialised).  A CTA owns a 128 x 128 tile of C, one fp32
// accumulator of 128 tensor-memory columns.  Thread 0 (the producer) loads a
// stage -- kStageK K-steps (128 bytes of every row) of A and B (128 rows
// each), one TMA box each with the 128-byte swizzle, which is the layout the
// MMA descriptor's 128-byte-swizzle mode reads (a K-step starts 32 bytes
// further into the 1 KB atoms), and the matching 512-byte scale tiles by bulk
// copies -- into one of kStages slots, signalling the slot's `full` barrier by
// transaction count.  Thread 32 (the MMA issuer) waits for `full`, copies the
// scale tiles to tensor memory and issues one N = 128 MMA per K-step, then
// commits to the slot's `empty` barrier, which the producer waits on before
// refilling the slot.  A last commit signals `acc`; all four warps then read
// the accumulator.  Two CTAs fit on an SM (108 KB of shared memory and 256
// tensor-memory columns each), so one CTA's epilogue and start-up overlap the
// other's MMAs; with one CTA of 128 x 256 tiles per SM (N = 256 MMAs, 512
// columns) the product ran 6 % slower.  TMA fills rows past M or N with zeros.
constexpr int kTileN = 128;
constexpr int kStageK = 4;                                // MMA K-steps (64 elements = 32 bytes each) per stage
constexpr int kStages = 3;
constexpr int kSlotA = kTileM * 128;                      // 128 rows x 128 bytes (128-byte swizzle): 16 KB
constexpr int kSlotB = kTileN * 128;                      // 16 KB
constexpr int kSlotSfa = kStageK * 512, kSlotSfb = kStageK * 512;
constexpr int kSlotBytes = kSlotA + kSlotB + kSlotSfa + kSlotSfb;   // 36 KB
constexpr int kMmSmem = kStages * kSlotBytes + 1024;                 // + alignment slack
constexpr uint32_t kSfColsPerStep = 8;                    // SFA, SFB: 4 columns each
constexpr uint32_t kTmemCols = 256;

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void mma_f4(uint32_t d, uint64_t da, uint64_t db, uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                       uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
        "l"(da), "l"(db), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc));
}

template <int ODT>
__global__ void __launch_bounds__(kMmThreads, 2)
    k_mm(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
         const uint8_t* __restrict__ SA, const uint8_t* __restrict__ SB, int64_t M, int64_t N, int64_t K,
         const float* gamax_a, const float* gamax_b, float bound, void* out) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t full[kStages], empty[kStages], accb;
    __shared__ uint32_t tmem_base;
    __shared__ int timed_out;

    const int tid = threadIdx.x, warp = tid >> 5;
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * kTileM, n0 = static_cast<int64_t>(blockIdx.x) * kTileN;
    const int64_t ksteps = K / kStepK;
    const int64_t nstages = (ksteps + kStageK - 1) / kStageK;

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(&tmem_base)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i]);
            mbar_init(&empty[i]);
        }
        mbar_init(&accb);
        timed_out = 0;
        asm volatile("fence.mbarrier_init.release.cluster;");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mapA)));
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mapB)));
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;");
    const uint32_t tmem = tmem_base;
    const uint32_t idesc = instr_desc(kTileM, kTileN);

    if (tid == 0) {
        // ---- producer ----
        for (int64_t t = 0; t < nstages; ++t) {
            const int s = static_cast<int>(t % kStages);
            if (t >= kStages && !mbar_wait(&empty[s], static_cast<uint32_t>(((t / kStages) - 1) & 1))) {
                timed_out = 1;
                break;
            }
            const int64_t k0 = t * kStageK;
            const int nk = static_cast<int>(ksteps - k0 < kStageK ? ksteps - k0 : kStageK);
            uint8_t* slot = smem + s * kSlotBytes;
            mbar_expect_tx(&full[s], static_cast<uint32_t>(kSlotA + kSlotB + nk * 1024));
            tma_2d(slot, &mapA, static_cast<int>(k0 * 32), static_cast<int>(m0), &full[s]);
            tma_2d(slot + kSlotA, &mapB, static_cast<int>(k0 * 32), static_cast<int>(n0), &full[s]);
            bulk_copy(slot + kSlotA + kSlotB, SA + ((m0 / 128) * ksteps + k0) * 512, nk * 512, &full[s]);
            bulk_copy(slot + kSlotA + kSlotB + kSlotSfa, SB + ((n0 / 128) * ksteps + k0) * 512, nk * 512, &full[s]);
        }
    } else if (tid == 32) {
        // ---- MMA issuer ----
        int64_t t = 0;
        for (; t < nstages; ++t) {
            const int s = static_cast<int>(t % kStages);
            if (timed_out || !mbar_wait(&full[s], static_cast<uint32_t>((t / kStages) & 1))) {
                timed_out = 1;
                break;
            }
            asm volatile("tcgen05.fence::after_thread_sync;");
            const uint8_t* slot = smem + s * kSlotBytes;
            const int64_t k0 = t * kStageK;
            const int nk = static_cast<int>(ksteps - k0 < kStageK ? ksteps - k0 : kStageK);
            for (int kk = 0; kk < nk; ++kk) {
                const uint32_t c = kColSfa + static_cast<uint32_t>(s * kStageK + kk) * kSfColsPerStep;
                const uint8_t* sf = slot + kSlotA + kSlotB;
                asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(tmem + c),
                             "l"(smem_desc(smem_addr(sf + kk * 512), 0, 128)));
                asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(tmem + c + 4),
                             "l"(smem_desc(smem_addr(sf + kSlotSfa + kk * 512), 0, 128)));
                const uint64_t da = smem_desc(smem_addr(slot + kk * 32), 16, 1024, 2);
                const uint32_t acc = (k0 + kk) > 0 ? 1u : 0u;
                mma_f4(tmem, da, smem_desc(smem_addr(slot + kSlotA + kk * 32), 16, 1024, 2), idesc, tmem + c,
                       tmem + c + 4, acc);
            }
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                smem_addr(&empty[s])));
        }
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_addr(&accb)));
    }
    // ---- epilogue: every warp reads its 32 accumulator lanes ----
    if (!mbar_wait(&accb, 0)) timed_out = 1;
    __syncwarp();
    asm volatile("tcgen05.fence::after_thread_sync;");
    const float alpha = __fmul_rn(decode_scale(gamax_a, bound), decode_scale(gamax_b, bound));
    const int64_t row = m0 + 32 * warp + (tid & 31);
    const bool bad = timed_out != 0;
    const int ncols = kTileN;
    for (int c0 = 0; c0 < ncols; c0 += 16) {
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

// 2D map of a [rows, K/2]-byte code matrix, boxes of box_rows x 128 bytes, 128-byte swizzle
bool encode_codes_map(CUtensorMap* map, const uint8_t* codes, int64_t rows, int64_t K, int box_rows) {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", reinterpret_cast<void**>(&encode), 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return false;
    }
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
    const cuuint32_t box[2] = {128, static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(codes), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int launch_mm(const uint8_t* A, const uint8_t* SA, const uint8_t* B, const uint8_t* SB, int64_t M, int64_t N,
              int64_t K, const float* gamax_a, const float* gamax_b, float bound, void* out, int out_dtype,
              void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    CUtensorMap mapA, mapB;
    if (!encode_codes_map(&mapA, A, M, K, kTileM) || !encode_codes_map(&mapB, B, N, K, kTileN))
        return static_cast<int>(cudaErrorInvalidValue);
    const dim3 grid(static_cast<unsigned>((N + kTileN - 1) / kTileN), static_cast<unsigned>(M / kTileM));
    static thread_local int configured_dev = -1;         // the attribute is per device
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_dev != dev) {
        cudaFuncSetAttribute(k_mm<NVFP4_F32>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMmSmem);
        cudaFuncSetAttribute(k_mm<NVFP4_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMmSmem);
        configured_dev = dev;
    }
    if (out_dtype == NVFP4_F32)
        k_mm<NVFP4_F32><<<grid, kMmThreads, kMmSmem, s>>>(mapA, mapB, SA, SB, M, N, K, gamax_a, gamax_b, bound, out);
    else
        k_mm<NVFP4_BF16><<<grid, kMmThreads, kMmSmem, s>>>(mapA, mapB, SA, SB, M, N, K, gamax_a, gamax_b, bound, out);
    return static_cast<int>(cudaGetLastError());
}

}  // namespace nvfp4
