// gemm.cu -- block-scaled NVFP4 GEMM on the sm_103a tensor cores (tcgen05).
//
//   D[M, N] = s_dec(A) * s_dec(B) * sum_k e2m1(A[m,k]) SA[m,k/16] * e2m1(B[n,k]) SB[n,k/16]
//
// The Fprop, Dgrad and Wgrad GEMMs of the NVFP4 linear layer (news page "NVIDIA
// NVFP4 paper: 4-bit pretrain hits FP8 parity (12B, 10T tokens)", ¶1 and ¶3:
// the recipe targets Blackwell tensor cores).  Both operands are K-major packed
// E2M1 (two per byte) with one E4M3 scale per 16 elements.
//
// Design (one CTA per SM, persistent over 128 x 256 output tiles):
//   warp 0      TMA producer: codes tiles via cp.async.bulk.tensor (128-byte
//               swizzle), scale tiles via 1-D cp.async.bulk, into a 4-stage
//               shared-memory ring guarded by full/empty mbarriers;
//   warp 1      allocates TMEM (512 columns) and, from one lane, issues
//               tcgen05.cp (scales -> TMEM) and tcgen05.mma
//               .kind::mxf4nvf4.block_scale.scale_vec::4X (M=128, N=256, K=64),
//               accumulating in fp32 in TMEM columns [0, 256);
//   warps 2-5   epilogue: tcgen05.ld of their 32-lane quarter, multiply by
//               alpha = s_dec(A) * s_dec(B), convert, store to global.
// Every wait is bounded (see mbar_wait_bounded): on a timeout the kernel
// records NVFP4_ERR_TIMEOUT, lets every role leave its loop, waits for its own
// copies and MMAs in flight, frees TMEM and returns.
//
// Shared memory per stage: A 128x128 B | B 256x128 B | SFA 2 KB | SFB 4 KB = 54 KB.
// TMEM: accumulator cols [0,256); scale slots at 256 + 48*stage:
//   SFA k-step j  -> 4 columns at +4j       (lane r%32, column r/32 = row r)
//   SFB k-step j  -> 8 columns at +16 + 8j  (two 128-row halves of the N tile)
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "device_common.cuh"
#include "host_common.h"

namespace nvfp4 {
namespace gemm {

constexpr int BM = 128, BN = 256, BK = 256;       // BK in E2M1 elements
constexpr int BKB = BK / 2;                       // 128 bytes per row per stage
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BKB;                 // 16 KB
constexpr int B_BYTES = BN * BKB;                 // 32 KB
constexpr int SFA_BYTES = 2048;                   // 128 rows x 16 scales
constexpr int SFB_BYTES = 4096;                   // 256 rows x 16 scales
constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
constexpr int TMEM_COLS = 512;
constexpr int ACC_COL = 0;
constexpr int SF_COL0 = 256;
constexpr int SF_STAGE_COLS = 48;
constexpr int NUM_THREADS = 192;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
static_assert(STAGE_BYTES % 1024 == 0, "stage tiles must stay 1024-byte aligned for the 128B swizzle");
static_assert(SF_COL0 + STAGES * SF_STAGE_COLS <= TMEM_COLS, "TMEM budget");

// Instruction descriptor, kind::mxf4nvf4: A and B E2M1 (format 1), both K-major,
// N>>3 at bit 17, scale format UE4M3 (bit 23 = 0), M>>4 at bit 24.
constexpr uint32_t IDESC = (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

struct Params {
    const uint8_t* sfa;
    const uint8_t* sfb;
    const float* sdec_a;
    const float* sdec_b;
    void* D;
    int64_t ldd;
    int M, N, K;
    int d_bf16;
    int vec_store;
    int nkt;                     // ceil(K / 256): k tiles, also the scale layout's tiles per row block
    int m_tiles, n_tiles;
    uint32_t* dev_status;
    uint64_t timeout_ns;
};

// ---- PTX wrappers ---------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar) : "memory");
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t desc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" :: "r"(taddr), "l"(desc) : "memory");
}

__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                       uint32_t sfb, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}"
        :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb) : "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(bar) : "memory");
}

__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
          "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Descriptor of a 32-row x 16-byte scale block (no swizzle, 8-row groups 128 B apart).
__device__ __forceinline__ uint64_t desc_sf(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(128 >> 4) << 32) | ((uint64_t)1 << 46);
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
gemm_nvfp4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* acc_full = empty + STAGES;
    uint64_t* acc_empty = acc_full + 1;
    uint64_t* drain = acc_empty + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 4);
        mbar_init(drain, 1);
        *abort_flag = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_addr(tmem_slot)), "r"(TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int tiles = p.m_tiles * p.n_tiles;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer
        uint32_t stage = 0, phase = 0;
        uint32_t issued_mask = 0, issued_phase = 0;      // per stage: ever issued / parity of last issue
        bool ok = true;
        for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
            const int mt = tile % p.m_tiles, nt = tile / p.m_tiles;
            const bool second_sfb = (nt * BN + 128) < p.N;
            const uint32_t bytes = STAGE_BYTES - (second_sfb ? 0 : 2048);
            for (int kt = 0; kt < p.nkt; ++kt) {
                if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, p.timeout_ns, abort_flag, p.dev_status)) {
                    ok = false;
                    break;
                }
                uint8_t* sA = smem + stage * STAGE_BYTES;
                uint8_t* sB = sA + A_BYTES;
                uint8_t* sSFA = sB + B_BYTES;
                uint8_t* sSFB = sSFA + SFA_BYTES;
                const uint32_t bar = smem_addr(&full[stage]);
                mbar_arrive_expect_tx(&full[stage], bytes);
                tma_load_2d(smem_addr(sA), &tmA, kt * BKB, mt * BM, bar);
                tma_load_2d(smem_addr(sB), &tmB, kt * BKB, nt * BN, bar);
                bulk_load(smem_addr(sSFA), p.sfa + ((size_t)mt * p.nkt + kt) * 2048u, 2048u, bar);
                bulk_load(smem_addr(sSFB), p.sfb + ((size_t)(2 * nt) * p.nkt + kt) * 2048u, 2048u, bar);
                if (second_sfb)
                    bulk_load(smem_addr(sSFB + 2048), p.sfb + ((size_t)(2 * nt + 1) * p.nkt + kt) * 2048u, 2048u, bar);
                issued_mask |= 1u << stage;
                issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
        if (!ok) {   // let every copy this thread started land before the CTA exits
            for (int s = 0; s < STAGES; ++s)
                if (issued_mask & (1u << s))
                    mbar_wait_bounded(&full[s], (issued_phase >> s) & 1u, p.timeout_ns, nullptr, p.dev_status);
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------ MMA issuer
        uint32_t stage = 0, phase = 0, acc_phase = 0;
        bool ok = true, issued = false;
        for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
            if (!mbar_wait_bounded(acc_empty, acc_phase ^ 1u, p.timeout_ns, abort_flag, p.dev_status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            for (int kt = 0; kt < p.nkt; ++kt) {
                if (!mbar_wait_bounded(&full[stage], phase, p.timeout_ns, abort_flag, p.dev_status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sA = smem_addr(smem + stage * STAGE_BYTES);
                const uint32_t sB = sA + A_BYTES;
                const uint32_t sSFA = sB + B_BYTES;
                const uint32_t sSFB = sSFA + SFA_BYTES;
                const uint32_t tsf = tmem + SF_COL0 + stage * SF_STAGE_COLS;
#pragma unroll
                for (int j = 0; j < 4; ++j) tc_cp_sf(tsf + 4 * j, desc_sf(sSFA + 512 * j));
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    tc_cp_sf(tsf + 16 + 8 * j, desc_sf(sSFB + 512 * j));
                    tc_cp_sf(tsf + 16 + 8 * j + 4, desc_sf(sSFB + 2048 + 512 * j));
                }
                const uint64_t da = desc_sw128(sA), db = desc_sw128(sB);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    tc_mma(tmem + ACC_COL, da + 2 * j, db + 2 * j, IDESC, tsf + 4 * j, tsf + 16 + 8 * j,
                           (kt | j) != 0 ? 1u : 0u);
                issued = true;
                tc_commit(smem_addr(&empty[stage]));
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
            if (!ok) break;
            tc_commit(smem_addr(acc_full));
            acc_phase ^= 1u;
        }
        if (!ok && issued) {   // wait for this thread's MMAs and copies before TMEM is freed
            tc_commit(smem_addr(drain));
            mbar_wait_bounded(drain, 0u, p.timeout_ns, nullptr, p.dev_status);
        }
    } else if (warp >= 2) {
        // ------------------------------------------------ epilogue
        const int q = warp & 3;                          // TMEM lane quarter of this warp
        const float alpha = __fmul_rn(*p.sdec_a, *p.sdec_b);
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
            const int mt = tile % p.m_tiles, nt = tile / p.m_tiles;
            if (!mbar_wait_bounded(acc_full, acc_phase, p.timeout_ns, abort_flag, p.dev_status)) break;
            tc_fence_after();
            const int row = mt * BM + q * 32 + lane;
            const int n0 = nt * BN;
            for (int c = 0; c < BN / 32; ++c) {
                const int nb = n0 + c * 32;
                if (nb >= p.N) break;                    // warp-uniform
                uint32_t v[32];
                tmem_ld_32cols(tmem + ((uint32_t)(q * 32) << 16) + ACC_COL + c * 32, v);
                if (row >= p.M) continue;
                const bool full_chunk = (nb + 32 <= p.N) && p.vec_store;
                if (p.d_bf16) {
                    __nv_bfloat16* drow = reinterpret_cast<__nv_bfloat16*>(p.D) + (int64_t)row * p.ldd + nb;
                    if (full_chunk) {
                        uint32_t w[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            __nv_bfloat162 h = __floats2bfloat162_rn(__fmul_rn(__uint_as_float(v[2 * i]), alpha),
                                                                     __fmul_rn(__uint_as_float(v[2 * i + 1]), alpha));
                            w[i] = *reinterpret_cast<uint32_t*>(&h);
                        }
                        uint4* d4 = reinterpret_cast<uint4*>(drow);
#pragma unroll
                        for (int i = 0; i < 4; ++i) d4[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (nb + i < p.N) drow[i] = __float2bfloat16_rn(__fmul_rn(__uint_as_float(v[i]), alpha));
                    }
                } else {
                    float* drow = reinterpret_cast<float*>(p.D) + (int64_t)row * p.ldd + nb;
                    if (full_chunk) {
                        float4* d4 = reinterpret_cast<float4*>(drow);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            d4[i] = make_float4(__fmul_rn(__uint_as_float(v[4 * i]), alpha),
                                                __fmul_rn(__uint_as_float(v[4 * i + 1]), alpha),
                                                __fmul_rn(__uint_as_float(v[4 * i + 2]), alpha),
                                                __fmul_rn(__uint_as_float(v[4 * i + 3]), alpha));
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (nb + i < p.N) drow[i] = __fmul_rn(__uint_as_float(v[i]), alpha);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);
            acc_phase ^= 1u;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(TMEM_COLS) : "memory");
    }
}

// ---- host ------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void* f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// Packed E2M1 codes [rows, cols/2 bytes], boxes of 128 bytes x box_rows, 128-byte swizzle.
bool make_codes_map(CUtensorMap* m, const void* codes, int64_t rows, int64_t cols, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)(cols / 2), (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(cols / 2)};
    cuuint32_t box[2] = {(cuuint32_t)BKB, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(codes), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace gemm

nvfp4_status gemm_impl(const nvfp4_qtensor* A, const nvfp4_qtensor* B, void* D, int32_t d_dtype, int64_t ldd,
                       uint32_t* dev_status, cudaStream_t stream) {
    using namespace gemm;
    if (!A || !B || !D) return NVFP4_ERR_INVALID_ARG;
    if (d_dtype != NVFP4_F32 && d_dtype != NVFP4_BF16) return NVFP4_ERR_INVALID_ARG;
    if (!A->codes || !B->codes || !A->scales_mma || !B->scales_mma || !A->s_dec || !B->s_dec)
        return NVFP4_ERR_INVALID_ARG;
    const int64_t M = A->rows, N = B->rows, K = A->cols;
    if (B->cols != K) return NVFP4_ERR_SHAPE;
    if (M < 1 || N < 1 || K < 32 || K % 32 != 0 || ldd < N) return NVFP4_ERR_SHAPE;
    if (M > (1ll << 30) || N > (1ll << 30) || K > (1ll << 30)) return NVFP4_ERR_SHAPE;
    if (!aligned16(A->codes) || !aligned16(B->codes) || !aligned16(A->scales_mma) || !aligned16(B->scales_mma))
        return NVFP4_ERR_ALIGNMENT;
    const size_t esz = d_dtype == NVFP4_BF16 ? 2 : 4;
    if ((reinterpret_cast<uintptr_t>(D) % esz) != 0) return NVFP4_ERR_ALIGNMENT;

    CUtensorMap ta, tb;
    if (!make_codes_map(&ta, A->codes, M, K, BM) || !make_codes_map(&tb, B->codes, N, K, BN)) return NVFP4_ERR_CUDA;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return NVFP4_ERR_CUDA;
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(gemm_nvfp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    });
    if (attr_err != cudaSuccess) return NVFP4_ERR_CUDA;

    Params p;
    p.sfa = A->scales_mma;
    p.sfb = B->scales_mma;
    p.sdec_a = A->s_dec;
    p.sdec_b = B->s_dec;
    p.D = D;
    p.ldd = ldd;
    p.M = (int)M;
    p.N = (int)N;
    p.K = (int)K;
    p.d_bf16 = d_dtype == NVFP4_BF16;
    p.vec_store = aligned16(D) && ((ldd * (int64_t)esz) % 16 == 0);
    p.nkt = (int)((K + BK - 1) / BK);
    p.m_tiles = (int)((M + BM - 1) / BM);
    p.n_tiles = (int)((N + BN - 1) / BN);
    p.dev_status = dev_status;
    p.timeout_ns = wait_timeout_ns();
    const int tiles = p.m_tiles * p.n_tiles;
    const int grid = std::max(1, std::min(tiles, sm_count(dev)));
    gemm_nvfp4_kernel<<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(ta, tb, p);
    if (cudaGetLastError() != cudaSuccess) return NVFP4_ERR_CUDA;
    return NVFP4_OK;
}

}  // namespace nvfp4

extern "C" nvfp4_status nvfp4_gemm(const nvfp4_qtensor* A, const nvfp4_qtensor* B, void* D, int32_t d_dtype,
                                   int64_t ldd, uint32_t* dev_status, void* stream) {
    return nvfp4::gemm_impl(A, B, D, d_dtype, ldd, dev_status, static_cast<cudaStream_t>(stream));
}
