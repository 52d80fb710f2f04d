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
//               tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X
//               (M=128, N=256, K=64), accumulating in fp32 in TMEM columns [0, 256);
//   warps 6-9   move each stage's E4M3 scale tiles smem -> registers -> TMEM
//               (tcgen05.st), off the tensor pipe: copying them with tcgen05.cp
//               serialised with the MMAs and cost a third of the run time;
//   warps 2-5   epilogue: tcgen05.ld of their 32-lane quarter, multiply by
//               alpha = s_dec(A) * s_dec(B), convert.  bf16 output: write a
//               128B-swizzled shared-memory tile, release the accumulator, then
//               one lane issues TMA bulk stores (3-stage ring + 64 KB staging);
//               fp32 or unaligned output: direct stores (4-stage ring).
// Every wait is bounded (see mbar_wait_bounded): on a timeout the kernel
// records NVFP4_ERR_TIMEOUT, lets every role leave its loop, waits for its own
// copies and MMAs in flight, frees TMEM and returns.
//
// Shared memory per stage: A 128x128 B | B 256x128 B | SFA 2 KB | SFB 4 KB = 54 KB.
// The single accumulator is released as soon as the epilogue has it in registers /
// shared memory, so the next tile's MMAs overlap the global stores.
// The scale tiles have their own barrier (sf_loaded) so the scale warps start while
// the codes tiles are still in flight.
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
constexpr int A_BYTES = BM * BKB;                 // 16 KB
constexpr int B_BYTES = BN * BKB;                 // 32 KB
constexpr int SFA_BYTES = 2048;                   // 128 rows x 16 scales
constexpr int SFB_BYTES = 4096;                   // 256 rows x 16 scales
constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
constexpr int TMEM_COLS = 512;
constexpr int ACC_COL = 0;
constexpr int SF_COL0 = 256;
constexpr int SF_STAGE_COLS = 48;
constexpr int NUM_THREADS = 320;                 // 10 warps: producer, MMA, 4 epilogue, 4 scale loaders
// bf16 output staged through shared memory for TMA stores: each epilogue warp owns
// 32 rows x 256 columns = four 32 x 64 boxes of 4 KB (128-byte swizzle).
constexpr int BOX_COLS = 64;
constexpr int BOX_BYTES = 32 * BOX_COLS * 2;
constexpr int STAGING_BYTES = 4 * 4 * BOX_BYTES;  // 64 KB
constexpr int BAR_BYTES = 256;
constexpr int SMEM_LIMIT = 232448;                // 227 KB per CTA on sm_103a

template <bool STAGED> struct Cfg {
    static constexpr int STAGES = STAGED ? 3 : 4;
    static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
    static constexpr int STAGING = STAGED ? STAGING_BYTES : 0;
    static constexpr int SLACK = STAGED ? (SMEM_LIMIT - RING_BYTES - STAGING_BYTES - BAR_BYTES) : 1024;
    static constexpr int SMEM_BYTES = RING_BYTES + STAGING + BAR_BYTES + SLACK;
    static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory budget");
    static_assert(SF_COL0 + STAGES * SF_STAGE_COLS <= TMEM_COLS, "TMEM budget");
};
static_assert(STAGE_BYTES % 1024 == 0, "stage tiles must stay 1024-byte aligned for the 128B swizzle");

// Instruction descriptor, kind::mxf4nvf4: A and B E2M1 (format 1), both K-major,
// N>>3 at bit 17, scale format UE4M3 (bit 23 = 0), M>>4 at bit 24.
constexpr uint32_t IDESC = (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
static_assert(IDESC == 0x08400480u, "instruction descriptor");

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
    int n_fastest;               // tile order: 1 = consecutive tiles walk N (A tile reused), 0 = walk M
    uint32_t* dev_status;
    uint64_t timeout_ns;
    uint32_t* maxima;            // EPI_SQAMAX / EPI_DSQR_AMAX: 2 x maxima_parts partial maxima (|X|, then |RHT(X)| / 4)
    int maxima_parts;            // partials per half of `maxima` (>= 4 x grid)
    uint64_t rht_seed;           // the RHT sign vector of the column quantization those maxima serve
    // Split tail (pair kernel, EPI_PLAIN, with a caller workspace): the r tiles of the last,
    // partial wave are cut into `split` parts along K, one part per cluster, so the last wave
    // takes 1 / split of a tile's time.  split = 1: every tile is computed whole.
    int split;
    float* split_ws;             // per tail tile, CTA and epilogue warp: 32 x 128 fp32 sums (left at 0)
    uint32_t* split_cnt;         // per tail tile, CTA and epilogue warp: halves arrived (left at 0)
};

// Epilogue variants of the CTA-pair kernel.
//   EPI_PLAIN   D = alpha * acc;
//   EPI_DSQR    D = dH = bf16(alpha * acc) * 2 relu(H)  (the squared-ReLU backward);
//   EPI_SQAMAX  D = H = alpha * acc, plus the tensor maxima that quantizing A = relu(H)^2 in
//               both orientations needs (|A| and |RHT(A)| along rows), as per-warp partials;
//   EPI_DSQR_AMAX  EPI_DSQR plus the same two maxima of dH itself.
constexpr int EPI_PLAIN = 0, EPI_DSQR = 1, EPI_SQAMAX = 2, EPI_DSQR_AMAX = 3;

// Tile order.  Consecutive persistent CTAs (clusters) take consecutive tiles, so the
// operand indexed by the slow coordinate is shared by the CTAs running together
// and read about once, while the other is swept once per slow step.  The host
// picks the order that re-sweeps the smaller operand (it stays in L2).
__device__ __forceinline__ void tile_coords(const Params& p, int tile, int m_count, int& m, int& n) {
    if (p.n_fastest) { n = tile % p.n_tiles; m = tile / p.n_tiles; }
    else { m = tile % m_count; n = tile / m_count; }
}

// Work item i of cluster c (of P) in the pair kernel: the whole tiles c, c + P, ... of the full
// waves, then at most one item of the last, partial wave -- the whole tile (split = 1) or, with
// split = S, part c % S of tail tile c / S: K tiles [part nkt / S, (part + 1) nkt / S).  The host
// keeps S <= nkt and (tail tiles) x S <= P.  False when cluster c has no item i.
struct PairItem {
    int tile, kb, ke;
    int part;                    // -1: a whole tile
};
__device__ __forceinline__ bool pair_item(const Params& p, int tiles, int c, int P, int i, PairItem& it) {
    const int waves = tiles / P;
    if (i < waves) {
        it.tile = c + i * P; it.kb = 0; it.ke = p.nkt; it.part = -1;
        return true;
    }
    if (i > waves) return false;
    const int r = tiles - waves * P;
    if (p.split <= 1) {
        if (c >= r) return false;
        it.tile = waves * P + c; it.kb = 0; it.ke = p.nkt; it.part = -1;
        return true;
    }
    if (c >= r * p.split) return false;
    it.part = c % p.split;
    it.tile = waves * P + c / p.split;
    it.kb = it.part * p.nkt / p.split;
    it.ke = (it.part + 1) * p.nkt / p.split;
    return true;
}

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

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* tm, uint32_t src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
                 :: "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(src) : "memory");
}
// Streaming data (the output tiles, the epilogue's H tiles) is marked evict-first in L2, so it
// does not push out the operand that consecutive tiles re-read.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void tma_store_2d_hint(const CUtensorMap* tm, uint32_t src, int x, int y, uint64_t pol) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%1, %2}], [%3], %4;"
                 :: "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(src), "l"(pol) : "memory");
}
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* tm, int x, int y, uint32_t bar,
                                                 uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar), "l"(pol) : "memory");
}
// 1-D bulk copy multicast to the CTAs of `mask` (same shared-memory offset and barrier offset in each).
__device__ __forceinline__ void bulk_load_mc(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar, uint16_t mask) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
                 " [%0], [%1], %2, [%3], %4;"
                 :: "r"(dst), "l"(src), "r"(bytes), "r"(bar), "h"(mask) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

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

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Ties 32 registers written by an asynchronous tcgen05.ld to a point after the
// tcgen05.wait::ld that precedes it: the compiler sees them modified here, so no
// use of them can be scheduled before the wait.
__device__ __forceinline__ void reg_fence32(uint32_t (&v)[32]) {
    asm volatile(""
                 : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]), "+r"(v[7]),
                   "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]), "+r"(v[14]),
                   "+r"(v[15]), "+r"(v[16]), "+r"(v[17]), "+r"(v[18]), "+r"(v[19]), "+r"(v[20]), "+r"(v[21]),
                   "+r"(v[22]), "+r"(v[23]), "+r"(v[24]), "+r"(v[25]), "+r"(v[26]), "+r"(v[27]), "+r"(v[28]),
                   "+r"(v[29]), "+r"(v[30]), "+r"(v[31]));
}

__device__ __forceinline__ void tmem_ld_32cols_nowait(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
          "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr) : "memory");
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
    reg_fence32(v);
}

// Each thread writes 16 consecutive 32-bit TMEM columns of its lane.
__device__ __forceinline__ void tmem_st_16cols(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
                 :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
                    "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]) : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Epilogue for one 32-row x 256-column slice (one warp): TMEM -> alpha -> global.
// Direct stores: each lane writes its row (bf16 or fp32), masked at the edges.
__device__ __forceinline__ void epilogue_direct(const Params& p, uint32_t tmem_row, int row, int n0, float alpha) {
    for (int c = 0; c < BN / 32; ++c) {
        const int nb = n0 + c * 32;
        if (nb >= p.N) break;                        // warp-uniform
        uint32_t v[32];
        tmem_ld_32cols(tmem_row + ACC_COL + c * 32, v);
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
}

// Staged bf16 epilogue: TMEM -> alpha -> bf16 -> this warp's four 32 x 64 boxes in
// shared memory, 128-byte swizzled (16-byte chunk c of row r at chunk c ^ (r & 7)),
// the layout the TMA store expects.  Lane = row within the slice.  The TMEM load of
// box b+1 is in flight while box b is converted, and `release` runs as soon as the
// last load has completed (before the last box is converted), so the MMA warp can
// start the next tile early.
template <typename Release>
__device__ __forceinline__ void epilogue_to_smem(uint32_t tmem_row, uint8_t* stg, int lane, float alpha,
                                                 Release&& release) {
    uint32_t va[64], vb[64];
    auto ld64 = [&](uint32_t (&v)[64], int b) {
        uint32_t (&lo)[32] = *reinterpret_cast<uint32_t (*)[32]>(&v[0]);
        uint32_t (&hi)[32] = *reinterpret_cast<uint32_t (*)[32]>(&v[32]);
        tmem_ld_32cols_nowait(tmem_row + ACC_COL + b * BOX_COLS, lo);
        tmem_ld_32cols_nowait(tmem_row + ACC_COL + b * BOX_COLS + 32, hi);
    };
    auto fence64 = [&](uint32_t (&v)[64]) {
        reg_fence32(*reinterpret_cast<uint32_t (*)[32]>(&v[0]));
        reg_fence32(*reinterpret_cast<uint32_t (*)[32]>(&v[32]));
    };
    auto store_box = [&](const uint32_t (&v)[64], int b) {
        uint8_t* row = stg + b * BOX_BYTES + lane * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                __nv_bfloat162 h = __floats2bfloat162_rn(__fmul_rn(__uint_as_float(v[8 * c + 2 * i]), alpha),
                                                         __fmul_rn(__uint_as_float(v[8 * c + 2 * i + 1]), alpha));
                w[i] = *reinterpret_cast<uint32_t*>(&h);
            }
            *reinterpret_cast<uint4*>(row + ((c ^ (lane & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    };
    ld64(va, 0);
    tmem_ld_wait();
    fence64(va);
    ld64(vb, 1);
    store_box(va, 0);
    tmem_ld_wait();
    fence64(vb);
    ld64(va, 2);
    store_box(vb, 1);
    tmem_ld_wait();
    fence64(va);
    ld64(vb, 3);
    store_box(va, 2);
    tmem_ld_wait();
    fence64(vb);
    release();
    store_box(vb, 3);
}

template <bool STAGED>
__global__ void __launch_bounds__(NUM_THREADS, 1)
gemm_nvfp4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmD, const Params p) {
    pdl_launch_dependents();
    pdl_wait();
    using C = Cfg<STAGED>;
    constexpr int STAGES = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* staging = smem + C::RING_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(staging + C::STAGING);
    uint64_t* empty = full + STAGES;
    uint64_t* acc_full = empty + STAGES;
    uint64_t* acc_empty = acc_full + 1;
    uint64_t* drain = acc_empty + 1;
    uint64_t* sf_loaded = drain + 1;                     // scale tiles of a stage have landed in smem
    uint64_t* sf_ready = sf_loaded + STAGES;             // ... and have been written to TMEM
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sf_ready + STAGES);
    volatile uint32_t* abort_flag = tmem_slot + 1;
    // the carve-out above must fit the dynamic allocation (the base is normally 1024-aligned)
    const bool layout_ok = (reinterpret_cast<uintptr_t>(tmem_slot + 2) - reinterpret_cast<uintptr_t>(smem_raw)) <=
                           (uintptr_t)C::SMEM_BYTES;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (!layout_ok) {
        if (threadIdx.x == 0) set_status(p.dev_status, NVFP4_ERR_UNSUPPORTED);
        return;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 4);
        mbar_init(drain, 1);
        for (int s = 0; s < STAGES; ++s) { mbar_init(&sf_loaded[s], 1); mbar_init(&sf_ready[s], 4); }
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
            int mt, nt;
            tile_coords(p, tile, p.m_tiles, mt, nt);
            const bool second_sfb = (nt * BN + 128) < p.N;
            const uint32_t sf_bytes = SFA_BYTES + SFB_BYTES - (second_sfb ? 0 : 2048);
            for (int kt = 0; kt < p.nkt; ++kt) {
                if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, p.timeout_ns, abort_flag, p.dev_status)) {
                    ok = false;
                    break;
                }
                uint8_t* sA = smem + stage * STAGE_BYTES;
                uint8_t* sB = sA + A_BYTES;
                uint8_t* sSFA = sB + B_BYTES;
                uint8_t* sSFB = sSFA + SFA_BYTES;
                const uint32_t sbar = smem_addr(&sf_loaded[stage]);
                mbar_arrive_expect_tx(&sf_loaded[stage], sf_bytes);
                bulk_load(smem_addr(sSFA), p.sfa + ((size_t)mt * p.nkt + kt) * 2048u, 2048u, sbar);
                bulk_load(smem_addr(sSFB), p.sfb + ((size_t)(2 * nt) * p.nkt + kt) * 2048u, 2048u, sbar);
                if (second_sfb)
                    bulk_load(smem_addr(sSFB + 2048), p.sfb + ((size_t)(2 * nt + 1) * p.nkt + kt) * 2048u, 2048u, sbar);
                const uint32_t bar = smem_addr(&full[stage]);
                mbar_arrive_expect_tx(&full[stage], A_BYTES + B_BYTES);
                tma_load_2d(smem_addr(sA), &tmA, kt * BKB, mt * BM, bar);
                tma_load_2d(smem_addr(sB), &tmB, kt * BKB, nt * BN, bar);
                issued_mask |= 1u << stage;
                issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
        if (!ok) {   // let every copy this thread started land before the CTA exits
            for (int s = 0; s < STAGES; ++s)
                if (issued_mask & (1u << s)) {
                    mbar_wait_bounded(&full[s], (issued_phase >> s) & 1u, p.timeout_ns, nullptr, p.dev_status);
                    mbar_wait_bounded(&sf_loaded[s], (issued_phase >> s) & 1u, p.timeout_ns, nullptr, p.dev_status);
                }
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
                if (!mbar_wait_bounded(&full[stage], phase, p.timeout_ns, abort_flag, p.dev_status) ||
                    !mbar_wait_bounded(&sf_ready[stage], phase, p.timeout_ns, abort_flag, p.dev_status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sA = smem_addr(smem + stage * STAGE_BYTES);
                const uint32_t sB = sA + A_BYTES;
                const uint32_t tsf = tmem + SF_COL0 + stage * SF_STAGE_COLS;
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
    } else if (warp >= 6) {
        // ------------------------------------------------ scale loaders: smem -> registers -> TMEM
        // Warp w writes TMEM lanes 32*(w%4)..+31.  Lane i of every warp writes the same
        // 16-byte rows: row i of each 512-byte scale atom holds the scales of tile rows
        // i, i+32, i+64, i+96, so TMEM lane i (of every lane quarter), column c gets
        // row 32c + i -- the operand layout of the block-scaled MMA (M = 128 for A;
        // two 128-row halves side by side for the 256-row B tile).
        const int q = warp & 3;
        const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16);
        uint32_t stage = 0, phase = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
            for (int kt = 0; kt < p.nkt; ++kt) {
                // sf_loaded[s] completes only after the producer refilled the stage, which
                // waited for the MMAs that last read this TMEM slot: the slot is free.
                if (!mbar_wait_bounded(&sf_loaded[stage], phase, p.timeout_ns, abort_flag, p.dev_status)) {
                    ok = false;
                    break;
                }
                const uint8_t* sSFA = smem + stage * STAGE_BYTES + A_BYTES + B_BYTES;
                const uint8_t* sSFB = sSFA + SFA_BYTES;
                uint32_t va[16], vb0[16], vb1[16];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint4 a4 = *reinterpret_cast<const uint4*>(sSFA + 512 * j + 16 * lane);
                    va[4 * j] = a4.x; va[4 * j + 1] = a4.y; va[4 * j + 2] = a4.z; va[4 * j + 3] = a4.w;
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
#pragma unroll
                    for (int nb = 0; nb < 2; ++nb) {
                        const uint4 b4 = *reinterpret_cast<const uint4*>(sSFB + 2048 * nb + 512 * j + 16 * lane);
                        const int o = 8 * j + 4 * nb;          // SFB column of this atom, k-step j
                        uint32_t* dst = o < 16 ? vb0 : vb1;
                        dst[(o & 15)] = b4.x; dst[(o & 15) + 1] = b4.y; dst[(o & 15) + 2] = b4.z; dst[(o & 15) + 3] = b4.w;
                    }
                }
                const uint32_t tsf = tq + SF_COL0 + stage * SF_STAGE_COLS;
                tmem_st_16cols(tsf, va);
                tmem_st_16cols(tsf + 16, vb0);
                tmem_st_16cols(tsf + 32, vb1);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sf_ready[stage]);
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
    } else if (warp >= 2) {
        // ------------------------------------------------ epilogue
        const int q = warp & 3;                          // TMEM lane quarter of this warp
        const float alpha = __fmul_rn(*p.sdec_a, *p.sdec_b);
        const uint32_t tmem_row = tmem + ((uint32_t)(q * 32) << 16);
        uint8_t* stg = staging + q * (4 * BOX_BYTES);
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
            int mt, nt;
            tile_coords(p, tile, p.m_tiles, mt, nt);
            const int m0 = mt * BM + q * 32, n0 = nt * BN;
            if (!mbar_wait_bounded(acc_full, acc_phase, p.timeout_ns, abort_flag, p.dev_status)) break;
            tc_fence_after();
            if constexpr (STAGED) {
                // the previous tile's stores must have finished reading this warp's boxes
                if (lane == 0) bulk_wait_read0();
                __syncwarp();
                epilogue_to_smem(tmem_row, stg, lane, alpha, [&] {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(acc_empty);   // the MMA may start the next tile now
                });
            } else {
                epilogue_direct(p, tmem_row, m0 + lane, n0, alpha);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acc_empty);
            }
            if constexpr (STAGED) {
                fence_proxy_async_smem();                // generic-proxy writes -> visible to TMA
                __syncwarp();
                if (lane == 0 && m0 < p.M) {
                    for (int b = 0; b < BN / BOX_COLS; ++b)
                        if (n0 + b * BOX_COLS < p.N) tma_store_2d(&tmD, smem_addr(stg + b * BOX_BYTES), n0 + b * BOX_COLS, m0);
                    bulk_commit();
                }
            }
            acc_phase ^= 1u;
        }
        if constexpr (STAGED) {
            if (lane == 0) bulk_wait0();
            __syncwarp();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(TMEM_COLS) : "memory");
    }
}

// ============================================================================
// CTA-pair kernel (tcgen05 cta_group::2): one 256 x 256 output tile per pair of
// SMs, persistent.  The leader CTA (cluster rank 0) issues MMAs with M = 256:
// rows 0-127 of the tile come from the leader's A tile, rows 128-255 from the
// follower's, and the 256 B rows (N) are split the same way; each CTA's TMEM
// receives its own 128 rows of the accumulator.  Per CTA and stage the ring
// holds A 16 KB + B 16 KB + scales 6 KB = 38 KB, five stages deep.
//
// Sixteen warps in four warpgroups; registers move from the first two warpgroups to the
// epilogue's (setmaxnreg: 96 each for warpgroups 0-1, 160 each for 2-3):
//   warp 0      TMA producer of the codes tiles (two tensor copies per K tile);
//   warp 2      producer of the scale tiles: its A rows' 2 KB, and one of the B tile's two
//               2 KB blocks multicast to both CTAs (each CTA needs all of B's scales; the
//               pair releases every stage at once, so the copies need no extra wait).
//               Issuing a TMA copy occupies the issuing thread for about 100
//               cycles, so with one thread issuing every copy the codes tiles of a
//               freed stage started late; each copy per K tile costs the kernel
//               2-3 % of its time, so the B scale blocks are split between the CTAs;
//   warp 1      (leader) one lane issues the MMAs and commits them to both CTAs;
//   warps 4-7   scale warps: shared memory -> registers -> TMEM (tcgen05.st), then
//               tell the leader that this CTA's scales and codes tiles are ready;
//   warps 8-15  epilogue, two warps per 32-lane TMEM quarter, each owning 128 of the
//               256 accumulator columns: two tcgen05.ld of 64 columns, one wait, and
//               the accumulator is handed back -- the MMAs of the next tile start
//               while the warps convert (x alpha with packed multiplies, bf16) their
//               two 32 x 64 boxes through one 128-byte swizzled 4 KB slot each and
//               TMA-store them.
// Cross-CTA signals: the leader's MMA commits are multicast to both CTAs'
// barriers; the follower's scale and epilogue warps arrive remotely on the
// leader's sf_ready / acc_empty barriers.
// ============================================================================
constexpr int P_THREADS = 512;                                         // 16 warps (4 warpgroups)
constexpr int P_EPI_WARP0 = 8;                                         // epilogue warps 8-15
constexpr int P_REGS_LOW = 96, P_REGS_HIGH = 160;                      // setmaxnreg split (of 128 each at launch)
static_assert(2 * 128 * P_REGS_LOW + 2 * 128 * P_REGS_HIGH <= P_THREADS * 128, "register split within the launch's registers");
constexpr int P_B_BYTES = 128 * BKB;                                   // half of N per CTA
constexpr int P_STAGE_BYTES = A_BYTES + P_B_BYTES + SFA_BYTES + SFB_BYTES;   // 38 KB
constexpr int P_STAGES = 5;
constexpr int P_STAGING_BYTES = 8 * BOX_BYTES;                         // one box slot per epilogue warp
constexpr int P_RING_BYTES = P_STAGES * P_STAGE_BYTES;
constexpr int P_SMEM_BYTES = P_RING_BYTES + P_STAGING_BYTES + BAR_BYTES + 1024;   // + base alignment
static_assert(P_STAGE_BYTES % 1024 == 0, "pair stages must stay 1024-byte aligned");
static_assert(P_SMEM_BYTES <= SMEM_LIMIT, "pair shared memory budget");
static_assert(SF_COL0 + P_STAGES * SF_STAGE_COLS <= TMEM_COLS, "pair TMEM budget");
// M = 256 (both CTAs), N = 256
constexpr uint32_t IDESC_PAIR = (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
// MXFP4 operands: the same E2M1 codes with UE8M0 scales (bit 23), one per 32 elements
// (scale_vec::2X: two scale bytes per row per K = 64 MMA, scale-factor IDs 0).
constexpr uint32_t IDESC_PAIR_MX = IDESC_PAIR | (1u << 23);
// Scale bytes of one 128-row block per 256-wide K tile: 16 E4M3 (NVFP4) or 8 UE8M0 (MXFP4) a row.
template <bool MX> struct PairSf { static constexpr uint32_t TILE = MX ? 1024u : 2048u; };

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
// Arrive on a barrier of another CTA of the cluster.  Default (CTA-scope) semantics:
// what it guards is already complete when it is issued (tcgen05.wait::st for the
// scale writes, a local TMA barrier for the codes tiles, tcgen05.ld for the
// accumulator), and a cluster-scope release fence on every k-tile stalled the
// issuing warps (membar) for most of the run time.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" :: "r"(cluster_addr) : "memory");
}
template <bool MX>
__device__ __forceinline__ void tc_mma_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t sfa, uint32_t sfb,
                                            uint32_t accumulate) {
    if constexpr (MX)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;\n\t}"
            :: "r"(d), "l"(a), "l"(b), "r"(IDESC_PAIR_MX), "r"(accumulate), "r"(sfa), "r"(sfb) : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}"
            :: "r"(d), "l"(a), "l"(b), "r"(IDESC_PAIR), "r"(accumulate), "r"(sfa), "r"(sfb) : "memory");
}
// Arrive on the barrier at this offset in both CTAs of the pair when the MMAs issued so far complete.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
                 :: "r"(bar), "h"((uint16_t)0x3) : "memory");
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 64 fp32 accumulator columns -> x alpha (packed multiplies) -> bf16 -> one 32 x 64
// box in shared memory, 128-byte swizzled (16-byte chunk c of row r at chunk
// c ^ (r & 7)), the layout the TMA store expects.  Lane = row.
__device__ __forceinline__ void box_to_smem(const uint32_t (&v)[64], uint8_t* box, int lane, float alpha) {
    uint8_t* row = box + lane * 128;
    const float2 al = make_float2(alpha, alpha);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 s = __fmul2_rn(make_float2(__uint_as_float(v[8 * c + 2 * i]),
                                                    __uint_as_float(v[8 * c + 2 * i + 1])), al);
            const __nv_bfloat162 h = __float22bfloat162_rn(s);
            w[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(row + ((c ^ (lane & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// The same box for D = dH = dA * 2 relu(H): the slot already holds the matching 32 x 64 box of
// H (TMA-loaded, same swizzle); each value is first rounded to bf16 exactly as the plain
// epilogue stores dA, then multiplied by (h > 0 ? 2h : +0) in fp32 and rounded to bf16 --
// the arithmetic of the separate squared-ReLU backward kernel, so the fused result equals
// GEMM-then-backward bit for bit.
__device__ __forceinline__ void box_to_smem_dsqr(const uint32_t (&v)[64], uint8_t* box, int lane, float alpha) {
    uint8_t* row = box + lane * 128;
    const float2 al = make_float2(alpha, alpha);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        uint4* slot = reinterpret_cast<uint4*>(row + ((c ^ (lane & 7)) << 4));
        const uint4 hq = *slot;
        const uint32_t hw[4] = {hq.x, hq.y, hq.z, hq.w};
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 s = __fmul2_rn(make_float2(__uint_as_float(v[8 * c + 2 * i]),
                                                    __uint_as_float(v[8 * c + 2 * i + 1])), al);
            const __nv_bfloat162 da = __float22bfloat162_rn(s);
            const float hl = bf16_lo(hw[i]), hh = bf16_hi(hw[i]);
            const float2 t = make_float2(hl > 0.0f ? __fmul_rn(2.0f, hl) : 0.0f, hh > 0.0f ? __fmul_rn(2.0f, hh) : 0.0f);
            const __nv_bfloat162 dh = __float22bfloat162_rn(__fmul2_rn(__bfloat1622float2(da), t));
            w[i] = *reinterpret_cast<const uint32_t*>(&dh);
        }
        *slot = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

template <int EPI>
__device__ __forceinline__ void box_out(const uint32_t (&v)[64], uint8_t* box, int lane, float alpha) {
    if constexpr (EPI == EPI_DSQR || EPI == EPI_DSQR_AMAX) box_to_smem_dsqr(v, box, lane, alpha);
    else box_to_smem(v, box, lane, alpha);
}

// Folds one stored 32 x 64 box (rows m0.., columns n0..) into the warp's running maxima of
// the tensor the next quantization reads -- the box's values x, or with SQR a = relu(x)^2
// formed as the quantizer's load transform forms it -- exactly as its dual amax pass computes
// them: mabs = max |a| and mrht = max |t| with t the unnormalised 16-point butterflies of
// (s_i * a_i) down each 16-row group (bit patterns of non-negative floats; a NaN lands above
// every finite value).  Lane l takes column pair 2l, 2l+1; rows past M and columns past N
// (both multiples of 16) are left out.
template <bool SQR>
__device__ __forceinline__ void box_maxima(const uint8_t* box, int lane, int m0, int M, int n0, int N,
                                           uint32_t sign_mask, uint32_t& mabs, uint32_t& mrht) {
    if (n0 + 2 * lane >= N) return;
#pragma unroll 1
    for (int g = 0; g < 2; ++g) {                        // one group at a time: bounded registers
        if (m0 + 16 * g >= M) break;
        float2 t[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int r = 16 * g + i;
            uint32_t w = *reinterpret_cast<const uint32_t*>(box + r * 128 + ((((lane >> 2) ^ (r & 7)) << 4) |
                                                                              ((lane & 3) << 2)));
            if constexpr (SQR) w = sqrelu_bf16x2(w);
            mabs = max(mabs, max((w << 16) & 0x7FFFFFFFu, w & 0x7FFF0000u));
            if ((sign_mask >> i) & 1u) w ^= 0x80008000u;
            t[i] = make_float2(bf16_lo(w), bf16_hi(w));
        }
        hadamard16_x2(t);
#pragma unroll
        for (int i = 0; i < 16; ++i)
            mrht = max(mrht, max(__float_as_uint(t[i].x) & 0x7FFFFFFFu, __float_as_uint(t[i].y) & 0x7FFFFFFFu));
    }
}

// One half of a split tail tile (see pair_item; the host splits in two, so two parts meet).
// The warp adds its 32 x 128 fp32 partial sums (va: columns 0-63, vb: 64-127 of its slice) into
// the tile's sum buffer in the workspace with vector reductions -- laid out as 32 groups of four
// columns x 32 lanes x 16 bytes, so each is one 512-byte run -- and counts itself in on the
// tile's counter.  The half that arrives second (returns true) loads the finished sums into
// va / vb for the normal epilogue and leaves buffer and counter at zero for the next call; the
// first returns false and stores nothing.  0 + a + b == 0 + b + a in fp32, so the result does not
// depend on which half finishes first, and no half waits for the other.  (The reductions flush
// subnormal values; the accumulator of E2M1 x E4M3 products is a multiple of 2^-20, never
// subnormal.)
__device__ __forceinline__ bool split_partial(const Params& p, int tail_tile, uint32_t rank, int e, int lane,
                                              uint32_t (&va)[64], uint32_t (&vb)[64]) {
    float4* buf = reinterpret_cast<float4*>(p.split_ws + (((size_t)tail_tile * 2 + rank) * 8 + e) * (32 * 128));
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const uint32_t* v = j < 16 ? &va[4 * j] : &vb[4 * (j - 16)];
        asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};"
                     :: "l"(buf + j * 32 + lane), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]) : "memory");
    }
    __threadfence();
    __syncwarp();
    uint32_t* cnt = p.split_cnt + ((size_t)tail_tile * 2 + rank) * 8 + e;
    uint32_t before = 0;
    if (lane == 0) before = atomicAdd(cnt, 1u);
    before = __shfl_sync(0xFFFFFFFFu, before, 0);
    if (before == 0) return false;
    __threadfence();
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const float4 x = __ldcg(buf + j * 32 + lane);
        uint32_t* v = j < 16 ? &va[4 * j] : &vb[4 * (j - 16)];
        v[0] = __float_as_uint(x.x); v[1] = __float_as_uint(x.y);
        v[2] = __float_as_uint(x.z); v[3] = __float_as_uint(x.w);
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) __stcg(buf + j * 32 + lane, make_float4(0.0f, 0.0f, 0.0f, 0.0f));
    if (lane == 0) *cnt = 0u;
    return true;
}

__device__ __forceinline__ void tmem_ld_64cols(uint32_t taddr, uint32_t (&v)[64]) {
    tmem_ld_32cols_nowait(taddr, *reinterpret_cast<uint32_t (*)[32]>(&v[0]));
    tmem_ld_32cols_nowait(taddr + 32, *reinterpret_cast<uint32_t (*)[32]>(&v[32]));
}
__device__ __forceinline__ void reg_fence64(uint32_t (&v)[64]) {
    reg_fence32(*reinterpret_cast<uint32_t (*)[32]>(&v[0]));
    reg_fence32(*reinterpret_cast<uint32_t (*)[32]>(&v[32]));
}

// MX: MXFP4 operands.  EPI: the epilogue variant (EPI_DSQR reads H through tmH: bf16, same
// shape and box as D).  SPLIT: the tail tiles are cut in two along K (p.split == 2; NVFP4 with
// EPI_PLAIN only) -- a separate instantiation, so kernels that never split carry none of it.
template <bool MX, int EPI, bool SPLIT = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(P_THREADS, 1)
gemm_nvfp4_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmH,
                       const Params p) {
    constexpr int STAGES = P_STAGES;
    constexpr bool DSQR = EPI == EPI_DSQR || EPI == EPI_DSQR_AMAX;   // output dH from dA and H
    constexpr bool AMAX = EPI == EPI_SQAMAX || EPI == EPI_DSQR_AMAX; // leave the output's tensor maxima
    constexpr bool SQR_MAX = EPI == EPI_SQAMAX;                      // ... of relu(output)^2
    // the next kernel may launch now; this one touches global memory only after pdl_wait below
    pdl_launch_dependents();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* staging = smem + P_RING_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(staging + P_STAGING_BYTES);   // local A/B landed
    uint64_t* empty = full + STAGES;                     // the stage's MMAs completed (leader's commit, both CTAs)
    uint64_t* sf_loaded = empty + STAGES;                // local scale tiles landed
    uint64_t* sf_ready = sf_loaded + STAGES;             // leader: 8 scale warps wrote TMEM and saw their A/B
    uint64_t* acc_full = sf_ready + STAGES;              // accumulator complete (leader's commit)
    uint64_t* acc_empty = acc_full + 1;                  // leader: 8 epilogue warps drained
    uint64_t* drain = acc_empty + 1;
    uint64_t* h_full = drain + 1;                        // DSQR: per epilogue warp, its H box landed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(h_full + 8);
    volatile uint32_t* abort_flag = tmem_slot + 1;
    // identical in both CTAs (same kernel, same dynamic smem base), so layout_ok is uniform
    const bool layout_ok = (reinterpret_cast<uintptr_t>(tmem_slot + 2) - reinterpret_cast<uintptr_t>(smem_raw)) <=
                           (uintptr_t)P_SMEM_BYTES;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    if (!layout_ok) {
        pdl_wait();
        if (threadIdx.x == 0) set_status(p.dev_status, NVFP4_ERR_UNSUPPORTED);
        return;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&sf_loaded[s], 1);
            mbar_init(&sf_ready[s], 8);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 16);
        mbar_init(drain, 1);
        for (int e = 0; e < 8; ++e) mbar_init(&h_full[e], 1);
        *abort_flag = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {    // one warp in each CTA of the pair allocates collectively
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_addr(tmem_slot)), "r"(TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    cluster_sync();                                      // barriers initialised in both CTAs
    tc_fence_after();
    // the prologue (barriers, TMEM) overlapped the previous kernel's tail; its results are needed now
    pdl_wait();
    const uint32_t tmem = *tmem_slot;
    const int m_pairs = (p.M + 255) / 256;
    const int tiles = m_pairs * p.n_tiles;
    const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
    const uint32_t sf_ready_leader = map_to_rank(smem_addr(&sf_ready[0]), 0);
    const uint32_t acc_empty_leader = map_to_rank(smem_addr(acc_empty), 0);
    // Registers move from the producer / MMA / scale warpgroups (0-1) to the epilogue's (2-3):
    // each warpgroup enters one branch whose first instruction is its setmaxnreg, so the
    // compiler allocates every role's code within its share.
    if (warp < P_EPI_WARP0) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" :: "n"(P_REGS_LOW));
    if (warp == 0 || warp == 2) {
        // ------------------------------------------------ producers (each CTA, its own halves):
        // warp 0 the codes tiles, warp 2 the scale tiles, both over the same ring
        if (lane == 0) {
            const bool codes = warp == 0;
            uint64_t* landed = codes ? full : sf_loaded;
            uint32_t stage = 0, phase = 0;
            uint32_t issued_mask = 0, issued_phase = 0;
            bool ok = true;
            PairItem it;
            for (int item = 0; ok && pair_item(p, tiles, cluster, nclusters, item, it); ++item) {
                int mp, nt;
                tile_coords(p, it.tile, m_pairs, mp, nt);
                const int mrow = mp * 256 + (int)rank * 128;      // this CTA's A rows
                const int nrow = nt * BN + (int)rank * 128;       // this CTA's B rows
                const bool second_sfb = (nt * BN + 128) < p.N;
                // rows past M (the follower's half of the last pair tile) have no scale block:
                // their codes load as zeros and their output rows are never stored
                const bool has_sfa = mrow < p.M;
                constexpr uint32_t SFT = PairSf<MX>::TILE;
                const uint32_t sf_bytes = (has_sfa ? SFT : 0) + (second_sfb ? 2 * SFT : SFT);
                for (int kt = it.kb; kt < it.ke; ++kt) {
                    if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, p.timeout_ns, abort_flag, p.dev_status)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sA = smem + stage * P_STAGE_BYTES;
                    const uint32_t bar = smem_addr(&landed[stage]);
                    if (codes) {
                        mbar_arrive_expect_tx(&full[stage], A_BYTES + P_B_BYTES);
                        tma_load_2d(smem_addr(sA), &tmA, kt * BKB, mrow, bar);
                        tma_load_2d(smem_addr(sA + A_BYTES), &tmB, kt * BKB, nrow, bar);
                    } else {
                        uint8_t* sSFA = sA + A_BYTES + P_B_BYTES;
                        uint8_t* sSFB = sSFA + SFA_BYTES;
                        mbar_arrive_expect_tx(&sf_loaded[stage], sf_bytes);
                        if (has_sfa)
                            bulk_load(smem_addr(sSFA), p.sfa + ((size_t)(mrow / 128) * p.nkt + kt) * SFT, SFT, bar);
                        // both CTAs need all of the tile's B scales: CTA r loads 128-row block r
                        // (when it exists) into both; the pair releases every stage at once
                        if (rank == 0 || second_sfb)
                            bulk_load_mc(smem_addr(sSFB + rank * SFT), p.sfb + ((size_t)(2 * nt + rank) * p.nkt + kt) * SFT,
                                         SFT, bar, (uint16_t)0x3);
                    }
                    issued_mask |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {   // let every copy this thread started land before the CTA exits
                for (int s = 0; s < STAGES; ++s)
                    if (issued_mask & (1u << s))
                        mbar_wait_bounded(&landed[s], (issued_phase >> s) & 1u, p.timeout_ns, nullptr, p.dev_status);
                // a multicast scale copy lands in the other CTA too, whose barrier this thread
                // cannot wait on: give it a fixed 50 us, far above a copy's latency
                if (!codes) {
                    const uint64_t t0 = global_ns();
                    while (global_ns() - t0 < 50000ull) {}
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (leader only)
        if (lane == 0 && leader) {
            uint32_t stage = 0, phase = 0, acc_phase = 0;
            bool ok = true, issued = false;
            PairItem it;
            for (int item = 0; ok && pair_item(p, tiles, cluster, nclusters, item, it); ++item) {
                if (!mbar_wait_bounded(acc_empty, acc_phase ^ 1u, p.timeout_ns, abort_flag, p.dev_status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int kt = it.kb; kt < it.ke; ++kt) {
                    if (!mbar_wait_bounded(&sf_ready[stage], phase, p.timeout_ns, abort_flag, p.dev_status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sA = smem_addr(smem + stage * P_STAGE_BYTES);
                    const uint64_t da = desc_sw128(sA), db = desc_sw128(sA + A_BYTES);
                    const uint32_t tsf = tmem + SF_COL0 + stage * SF_STAGE_COLS;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        tc_mma_pair<MX>(tmem + ACC_COL, da + 2 * j, db + 2 * j, tsf + 4 * j, tsf + 16 + 8 * j,
                                        (kt != it.kb || j != 0) ? 1u : 0u);
                    issued = true;
                    tc_commit_pair(smem_addr(&empty[stage]));
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                tc_commit_pair(smem_addr(acc_full));
                acc_phase ^= 1u;
            }
            if (!ok && issued) {
                tc_commit_pair(smem_addr(drain));
                mbar_wait_bounded(drain, 0u, p.timeout_ns, nullptr, p.dev_status);
            }
        }
    } else if (warp >= 4 && warp < P_EPI_WARP0) {
        // ------------------------------------------------ scale warps 4-7 (each CTA, its own TMEM)
        const int q = warp & 3;
        const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16);
        uint32_t stage = 0, phase = 0;
        bool ok = true;
        PairItem it;
        for (int item = 0; ok && pair_item(p, tiles, cluster, nclusters, item, it); ++item) {
            for (int kt = it.kb; kt < it.ke; ++kt) {
                if (!mbar_wait_bounded(&sf_loaded[stage], phase, p.timeout_ns, abort_flag, p.dev_status)) {
                    ok = false;
                    break;
                }
                const uint8_t* sSFA = smem + stage * P_STAGE_BYTES + A_BYTES + P_B_BYTES;
                const uint8_t* sSFB = sSFA + SFA_BYTES;
                uint32_t va[16], vb0[16], vb1[16];
                if constexpr (!MX) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint4 a4 = *reinterpret_cast<const uint4*>(sSFA + 512 * j + 16 * lane);
                        va[4 * j] = a4.x; va[4 * j + 1] = a4.y; va[4 * j + 2] = a4.z; va[4 * j + 3] = a4.w;
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
#pragma unroll
                        for (int nb = 0; nb < 2; ++nb) {
                            const uint4 b4 = *reinterpret_cast<const uint4*>(sSFB + 2048 * nb + 512 * j + 16 * lane);
                            const int o = 8 * j + 4 * nb;
                            uint32_t* dst = o < 16 ? vb0 : vb1;
                            dst[(o & 15)] = b4.x; dst[(o & 15) + 1] = b4.y; dst[(o & 15) + 2] = b4.z;
                            dst[(o & 15) + 3] = b4.w;
                        }
                    }
                } else {
                    // a 512-byte piece holds 4 scales (= two K = 64 steps) per row: the low
                    // halfword of a row's word feeds step 2h, the high one step 2h + 1, each
                    // written to the low halfword of that step's column (scale-factor ID 0)
                    auto split = [](uint32_t w, int step_odd) { return step_odd ? (w >> 16) : (w & 0xFFFFu); };
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint4 a4 = *reinterpret_cast<const uint4*>(sSFA + 512 * h + 16 * lane);
                        const uint32_t aw[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                        for (int odd = 0; odd < 2; ++odd)
#pragma unroll
                            for (int c = 0; c < 4; ++c) va[4 * (2 * h + odd) + c] = split(aw[c], odd);
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
#pragma unroll
                        for (int nb = 0; nb < 2; ++nb) {
                            const uint4 b4 = *reinterpret_cast<const uint4*>(sSFB + 1024 * nb + 512 * h + 16 * lane);
                            const uint32_t bw[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                            for (int odd = 0; odd < 2; ++odd) {
                                const int o = 8 * (2 * h + odd) + 4 * nb;
                                uint32_t* dst = o < 16 ? vb0 : vb1;
#pragma unroll
                                for (int c = 0; c < 4; ++c) dst[(o & 15) + c] = split(bw[c], odd);
                            }
                        }
                    }
                }
                const uint32_t tsf = tq + SF_COL0 + stage * SF_STAGE_COLS;
                tmem_st_16cols(tsf, va);
                tmem_st_16cols(tsf + 16, vb0);
                tmem_st_16cols(tsf + 32, vb1);
                tmem_st_wait();
                // this CTA's codes tiles must have landed too before the leader may issue
                if (!mbar_wait_bounded(&full[stage], phase, p.timeout_ns, abort_flag, p.dev_status)) {
                    ok = false;
                    break;
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(sf_ready_leader + 8u * stage);
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
    }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" :: "n"(P_REGS_HIGH));
        // ------------------------------------------------ epilogue (warps 8-15, each CTA, its 128 rows)
        const int e = warp - P_EPI_WARP0;                // 0-7
        const int q = warp & 3;                          // TMEM lane quarter (warp % 4)
        const int h = e >> 2;                            // accumulator columns [128 h, 128 h + 128)
        const float alpha = MX ? 1.0f : __fmul_rn(*p.sdec_a, *p.sdec_b);   // MXFP4 has no tensor scale
        const uint32_t tmem_row = tmem + ((uint32_t)(q * 32) << 16) + ACC_COL + 128u * h;
        uint8_t* slot = staging + e * BOX_BYTES;
        const uint64_t stream_pol = l2_evict_first_policy();
        uint32_t acc_phase = 0, h_phase = 0;
        bool h_pending = false;                          // DSQR: an H box in flight into the slot
        uint32_t mabs = 0u, mrht = 0u;                   // AMAX: running maxima (float bits)
        const uint32_t sign_mask = AMAX ? rht_sign_mask(p.rht_seed) : 0u;
        bool ok = true;
        PairItem it;
        for (int item = 0; ok && pair_item(p, tiles, cluster, nclusters, item, it); ++item) {
            int mp, nt;
            tile_coords(p, it.tile, m_pairs, mp, nt);
            const int m0 = mp * 256 + (int)rank * 128 + q * 32, nb = nt * BN + 128 * h;
            // DSQR: the H box of output box b (columns nb + 64 b) into the slot, and the wait for it
            // (boxes past M or N read the fill value; their results are never stored)
            auto load_h = [&](int b) {
                if (lane == 0) {
                    mbar_arrive_expect_tx(&h_full[e], BOX_BYTES);
                    tma_load_2d_hint(smem_addr(slot), &tmH, nb + b * BOX_COLS, m0, smem_addr(&h_full[e]), stream_pol);
                }
                h_pending = true;
            };
            auto wait_h = [&]() -> bool {
                if (!mbar_wait_bounded(&h_full[e], h_phase, p.timeout_ns, abort_flag, p.dev_status)) return false;
                h_phase ^= 1u;
                h_pending = false;
                return true;
            };
            // box b from the slot: TMA store (clipped at M and N), then its maxima
            auto store_box = [&](int b) {
                fence_proxy_async_smem();                // generic-proxy writes -> visible to TMA
                __syncwarp();
                if (lane == 0) {
                    if (m0 < p.M && nb + b * BOX_COLS < p.N)
                        tma_store_2d_hint(&tmD, smem_addr(slot), nb + b * BOX_COLS, m0, stream_pol);
                    bulk_commit();
                }
                if constexpr (AMAX) box_maxima<SQR_MAX>(slot, lane, m0, p.M, nb + b * BOX_COLS, p.N, sign_mask, mabs, mrht);
            };
            auto slot_free = [&]() {                     // the last store has read the slot (and every lane is done with it)
                __syncwarp();
                if (lane == 0) bulk_wait_read0();
                __syncwarp();
            };
            slot_free();
            if constexpr (DSQR) {
                if (lane == 0) fence_proxy_async_smem();
                load_h(0);
            }
            if (!mbar_wait_bounded(acc_full, acc_phase, p.timeout_ns, abort_flag, p.dev_status)) break;
            tc_fence_after();
            uint32_t va[64], vb[64];
            tmem_ld_64cols(tmem_row, va);
            tmem_ld_64cols(tmem_row + 64, vb);
            tmem_ld_wait();
            reg_fence64(va);
            reg_fence64(vb);
            // this warp's 128 columns are in registers: hand its share of the accumulator back
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(acc_empty_leader);
            acc_phase ^= 1u;
            if constexpr (SPLIT) {
                if (it.part >= 0 && !split_partial(p, it.tile - tiles / nclusters * nclusters, rank, e, lane, va, vb))
                    continue;
            }
            if constexpr (DSQR) {
                if (!wait_h()) { ok = false; break; }
            }
            box_out<EPI>(va, slot, lane, alpha);
            store_box(0);
            slot_free();
            if constexpr (DSQR) {
                if (lane == 0) fence_proxy_async_smem();
                load_h(1);
                if (!wait_h()) { ok = false; break; }
            }
            box_out<EPI>(vb, slot, lane, alpha);
            store_box(1);
        }
        if constexpr (AMAX) {
            // this warp's partials; the first CTA zeroes the slots no CTA of this grid owns
            mabs = __reduce_max_sync(0xFFFFFFFFu, mabs);
            mrht = __reduce_max_sync(0xFFFFFFFFu, mrht);
            const int gid = (int)blockIdx.x * kMaximaWarpsPerCta + e;
            if (lane == 0) {
                p.maxima[gid] = mabs;
                p.maxima[p.maxima_parts + gid] = __float_as_uint(__fmul_rn(__uint_as_float(mrht), 0.25f)) & 0x7FFFFFFFu;
            }
            if (blockIdx.x == 0)
                for (int i = (int)gridDim.x * kMaximaWarpsPerCta + e * 32 + lane; i < p.maxima_parts;
                     i += kMaximaWarpsPerCta * 32) {
                    p.maxima[i] = 0u;
                    p.maxima[p.maxima_parts + i] = 0u;
                }
        }
        if (h_pending)                                   // after an abort: let the H copy land first
            mbar_wait_bounded(&h_full[e], h_phase, p.timeout_ns, nullptr, p.dev_status);
        if (lane == 0) bulk_wait0();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();                                      // neither CTA leaves while the other may signal it
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(TMEM_COLS) : "memory");
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

// bf16 D [M, N] (pitch ldd elements): 64 x 32 boxes, 128-byte swizzle, for the TMA stores.
bool make_out_map(CUtensorMap* m, void* D, int64_t M, int64_t N, int64_t ldd) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
    cuuint64_t strides[1] = {(cuuint64_t)(ldd * 2)};
    cuuint32_t box[2] = {(cuuint32_t)BOX_COLS, 32u};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <bool STAGED>
cudaError_t launch(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& td, const Params& p, int grid,
                   cudaStream_t stream) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(gemm_nvfp4_kernel<STAGED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        Cfg<STAGED>::SMEM_BYTES);
    });
    if (attr_err != cudaSuccess) return attr_err;
    return launch_pdl(gemm_nvfp4_kernel<STAGED>, dim3(grid), dim3(NUM_THREADS), Cfg<STAGED>::SMEM_BYTES, stream, ta, tb,
                      td, p);
}

// Split-tail workspace: a sum buffer per tail tile (at most one per cluster; each CTA's 128 x 256
// fp32), then the arrival counters (per tail tile, CTA and epilogue warp); both start at zero
// and every call leaves them at zero.
constexpr int kSplitMaxWaves = 16;       // split the tail only below this many full waves
inline size_t split_partials_bytes(int sms) { return (size_t)(sms / 2) * 2 * 128 * 256 * sizeof(float); }
inline size_t split_ws_bytes(int sms) { return split_partials_bytes(sms) + (size_t)(sms / 2) * 2 * 8 * sizeof(uint32_t); }

// One-time set-up of a pair-kernel instantiation: its shared memory, the register check and
// the clusters that fit at once.
template <bool MX, int EPI, bool SPLIT>
cudaError_t pair_setup(int sms, int* max_clusters) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    static int clusters = 0;
    std::call_once(once, [sms] {
        attr_err = cudaFuncSetAttribute(gemm_nvfp4_pair_kernel<MX, EPI, SPLIT>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM_BYTES);
        if (attr_err != cudaSuccess) return;
        // The kernel moves registers between warpgroups with setmaxnreg; the epilogue's
        // increase only completes if the launch holds at least the split's total, so a build
        // that allocated fewer registers per thread is never launched.
        cudaFuncAttributes fa;
        attr_err = cudaFuncGetAttributes(&fa, gemm_nvfp4_pair_kernel<MX, EPI, SPLIT>);
        if (attr_err != cudaSuccess) return;
        if (fa.numRegs * P_THREADS < 2 * 128 * P_REGS_LOW + 2 * 128 * P_REGS_HIGH) {
            attr_err = cudaErrorInvalidConfiguration;
            return;
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
        cfg.blockDim = dim3(P_THREADS, 1, 1);
        cfg.dynamicSmemBytes = P_SMEM_BYTES;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, gemm_nvfp4_pair_kernel<MX, EPI, SPLIT>, &cfg) != cudaSuccess || n <= 0)
            n = sms / 2;
        clusters = n;
    });
    *max_clusters = clusters;
    return attr_err;
}

template <bool MX, int EPI = EPI_PLAIN>
cudaError_t launch_pair(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& td, const CUtensorMap& th,
                        Params p, int pair_tiles, int sms, cudaStream_t stream, void* split_ws = nullptr) {
    int max_clusters = 0;
    const cudaError_t err = pair_setup<MX, EPI, false>(sms, &max_clusters);
    if (err != cudaSuccess) return err;
    const int clusters = std::max(1, std::min(pair_tiles, max_clusters));
    // Split tail: cut the last partial wave's r tiles in two along K so that it takes half a
    // tile's time, when there are clusters for both halves (2 r <= clusters), K spans two K
    // tiles, and the waves are few enough for half a tile to outweigh the split kernel's longer
    // epilogue (measured: worth it at 9 waves, not at 22).  Two halves meet by order-free fp32
    // reductions (deterministic); more parts would need an order-fixed sum the reductions
    // cannot give.  NVFP4 only (MXFP4's power-of-two scales reach the subnormal range the
    // reductions flush).
    p.split = 1;
    const int r = pair_tiles % clusters;
    if constexpr (EPI == EPI_PLAIN && !MX) {
        if (split_ws && r != 0 && 2 * r <= clusters && p.nkt >= 2 && pair_tiles / clusters < kSplitMaxWaves) {
            int split_clusters = 0;
            const cudaError_t e2 = pair_setup<MX, EPI, true>(sms, &split_clusters);
            if (e2 != cudaSuccess) return e2;
            if (split_clusters == max_clusters) {
                p.split = 2;
                p.split_ws = static_cast<float*>(split_ws);
                p.split_cnt = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(split_ws) + split_partials_bytes(sms));
                return launch_pdl(gemm_nvfp4_pair_kernel<MX, EPI, true>, dim3(2 * clusters), dim3(P_THREADS),
                                  P_SMEM_BYTES, stream, ta, tb, td, th, p);
            }
        }
    }
    return launch_pdl(gemm_nvfp4_pair_kernel<MX, EPI, false>, dim3(2 * clusters), dim3(P_THREADS), P_SMEM_BYTES,
                      stream, ta, tb, td, th, p);
}

int g_force_path = 0;      // 0: automatic, 1: single-CTA kernel, 2: CTA-pair kernel (tests)

}  // namespace gemm

nvfp4_status gemm_impl(const nvfp4_qtensor* A, const nvfp4_qtensor* B, void* D, int32_t d_dtype, int64_t ldd,
                       uint32_t* dev_status, cudaStream_t stream, void* ws, size_t ws_bytes) {
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
    if (ws && (ws_bytes < split_ws_bytes(sm_count(dev)) || !aligned16(ws))) return NVFP4_ERR_WORKSPACE;
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
    // re-sweep the smaller operand: walk N fastest when A is the larger one
    p.n_fastest = (M > N) ? 1 : 0;
    p.dev_status = dev_status;
    p.timeout_ns = wait_timeout_ns();
    const int tiles = p.m_tiles * p.n_tiles;
    const int grid = std::max(1, std::min(tiles, sm_count(dev)));
    // bf16 output with a 16-byte aligned base and pitch goes through the staged TMA-store epilogue
    CUtensorMap td;
    const bool staged = p.d_bf16 && p.vec_store && make_out_map(&td, D, M, N, ldd);
    if (!staged) std::memset(&td, 0, sizeof(td));
    // The CTA-pair kernel needs the staged bf16 epilogue and enough 256 x 256 tiles to fill the SMs.
    const int pair_tiles = (int)((M + 255) / 256) * p.n_tiles;
    bool pair = staged && (pair_tiles * 2 >= sm_count(dev) || g_force_path == 2);
    if (g_force_path == 1) pair = false;
    cudaError_t e;
    if (pair) {
        CUtensorMap tb2;      // B boxes of 128 rows (each CTA loads its half of the N tile)
        if (!make_codes_map(&tb2, B->codes, N, K, 128)) return NVFP4_ERR_CUDA;
        e = launch_pair<false>(ta, tb2, td, td, p, pair_tiles, sm_count(dev), stream, ws);
    } else {
        e = staged ? launch<true>(ta, tb, td, p, grid, stream) : launch<false>(ta, tb, td, p, grid, stream);
    }
    return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

// MXFP4 operands through the CTA-pair kernel (bf16 output, 16-byte aligned base and pitch).
nvfp4_status mx_gemm_impl(const nvfp4_qtensor* A, const nvfp4_qtensor* B, void* D, int32_t d_dtype, int64_t ldd,
                          uint32_t* dev_status, cudaStream_t stream) {
    using namespace gemm;
    if (!A || !B || !D) return NVFP4_ERR_INVALID_ARG;
    if (d_dtype != NVFP4_F32 && d_dtype != NVFP4_BF16) return NVFP4_ERR_INVALID_ARG;
    if (d_dtype != NVFP4_BF16) return NVFP4_ERR_UNSUPPORTED;
    if (!A->codes || !B->codes || !A->scales_mma || !B->scales_mma) return NVFP4_ERR_INVALID_ARG;
    const int64_t M = A->rows, N = B->rows, K = A->cols;
    if (B->cols != K) return NVFP4_ERR_SHAPE;
    if (M < 1 || N < 1 || K < 32 || K % 32 != 0 || ldd < N) return NVFP4_ERR_SHAPE;
    if (M > (1ll << 30) || N > (1ll << 30) || K > (1ll << 30)) return NVFP4_ERR_SHAPE;
    if (!aligned16(A->codes) || !aligned16(B->codes) || !aligned16(A->scales_mma) || !aligned16(B->scales_mma) ||
        !aligned16(D) || (ldd * 2) % 16 != 0)
        return NVFP4_ERR_ALIGNMENT;
    CUtensorMap ta, tb, td;
    if (!make_codes_map(&ta, A->codes, M, K, BM) || !make_codes_map(&tb, B->codes, N, K, 128) ||
        !make_out_map(&td, D, M, N, ldd))
        return NVFP4_ERR_CUDA;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return NVFP4_ERR_CUDA;
    Params p;
    std::memset(&p, 0, sizeof(p));
    p.sfa = A->scales_mma;
    p.sfb = B->scales_mma;
    p.D = D;
    p.ldd = ldd;
    p.M = (int)M;
    p.N = (int)N;
    p.K = (int)K;
    p.d_bf16 = 1;
    p.vec_store = 1;
    p.nkt = (int)((K + BK - 1) / BK);
    p.m_tiles = (int)((M + BM - 1) / BM);
    p.n_tiles = (int)((N + BN - 1) / BN);
    p.n_fastest = (M > N) ? 1 : 0;
    p.dev_status = dev_status;
    p.timeout_ns = wait_timeout_ns();
    const int pair_tiles = (int)((M + 255) / 256) * p.n_tiles;
    const cudaError_t e = launch_pair<true>(ta, tb, td, td, p, pair_tiles, sm_count(dev), stream);
    return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

// dH = bf16(dA) * 2 relu(H) with dA = s_dec(A) s_dec(B) A B^T: the NVFP4 GEMM with the squared-ReLU
// backward in its epilogue (CTA-pair kernel; bf16 H and D, 16-byte aligned bases and pitches).
// With `maxima`, the epilogue also leaves dH's two tensor maxima for its dual quantization.
nvfp4_status gemm_sqrelu_bwd_impl(const nvfp4_qtensor* A, const nvfp4_qtensor* B, const void* H, int64_t ldh,
                                  void* D, int64_t ldd, uint64_t rht_seed, uint32_t* maxima, size_t maxima_bytes,
                                  uint32_t* dev_status, cudaStream_t stream) {
    using namespace gemm;
    if (!A || !B || !H || !D) return NVFP4_ERR_INVALID_ARG;
    if (!A->codes || !B->codes || !A->scales_mma || !B->scales_mma || !A->s_dec || !B->s_dec)
        return NVFP4_ERR_INVALID_ARG;
    const int64_t M = A->rows, N = B->rows, K = A->cols;
    if (B->cols != K) return NVFP4_ERR_SHAPE;
    if (M < 1 || N < 1 || K < 32 || K % 32 != 0 || ldd < N || ldh < N) return NVFP4_ERR_SHAPE;
    if (maxima && (M % 16 != 0 || N % 16 != 0)) return NVFP4_ERR_SHAPE;
    if (M > (1ll << 30) || N > (1ll << 30) || K > (1ll << 30)) return NVFP4_ERR_SHAPE;
    if (!aligned16(A->codes) || !aligned16(B->codes) || !aligned16(A->scales_mma) || !aligned16(B->scales_mma) ||
        !aligned16(D) || !aligned16(H) || (ldd * 2) % 16 != 0 || (ldh * 2) % 16 != 0 ||
        (reinterpret_cast<uintptr_t>(maxima) & 3u) != 0)
        return NVFP4_ERR_ALIGNMENT;
    CUtensorMap ta, tb, td, th;
    if (!make_codes_map(&ta, A->codes, M, K, BM) || !make_codes_map(&tb, B->codes, N, K, 128) ||
        !make_out_map(&td, D, M, N, ldd) || !make_out_map(&th, const_cast<void*>(H), M, N, ldh))
        return NVFP4_ERR_CUDA;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return NVFP4_ERR_CUDA;
    if (maxima && maxima_bytes < 2 * sizeof(uint32_t) * kMaximaWarpsPerCta * (size_t)sm_count(dev))
        return NVFP4_ERR_WORKSPACE;                   // one partial per epilogue warp of every CTA
    Params p;
    std::memset(&p, 0, sizeof(p));
    p.sfa = A->scales_mma;
    p.sfb = B->scales_mma;
    p.sdec_a = A->s_dec;
    p.sdec_b = B->s_dec;
    p.D = D;
    p.ldd = ldd;
    p.M = (int)M;
    p.N = (int)N;
    p.K = (int)K;
    p.d_bf16 = 1;
    p.vec_store = 1;
    p.nkt = (int)((K + BK - 1) / BK);
    p.m_tiles = (int)((M + BM - 1) / BM);
    p.n_tiles = (int)((N + BN - 1) / BN);
    p.n_fastest = (M > N) ? 1 : 0;
    p.dev_status = dev_status;
    p.timeout_ns = wait_timeout_ns();
    p.maxima = maxima;
    p.maxima_parts = (int)std::min<size_t>(maxima_bytes / (2 * sizeof(uint32_t)), 1u << 30);
    p.rht_seed = rht_seed;
    const int pair_tiles = (int)((M + 255) / 256) * p.n_tiles;
    const cudaError_t e = maxima
        ? launch_pair<false, EPI_DSQR_AMAX>(ta, tb, td, th, p, pair_tiles, sm_count(dev), stream)
        : launch_pair<false, EPI_DSQR>(ta, tb, td, th, p, pair_tiles, sm_count(dev), stream);
    return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

// H = s_dec(A) s_dec(B) A B^T in bf16, plus the partial maxima that quantizing A = relu(H)^2
// in both orientations needs (CTA-pair kernel, EPI_SQAMAX).
nvfp4_status gemm_sqrelu_maxima_impl(const nvfp4_qtensor* A, const nvfp4_qtensor* B, void* D, int64_t ldd,
                                     uint64_t rht_seed, uint32_t* maxima, size_t maxima_bytes, uint32_t* dev_status,
                                     cudaStream_t stream) {
    using namespace gemm;
    if (!A || !B || !D || !maxima) return NVFP4_ERR_INVALID_ARG;
    if (!A->codes || !B->codes || !A->scales_mma || !B->scales_mma || !A->s_dec || !B->s_dec)
        return NVFP4_ERR_INVALID_ARG;
    const int64_t M = A->rows, N = B->rows, K = A->cols;
    if (B->cols != K) return NVFP4_ERR_SHAPE;
    if (M < 1 || N < 1 || K < 32 || K % 32 != 0 || ldd < N || M % 16 != 0 || N % 16 != 0) return NVFP4_ERR_SHAPE;
    if (M > (1ll << 30) || N > (1ll << 30) || K > (1ll << 30)) return NVFP4_ERR_SHAPE;
    if (!aligned16(A->codes) || !aligned16(B->codes) || !aligned16(A->scales_mma) || !aligned16(B->scales_mma) ||
        !aligned16(D) || (ldd * 2) % 16 != 0 || (reinterpret_cast<uintptr_t>(maxima) & 3u) != 0)
        return NVFP4_ERR_ALIGNMENT;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return NVFP4_ERR_CUDA;
    if (maxima_bytes < 2 * sizeof(uint32_t) * kMaximaWarpsPerCta * (size_t)sm_count(dev))
        return NVFP4_ERR_WORKSPACE;                   // one partial per epilogue warp of every CTA
    CUtensorMap ta, tb, td;
    if (!make_codes_map(&ta, A->codes, M, K, BM) || !make_codes_map(&tb, B->codes, N, K, 128) ||
        !make_out_map(&td, D, M, N, ldd))
        return NVFP4_ERR_CUDA;
    Params p;
    std::memset(&p, 0, sizeof(p));
    p.sfa = A->scales_mma;
    p.sfb = B->scales_mma;
    p.sdec_a = A->s_dec;
    p.sdec_b = B->s_dec;
    p.D = D;
    p.ldd = ldd;
    p.M = (int)M;
    p.N = (int)N;
    p.K = (int)K;
    p.d_bf16 = 1;
    p.vec_store = 1;
    p.nkt = (int)((K + BK - 1) / BK);
    p.m_tiles = (int)((M + BM - 1) / BM);
    p.n_tiles = (int)((N + BN - 1) / BN);
    p.n_fastest = (M > N) ? 1 : 0;
    p.dev_status = dev_status;
    p.timeout_ns = wait_timeout_ns();
    p.maxima = maxima;
    p.maxima_parts = (int)std::min<size_t>(maxima_bytes / (2 * sizeof(uint32_t)), 1u << 30);
    p.rht_seed = rht_seed;
    const int pair_tiles = (int)((M + 255) / 256) * p.n_tiles;
    const cudaError_t e = launch_pair<false, EPI_SQAMAX>(ta, tb, td, td, p, pair_tiles, sm_count(dev), stream);
    return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

}  // namespace nvfp4

extern "C" size_t nvfp4_sqrelu_maxima_bytes(int32_t device) {
    const int sms = nvfp4::sm_count(device);
    return sms > 0 ? 2u * sizeof(uint32_t) * nvfp4::kMaximaWarpsPerCta * (size_t)sms : 0u;
}

extern "C" nvfp4_status nvfp4_gemm_sqrelu_maxima(const nvfp4_qtensor* A, const nvfp4_qtensor* B, void* H, int64_t ldh,
                                                 uint64_t rht_seed, uint32_t* maxima, size_t maxima_bytes,
                                                 uint32_t* dev_status, void* stream) {
    return nvfp4::gemm_sqrelu_maxima_impl(A, B, H, ldh, rht_seed, maxima, maxima_bytes, dev_status,
                                          static_cast<cudaStream_t>(stream));
}

extern "C" nvfp4_status nvfp4_gemm_sqrelu_bwd(const nvfp4_qtensor* A, const nvfp4_qtensor* B, const void* H,
                                              int64_t ldh, void* D, int64_t ldd, uint32_t* dev_status,
                                              void* stream) {
    return nvfp4::gemm_sqrelu_bwd_impl(A, B, H, ldh, D, ldd, 0, nullptr, 0, dev_status,
                                       static_cast<cudaStream_t>(stream));
}

extern "C" nvfp4_status nvfp4_gemm_sqrelu_bwd_maxima(const nvfp4_qtensor* A, const nvfp4_qtensor* B, const void* H,
                                                     int64_t ldh, void* D, int64_t ldd, uint64_t rht_seed,
                                                     uint32_t* maxima, size_t maxima_bytes, uint32_t* dev_status,
                                                     void* stream) {
    if (!maxima) return NVFP4_ERR_INVALID_ARG;
    return nvfp4::gemm_sqrelu_bwd_impl(A, B, H, ldh, D, ldd, rht_seed, maxima, maxima_bytes, dev_status,
                                       static_cast<cudaStream_t>(stream));
}

extern "C" nvfp4_status nvfp4_mx_gemm(const nvfp4_qtensor* A, const nvfp4_qtensor* B, void* D, int32_t d_dtype,
                                      int64_t ldd, uint32_t* dev_status, void* stream) {
    return nvfp4::mx_gemm_impl(A, B, D, d_dtype, ldd, dev_status, static_cast<cudaStream_t>(stream));
}

// Test hook: 0 chooses the kernel automatically, 1 forces the single-CTA kernel,
// 2 forces the CTA-pair kernel where its epilogue applies (bf16, aligned output).
extern "C" void nvfp4_gemm_force_path(int32_t path) { nvfp4::gemm::g_force_path = (path >= 0 && path <= 2) ? path : 0; }

extern "C" nvfp4_status nvfp4_gemm(const nvfp4_qtensor* A, const nvfp4_qtensor* B, void* D, int32_t d_dtype,
                                   int64_t ldd, uint32_t* dev_status, void* stream) {
    return nvfp4::gemm_impl(A, B, D, d_dtype, ldd, dev_status, static_cast<cudaStream_t>(stream), nullptr, 0);
}

extern "C" size_t nvfp4_gemm_workspace_bytes(int32_t device) {
    const int sms = nvfp4::sm_count(device);
    return sms > 0 ? nvfp4::gemm::split_ws_bytes(sms) : 0u;
}

extern "C" nvfp4_status nvfp4_gemm_ws(const nvfp4_qtensor* A, const nvfp4_qtensor* B, void* D, int32_t d_dtype,
                                      int64_t ldd, void* workspace, size_t workspace_bytes, uint32_t* dev_status,
                                      void* stream) {
    return nvfp4::gemm_impl(A, B, D, d_dtype, ldd, dev_status, static_cast<cudaStream_t>(stream), workspace,
                            workspace_bytes);
}
