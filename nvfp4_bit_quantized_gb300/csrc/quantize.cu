// quantize.cu -- NVFP4 quantizers for sm_103a (HBM-bound, two passes).
//
// Pass 1 (amax): per-CTA partial maxima of |x| (of |RHT(x)| for the Wgrad
// operands), written to the workspace; no atomics, no memset.
// Pass 2 (encode): every CTA reduces the partials to the tensor amax (an
// order-free max, so every CTA gets the same value), derives s_enc, then
// encodes its blocks: block amax -> E4M3 scale -> E2M1 codes -> packed nibbles,
// canonical and tensor-core-layout scales.
//
// Method: news page "NVIDIA NVFP4 paper: 4-bit pretrain hits FP8 parity (12B,
// 10T tokens)", ¶2 (format, 2D weight blocks, RHT on Wgrad inputs, SR on
// gradients only).  Readings of what the page leaves open: include/nvfp4.h.
//
// Thread mappings (16-byte chunks = 8 bf16 or 4 fp32 values, VEC below):
//   row kernel  : a warp reads 32 consecutive chunks of one row (512 B, fully
//                 coalesced); a 16-element block spans 16/VEC lanes.
//   col / 16x16 : a thread owns a 16-row x VEC-column patch; lane = 8*rg + cc
//                 (rg: 4 row groups of 16, cc: 8 column chunks), so one warp
//                 covers 64 rows x 8*VEC columns; every load instruction reads
//                 4 full 128-byte lines, every transposed store writes full
//                 32-byte sectors (4 lanes x 8 bytes per output row).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <map>
#include <mutex>
#include <set>
#include <utility>

#include "device_common.cuh"
#include "host_common.h"

namespace nvfp4 {

constexpr int kThreads = 256;
constexpr int kMaxPartials = 4096;

// Byte offset of (row r, scale-column s) in the tensor-core scale layout.  32-bit
// arithmetic: the host rejects operands whose scale layout reaches 4 GB.
__device__ __forceinline__ uint32_t mma_sf_offset(int64_t r, int64_t s, int64_t nkb) {
    const uint32_t r32 = (uint32_t)r, s32 = (uint32_t)s;
    return ((((r32 >> 7) * (uint32_t)nkb + (s32 >> 4)) << 11) | (((s32 >> 2) & 3u) << 9) | ((r32 & 31u) << 4) |
            (((r32 >> 5) & 3u) << 2) | (s32 & 3u));
}

// Walks the sequence k = start, start + step, ... as (k / width, k % width) without a
// division per step (a 64-bit division costs tens of ALU instructions, which
// these ALU-bound kernels cannot afford per 16-byte chunk).
struct Walk2D {
    int64_t row, col;              // current position
    int64_t drow, dcol, width;     // step = drow * width + dcol, 0 <= dcol < width
    __device__ __forceinline__ Walk2D(int64_t start, int64_t step, int64_t w)
        : row(start / w), col(start % w), drow(step / w), dcol(step % w), width(w) {}
    __device__ __forceinline__ void advance() {
        row += drow;
        col += dcol;
        if (col >= width) { col -= width; ++row; }
    }
};

// ---------------------------------------------------------------------------
// Pass 1: amax
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t abs_bits_max(uint4 v, const uint16_t*) {
    uint32_t m = __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                          __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
    return max(m >> 16, m & 0xFFFFu) << 16;           // bf16 |x| as fp32 bits
}
__device__ __forceinline__ uint32_t abs_bits_max(uint4 v, const float*) {
    return max(max(v.x & 0x7FFFFFFFu, v.y & 0x7FFFFFFFu), max(v.z & 0x7FFFFFFFu, v.w & 0x7FFFFFFFu));
}

__device__ __forceinline__ uint4 sqrelu_bf16x8(uint4 v) {
    return make_uint4(sqrelu_bf16x2(v.x), sqrelu_bf16x2(v.y), sqrelu_bf16x2(v.z), sqrelu_bf16x2(v.w));
}
// Applies the load transform of a kernel (identity, or the squared ReLU for bf16).
template <typename T, bool SQR>
__device__ __forceinline__ uint4 pre16(uint4 v) {
    if constexpr (SQR && sizeof(T) == 2) return sqrelu_bf16x8(v);
    else return v;
}

__device__ __forceinline__ void block_max_store(uint32_t m, uint32_t* partials) {
    __shared__ uint32_t red[kThreads / 32];
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x < 32) {
        uint32_t v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0u;
        v = __reduce_max_sync(0xFFFFFFFFu, v);
        if (threadIdx.x == 0) partials[blockIdx.x] = v;
    }
}

// |x| max, unsigned compare of the magnitude bits (NaN sorts above Inf).
template <typename T, bool SQR = false>
__global__ void __launch_bounds__(kThreads) amax_kernel(const T* __restrict__ x, int64_t R, int64_t C,
                                                        int64_t ldx, uint32_t* __restrict__ partials) {
    pdl_launch_dependents();
    pdl_wait();
    constexpr int VEC = Vec<T>::N;
    const int lane = threadIdx.x & 31;
    const int64_t cpr = C / VEC;
    const int64_t spr = (cpr + 31) / 32;
    const int64_t nseg = R * spr;
    const int64_t warp0 = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    const int64_t nwarps = (int64_t)gridDim.x * (kThreads / 32);
    uint32_t m = 0;
    constexpr int U = 4;
    if (nseg == 0) { block_max_store(0u, partials); return; }
    Walk2D w(warp0, nwarps, spr);
    for (int64_t base = warp0; base < nseg; base += nwarps * U) {
        uint4 v[U];
        bool ok[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t seg = base + (int64_t)u * nwarps;
            ok[u] = false;
            if (seg < nseg) {
                const int64_t ch = w.col * 32 + lane;
                if (ch < cpr) {
                    v[u] = pre16<T, SQR>(ld_stream(x + w.row * ldx + ch * VEC));
                    ok[u] = true;
                }
            }
            w.advance();
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (ok[u]) m = max(m, abs_bits_max(v[u], (const T*)nullptr));
    }
    block_max_store(m, partials);
}

// |x| max over a contiguous tensor (row pitch == C) as one flat array of 16-byte
// chunks: no 2D index arithmetic per chunk.
template <typename T, bool SQR = false>
__global__ void __launch_bounds__(kThreads) amax_flat_kernel(const T* __restrict__ x, int64_t nchunks,
                                                             uint32_t* __restrict__ partials) {
    pdl_launch_dependents();
    pdl_wait();
    constexpr int VEC = Vec<T>::N;
    constexpr int U = 8;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    uint32_t m = 0;
    for (int64_t base = (int64_t)blockIdx.x * kThreads + threadIdx.x; base < nchunks; base += stride * U) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (base + u * stride < nchunks) v[u] = pre16<T, SQR>(ld_stream(x + (base + u * stride) * VEC));
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (base + u * stride < nchunks) m = max(m, abs_bits_max(v[u], (const T*)nullptr));
    }
    block_max_store(m, partials);
}

// max |v_i| of 16 values as a tree (short dependency chains).
__device__ __forceinline__ float abs_max16(const float (&v)[16]) {
    float a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = fmaxf(fabsf(v[2 * i]), fabsf(v[2 * i + 1]));
#pragma unroll
    for (int s = 4; s >= 1; s >>= 1)
#pragma unroll
        for (int i = 0; i < s; ++i) a[i] = fmaxf(a[i], a[i + s]);
    return a[0];
}

// max(|a|, |b|) of packed bf16 pairs (sign bits of the result unspecified).
__device__ __forceinline__ uint32_t max_abs_bf16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
// The larger |.| of a packed bf16 pair as fp32 bits.
__device__ __forceinline__ uint32_t bf16x2_abs_max_bits(uint32_t m) {
    m &= 0x7FFF7FFFu;
    return max(m << 16, m & 0xFFFF0000u);
}

// In-place transpose of an 8 x 8 matrix of nibbles held as 8 words (element (i, j) in
// nibble j of word i -> nibble i of word j): three rounds of block swaps (4 x 4, 2 x 2,
// 1 x 1), each a shift, a masked xor and two xors per word pair.
__device__ __forceinline__ void transpose_nibbles8(uint32_t (&w)[8]) {
    auto swap = [&](int a, int b, int k, uint32_t m) {
        const uint32_t t = ((w[a] >> k) ^ w[b]) & m;
        w[a] ^= t << k;
        w[b] ^= t;
    };
#pragma unroll
    for (int i = 0; i < 4; ++i) swap(i, i + 4, 16, 0x0000FFFFu);
    swap(0, 2, 8, 0x00FF00FFu); swap(1, 3, 8, 0x00FF00FFu); swap(4, 6, 8, 0x00FF00FFu); swap(5, 7, 8, 0x00FF00FFu);
#pragma unroll
    for (int i = 0; i < 8; i += 2) swap(i, i + 1, 4, 0x0F0F0F0Fu);
}

// ---- Patch pipeline.  The column and 16x16 kernels (and the RHT maxima) give each
// lane a 16-row x 16-byte patch of a warp's 64-row x (8 * 16 B) tile.  Their per-patch
// arithmetic is long and their register footprint leaves one CTA per SM, so each
// lane copies its next patch global -> shared memory with cp.async (no registers held)
// while it transforms the current one: two slots per lane, laid out [slot][row][lane]
// x 16 B so that reading a row back is one conflict-free 512-byte access per warp.
extern __shared__ __align__(16) uint8_t patch_smem[];
constexpr int kPatchSlotBytes = 16 * 32 * 16;
constexpr int kPatchThreads = 128;                                          // 4 warps per CTA
constexpr int kPatchCtasPerSm = 3;                                          // by registers (~140 / thread) and shared memory
constexpr int kPatchSmemBytes = (kPatchThreads / 32) * 2 * kPatchSlotBytes;   // 64 KB per CTA
// The maxima passes and the 16x16 encoder do little arithmetic per byte: two copies in flight per
// warp (three slots, 96 KB per CTA, two CTAs per SM) keep more bytes on the way than the row /
// column encoders' one (those are bound by their arithmetic and want the third CTA's warps).
constexpr int kAmaxAhead = 2;
constexpr int kAmaxCtasPerSm = 2;
constexpr int kAmaxSmemBytes = (kPatchThreads / 32) * (kAmaxAhead + 1) * kPatchSlotBytes;
constexpr int kBandGroup = 8;                                               // bands per tile group (power of 2)

template <typename T, int AHEAD = 1>
struct PatchPipe {
    static constexpr int VEC = Vec<T>::N;
    static constexpr int SLOTS = AHEAD + 1;         // the current patch + AHEAD copies in flight
    const T* x;
    int64_t ldx, R, C, tiles, nwarps;
    int64_t tile;                    // tile index of the current patch
    int64_t itile;                   // tile index of the next copy to issue
    Walk2D w;
    int rg, cc;
    uint32_t sbase;                  // shared address of this lane's slot 0, row 0
    uint32_t islot = 0, rslot = 0;   // slot of the next copy / of the current patch
    int64_t r0 = 0, c0 = 0;          // current patch
    bool ok = false;
    int64_t qr[AHEAD], qc[AHEAD];    // copies in flight, oldest first
    bool qok[AHEAD];
    uint32_t qslot[AHEAD];

    // Tile order: groups of kBandGroup 64-row bands, column-major inside a group, so
    // neighbouring warps (the warps of a CTA and of the next CTA) take vertically adjacent
    // tiles and their transposed outputs (32 bytes per output row each) land as whole
    // 128-byte lines and longer runs.  Tiles past the last band are skipped like any other
    // out-of-range patch.
    __device__ __forceinline__ PatchPipe(const T* x_, int64_t ldx_, int64_t R_, int64_t C_, int64_t warp0,
                                         int64_t nwarps_, int64_t /*tiles*/, int64_t tiles_c, uint8_t* smem)
        : x(x_), ldx(ldx_), R(R_), C(C_),
          tiles((((R_ + 63) / 64 + kBandGroup - 1) / kBandGroup) * kBandGroup * tiles_c), nwarps(nwarps_),
          tile(warp0), itile(warp0), w(warp0, nwarps_, kBandGroup * (tiles_c > 0 ? tiles_c : 1)) {
        const int lane = threadIdx.x & 31;
        rg = lane >> 3;
        cc = lane & 7;
        sbase = smem_addr(smem) + (uint32_t)((threadIdx.x >> 5) * SLOTS * kPatchSlotBytes + lane * 16);
#pragma unroll
        for (int k = 0; k < AHEAD; ++k) issue_next(k);
    }
    __device__ __forceinline__ static void commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
    // copies the patch at the walker's position (tile itile) into the next slot as queue entry k
    // (one commit group, empty past the last tile), then steps the walker
    __device__ __forceinline__ void issue_next(int k) {
        qslot[k] = islot;
        qok[k] = false;
        qr[k] = 0;
        qc[k] = 0;
        if (itile < tiles) {
            const int64_t nr = (w.row * kBandGroup + (w.col & (kBandGroup - 1))) * 64 + rg * 16;
            const int64_t nc = (w.col / kBandGroup) * (8 * VEC) + cc * VEC;
            qr[k] = nr;
            qc[k] = nc;
            qok[k] = nr < R && nc < C;
            if (qok[k]) {
                const char* src = reinterpret_cast<const char*>(x + nr * ldx + nc);
                const int64_t pitch = ldx * (int64_t)sizeof(T);
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                                 :: "r"(sbase + islot * kPatchSlotBytes + i * 512), "l"(src + i * pitch) : "memory");
            }
        }
        commit();
        w.advance();
        itile += nwarps;
        islot = islot + 1 == SLOTS ? 0u : islot + 1;
    }
    // Makes the next patch of this warp current (r0, c0, ok) and starts the copy AHEAD patches
    // after it; false when the warp has no patch left.
    __device__ __forceinline__ bool next() {
        if (tile >= tiles) return false;
        r0 = qr[0];
        c0 = qc[0];
        ok = qok[0];
        rslot = qslot[0];
#pragma unroll
        for (int k = 0; k + 1 < AHEAD; ++k) {
            qr[k] = qr[k + 1];
            qc[k] = qc[k + 1];
            qok[k] = qok[k + 1];
            qslot[k] = qslot[k + 1];
        }
        issue_next(AHEAD - 1);
        tile += nwarps;
        asm volatile("cp.async.wait_group %0;" :: "n"(AHEAD) : "memory");   // the current patch has landed
        return true;
    }
    __device__ __forceinline__ uint4 read_row(int i) const {
        uint4 r;
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                     : "r"(sbase + rslot * kPatchSlotBytes + i * 512) : "memory");
        return r;
    }
    __device__ __forceinline__ void read(uint4 (&v)[16]) const {
#pragma unroll
        for (int i = 0; i < 16; ++i)
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v[i].x), "=r"(v[i].y), "=r"(v[i].z), "=r"(v[i].w)
                         : "r"(sbase + rslot * kPatchSlotBytes + i * 512) : "memory");
    }
};

// Unpacks a patch into t[col][row] as fp32.
template <typename T>
__device__ __forceinline__ void unpack_patch(const uint4 (&v)[16], float (&t)[Vec<T>::N][16]) {
    constexpr int VEC = Vec<T>::N;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        float f[VEC];
        Vec<T>::unpack(v[i], f);
#pragma unroll
        for (int j = 0; j < VEC; ++j) t[j][i] = f[j];
    }
}

// ---- bf16 patches: 16 rows x 8 columns per thread, kept as column pairs so the
// transform and the scaling use packed two-wide fp32 instructions.

// max(|m|, |v|), NaN propagating (the sign bit of the result is unspecified).
__device__ __forceinline__ float max_abs_nan(float m, float v) {
    float r;
    asm("max.NaN.xorsign.abs.f32 %0, %1, %2;" : "=f"(r) : "f"(m), "f"(v));
    return r;
}
__device__ __forceinline__ uint32_t max_abs_nan_bf16x2(uint32_t m, uint32_t v) {
    uint32_t r;
    asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(m), "r"(v));
    return r;
}

// Unpacks a bf16 patch as t[k][i] = (x[r0+i][c0+2k], x[r0+i][c0+2k+1]), negating row i
// where bit i of `neg` is set (the RHT signs).  With PLAIN, returns the packed bf16 |x|
// maximum of the patch (NaN propagating), else 0.
template <bool PLAIN>
__device__ __forceinline__ uint32_t unpack_patch_bf16(const uint4 (&v)[16], uint32_t neg, float2 (&t)[4][16]) {
    uint32_t m = 0u;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t s = ((neg >> i) & 1u) ? 0x80008000u : 0u;
        const uint32_t w[4] = {v[i].x ^ s, v[i].y ^ s, v[i].z ^ s, v[i].w ^ s};
        if (PLAIN) m = max_abs_nan_bf16x2(m, max_abs_nan_bf16x2(max_abs_nan_bf16x2(w[0], w[1]),
                                                                max_abs_nan_bf16x2(w[2], w[3])));
#pragma unroll
        for (int k = 0; k < 4; ++k) t[k][i] = make_float2(bf16_lo(w[k]), bf16_hi(w[k]));
    }
    return m;
}

// |.| maxima of the two columns of a pair (NaN propagating), as a tree for ILP.
__device__ __forceinline__ void col_pair_abs_max(const float2 (&t)[16], float& m0, float& m1) {
    float a[8], b[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) { a[i] = max_abs_nan(t[2 * i].x, t[2 * i + 1].x); b[i] = max_abs_nan(t[2 * i].y, t[2 * i + 1].y); }
#pragma unroll
    for (int s = 4; s >= 1; s >>= 1)
#pragma unroll
        for (int i = 0; i < s; ++i) { a[i] = max_abs_nan(a[i], a[i + s]); b[i] = max_abs_nan(b[i], b[i + s]); }
    m0 = a[0];
    m1 = b[0];
}

// For bf16 inputs every RHT intermediate is a multiple of 2^-133 (the bf16 quantum), so
// multiplying by 1/4 is exact; the quarter is folded into the block and tensor maxima
// (max|t/4| = max|t| / 4) and into the element multiplier (t * (e_b / 4) == (t / 4) * e_b
// whenever e_b / 4 is exact, i.e. e_b >= 2^-124; the smallest e_b of a tensor belongs to the
// largest scale code 126, so one check per CTA decides).

// amax of RHT(x) along rows: the Wgrad operands' tensor amax after the transform.
template <typename T>
__global__ void __launch_bounds__(kPatchThreads, kAmaxCtasPerSm) amax_rht_kernel(const T* __restrict__ x, int64_t R, int64_t C,
                                                            int64_t ldx, uint64_t rht_seed,
                                                            uint32_t* __restrict__ partials) {
    pdl_launch_dependents();
    pdl_wait();
    constexpr int VEC = Vec<T>::N;
    const int64_t tiles_c = (C + 8 * VEC - 1) / (8 * VEC);
    const int64_t tiles = ((R + 63) / 64) * tiles_c;
    const int64_t warp0 = (int64_t)blockIdx.x * (kPatchThreads / 32) + (threadIdx.x >> 5);
    const int64_t nwarps = (int64_t)gridDim.x * (kPatchThreads / 32);
    const uint32_t sign_mask = rht_sign_mask(rht_seed);
    if constexpr (sizeof(T) == 2) {
        float m = 0.0f;
        PatchPipe<T, kAmaxAhead> pp(x, ldx, R, C, warp0, nwarps, tiles, tiles_c, patch_smem);
        while (pp.next()) {
            if (!pp.ok) continue;
            const int64_t r0 = pp.r0, c0 = pp.c0;
            uint4 v[16];
            pp.read(v);
            float2 t[4][16];
            unpack_patch_bf16<false>(v, sign_mask, t);
            float pm[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                hadamard16_x2(t[k]);
                float m0, m1;
                col_pair_abs_max(t[k], m0, m1);
                pm[k] = max_abs_nan(m0, m1);
            }
            m = max_abs_nan(m, max_abs_nan(max_abs_nan(pm[0], pm[1]), max_abs_nan(pm[2], pm[3])));
        }
        block_max_store(__float_as_uint(__fmul_rn(fabsf(m), 0.25f)) & 0x7FFFFFFFu, partials);
        return;
    }
    float m = 0.0f;
    bool bad = false;                                // NaN: fmaxf would drop it
    PatchPipe<T, kAmaxAhead> pp(x, ldx, R, C, warp0, nwarps, tiles, tiles_c, patch_smem);
    while (pp.next()) {
        if (!pp.ok) continue;
        const int64_t r0 = pp.r0, c0 = pp.c0;
        uint4 v[16];
        pp.read(v);
        float t[VEC][16];
        unpack_patch<T>(v, t);
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            rht16(t[j], sign_mask);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float a = fabsf(t[j][i]);
                m = fmaxf(m, a);
                bad |= !(a <= FLT_MAX);
            }
        }
    }
    block_max_store(bad ? 0x7FC00000u : __float_as_uint(m), partials);
}

// Both tensor amaxes of a dual quantization in one read: |x| (row operand) and
// |RHT(x)| along rows (column operand).
template <typename T, bool SQR = false>
__global__ void __launch_bounds__(kPatchThreads, kAmaxCtasPerSm) amax_dual_kernel(const T* __restrict__ x, int64_t R, int64_t C,
                                                             int64_t ldx, uint64_t rht_seed,
                                                             uint32_t* __restrict__ partials_plain,
                                                             uint32_t* __restrict__ partials_rht) {
    pdl_launch_dependents();
    pdl_wait();
    constexpr int VEC = Vec<T>::N;
    const int64_t tiles_c = (C + 8 * VEC - 1) / (8 * VEC);
    const int64_t tiles = ((R + 63) / 64) * tiles_c;
    const int64_t warp0 = (int64_t)blockIdx.x * (kPatchThreads / 32) + (threadIdx.x >> 5);
    const int64_t nwarps = (int64_t)gridDim.x * (kPatchThreads / 32);
    const uint32_t sign_mask = rht_sign_mask(rht_seed);
    float mp = 0.0f, mr = 0.0f;
    bool bad = false;
    if constexpr (sizeof(T) == 2) {
        uint32_t mpk = 0u;                           // packed bf16 |x| maxima
        PatchPipe<T, kAmaxAhead> pp(x, ldx, R, C, warp0, nwarps, tiles, tiles_c, patch_smem);
        while (pp.next()) {
            if (!pp.ok) continue;
            const int64_t r0 = pp.r0, c0 = pp.c0;
            uint4 v[16];
            pp.read(v);
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = pre16<T, SQR>(v[i]);
            float2 t[4][16];
            mpk = max_abs_nan_bf16x2(mpk, unpack_patch_bf16<true>(v, sign_mask, t));
            float pm[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                hadamard16_x2(t[k]);
                float m0, m1;
                col_pair_abs_max(t[k], m0, m1);
                pm[k] = max_abs_nan(m0, m1);
            }
            mr = max_abs_nan(mr, max_abs_nan(max_abs_nan(pm[0], pm[1]), max_abs_nan(pm[2], pm[3])));
        }
        mp = __uint_as_float(bf16x2_abs_max_bits(mpk));
        mr = __uint_as_float(__float_as_uint(__fmul_rn(fabsf(mr), 0.25f)) & 0x7FFFFFFFu);
    } else {
    PatchPipe<T, kAmaxAhead> pp(x, ldx, R, C, warp0, nwarps, tiles, tiles_c, patch_smem);
    while (pp.next()) {
        if (!pp.ok) continue;
        const int64_t r0 = pp.r0, c0 = pp.c0;
        uint4 v[16];
        pp.read(v);
        float t[VEC][16];
        unpack_patch<T>(v, t);
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float a = fabsf(t[j][i]);
                mp = fmaxf(mp, a);
                bad |= !(a <= FLT_MAX);
            }
            rht16(t[j], sign_mask);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float a = fabsf(t[j][i]);
                mr = fmaxf(mr, a);
                bad |= !(a <= FLT_MAX);
            }
        }
    }
    }
    __shared__ uint32_t red[2][kThreads / 32];
    uint32_t vp = bad ? 0x7FC00000u : __float_as_uint(mp);
    uint32_t vr = bad ? 0x7FC00000u : __float_as_uint(mr);
    vp = __reduce_max_sync(0xFFFFFFFFu, vp);
    vr = __reduce_max_sync(0xFFFFFFFFu, vr);
    if ((threadIdx.x & 31) == 0) { red[0][threadIdx.x >> 5] = vp; red[1][threadIdx.x >> 5] = vr; }
    __syncthreads();
    if (threadIdx.x < 32) {
        uint32_t a = threadIdx.x < (blockDim.x >> 5) ? red[0][threadIdx.x] : 0u;
        uint32_t b = threadIdx.x < (blockDim.x >> 5) ? red[1][threadIdx.x] : 0u;
        a = __reduce_max_sync(0xFFFFFFFFu, a);
        b = __reduce_max_sync(0xFFFFFFFFu, b);
        if (threadIdx.x == 0) { partials_plain[blockIdx.x] = a; partials_rht[blockIdx.x] = b; }
    }
}

// ---------------------------------------------------------------------------
// Pass 2 prologue: reduce the partials to s_enc (same value in every CTA).
// ---------------------------------------------------------------------------
struct Scales { float s_enc; bool finite; };

// Per-CTA table of the element multiplier e_b = s_enc / S_b for every non-negative
// E4M3 scale code (one division per code instead of one per block).
__shared__ float g_eb_table[128];

__device__ __forceinline__ Scales tensor_scales(const uint32_t* __restrict__ partials, int nparts,
                                                float* s_dec_out, uint32_t* dev_status, float* table = g_eb_table) {
    __shared__ uint32_t red[kThreads / 32];
    __shared__ uint32_t total;
    uint32_t m = 0;
    for (int i = threadIdx.x; i < nparts; i += blockDim.x) m = max(m, partials[i]);
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x < 32) {
        uint32_t v = threadIdx.x < (blockDim.x / 32) ? red[threadIdx.x] : 0u;
        v = __reduce_max_sync(0xFFFFFFFFu, v);
        if (threadIdx.x == 0) total = v;
    }
    __syncthreads();
    const uint32_t bits = total;
    Scales s;
    s.finite = bits < 0x7F800000u;
    const float amax_t = s.finite ? __uint_as_float(bits) : 0.0f;
    s.s_enc = tensor_s_enc(amax_t);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        *s_dec_out = __fdiv_rn(1.0f, s.s_enc);
        if (!s.finite) set_status(dev_status, NVFP4_ERR_NONFINITE);
    }
    if (threadIdx.x < 128) table[threadIdx.x] = block_multiplier(threadIdx.x, s.s_enc);
    __syncthreads();
    return s;
}

struct QOut {
    uint8_t* codes;
    uint8_t* scales;
    uint8_t* scales_mma;
    uint8_t* codes_t;
    uint8_t* scales_mma_t;
    float* s_dec;
};

// ---------------------------------------------------------------------------
// Pass 2, 1x16 blocks along rows.  One 16-element block per lane (a warp covers 32
// consecutive blocks of one row: 1 KB of bf16, fully coalesced), so the block amax,
// the scale and its stores need no cross-lane traffic.  U warp segments per
// iteration issue all their loads before any is used.
// ---------------------------------------------------------------------------
template <typename T> struct Block16;
template <> struct Block16<uint16_t> {            // 32 bytes
    static constexpr int WORDS = 8;
    __device__ __forceinline__ static void load(const uint16_t* p, bool v8, uint32_t (&w)[8]) {
        if (v8) {
            ld_stream32(p, w);
        } else {
            const uint4 a = ld_stream(p), b = ld_stream(p + 8);
            w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
        }
    }
    __device__ __forceinline__ static void unpack(const uint32_t (&w)[8], float (&f)[16]) {
#pragma unroll
        for (int i = 0; i < 8; ++i) { f[2 * i] = bf16_lo(w[i]); f[2 * i + 1] = bf16_hi(w[i]); }
    }
};
template <> struct Block16<float> {               // 64 bytes
    static constexpr int WORDS = 16;
    __device__ __forceinline__ static void load(const float* p, bool v8, uint32_t (&w)[16]) {
        if (v8) {
            uint32_t a[8], b[8];
            ld_stream32(p, a);
            ld_stream32(p + 8, b);
#pragma unroll
            for (int i = 0; i < 8; ++i) { w[i] = a[i]; w[8 + i] = b[i]; }
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 a = ld_stream(p + 4 * q);
                w[4 * q] = a.x; w[4 * q + 1] = a.y; w[4 * q + 2] = a.z; w[4 * q + 3] = a.w;
            }
        }
    }
    __device__ __forceinline__ static void unpack(const uint32_t (&w)[16], float (&f)[16]) {
#pragma unroll
        for (int i = 0; i < 16; ++i) f[i] = __uint_as_float(w[i]);
    }
};

// Where one row block's results go: its 8 code bytes, its scale in the canonical and in
// the tensor-core layout (either may be null), and its Philox group (element index / 16).
struct RowDst {
    uint8_t* codes;
    uint8_t* scale;
    uint8_t* scale_mma;
    uint64_t group;
};
__device__ __forceinline__ RowDst row_dst(const QOut& out, int64_t r, int64_t col, int64_t C, int64_t nkb) {
    RowDst d;
    d.codes = out.codes + r * (C / 2) + col / 2;
    d.scale = out.scales ? out.scales + r * (C / 16) + col / 16 : nullptr;
    d.scale_mma = out.scales_mma ? out.scales_mma + mma_sf_offset(r, col / 16, nkb) : nullptr;
    d.group = (uint64_t)(r * C + col) >> 4;                  // C % 16 == 0
    return d;
}

// One 1x16 row block of bf16 x (as eight packed words): the block scale, the sixteen
// codes and their stores.
template <bool SR>
__device__ __forceinline__ void encode_row_block_bf16(const uint32_t (&w)[8], const RowDst& d, float s_enc,
                                                      const float* eb_table, const PhiloxKey& key, uint32_t sr_offset) {
    const uint32_t m = max_abs_bf16x2(max_abs_bf16x2(max_abs_bf16x2(w[0], w[1]), max_abs_bf16x2(w[2], w[3])),
                                      max_abs_bf16x2(max_abs_bf16x2(w[4], w[5]), max_abs_bf16x2(w[6], w[7])));
    const uint32_t sb = block_scale_code_bf16(__uint_as_float(bf16x2_abs_max_bits(m)), s_enc);
    const float2 eb = make_float2(eb_table[sb], eb_table[sb]);
    float y[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float2 v = __fmul2_rn(make_float2(bf16_lo(w[j]), bf16_hi(w[j])), eb);
        y[2 * j] = v.x;
        y[2 * j + 1] = v.y;
    }
    uint2 codes;
    if constexpr (SR) {
        const Philox4 p = sr_philox(key, 0u, sr_offset, d.group);
        codes = e2m1x16_sr(y, p.w);
    } else {
        codes = e2m1x16_rn(y);
    }
    *reinterpret_cast<uint2*>(d.codes) = codes;
    if (d.scale) *d.scale = (uint8_t)sb;
    if (d.scale_mma) *d.scale_mma = (uint8_t)sb;
}

template <typename T, bool SR, bool SQR = false>
__global__ void __launch_bounds__(kThreads) encode_row_kernel(const T* __restrict__ x, int64_t R, int64_t C,
                                                              int64_t ldx, const uint32_t* __restrict__ partials,
                                                              int nparts, QOut out, const PhiloxKey sr_key,
                                                              uint32_t sr_offset, int v8, uint32_t* dev_status) {
    pdl_launch_dependents();
    pdl_wait();
    using B = Block16<T>;
    const Scales sc = tensor_scales(partials, nparts, out.s_dec, dev_status);
    const PhiloxKey& key = sr_key;
    const int lane = threadIdx.x & 31;
    const int64_t bpr = C / 16;                      // blocks per row
    const int64_t spr = (bpr + 31) / 32;             // warp segments per row
    const int64_t nseg = R * spr;
    const int64_t nkb = (C + 255) / 256;
    const int64_t warp0 = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    const int64_t nwarps = (int64_t)gridDim.x * (kThreads / 32);
    if (warp0 >= nseg) return;
    // One warp segment at a time, two buffers: the next segment's load is in flight
    // while the current one is encoded.
    Walk2D w(warp0, nwarps, spr);
    auto fetch = [&](int64_t seg, uint32_t (&buf)[B::WORDS], int64_t& r, int64_t& bk) -> bool {
        r = w.row;
        bk = w.col * 32 + lane;
        w.advance();
        const bool ok = seg < nseg && bk < bpr;
        if (ok) B::load(x + r * ldx + bk * 16, v8 != 0, buf);
        return ok;
    };
    auto encode = [&](uint32_t (&raw)[B::WORDS], int64_t r, int64_t bk) {
        if constexpr (sizeof(T) == 2) {
            if constexpr (SQR) {
#pragma unroll
                for (int i = 0; i < B::WORDS; ++i) raw[i] = sqrelu_bf16x2(raw[i]);
            }
            encode_row_block_bf16<SR>(raw, row_dst(out, r, bk * 16, C, nkb), sc.s_enc, g_eb_table, key, sr_offset);
            return;
        }
        float f[16];
        B::unpack(raw, f);
        const uint32_t sb = block_scale_code(abs_max16(f), sc.s_enc);
        const float2 eb = make_float2(g_eb_table[sb], g_eb_table[sb]);
        float y[16];
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
            const float2 v = __fmul2_rn(make_float2(f[j], f[j + 1]), eb);
            y[j] = v.x;
            y[j + 1] = v.y;
        }
        const int64_t col = bk * 16;
        uint2 codes;
        if constexpr (SR) {
            const Philox4 p = sr_philox(key, 0u, sr_offset, (uint64_t)(r * C + col) >> 4);   // C % 16 == 0
            codes = e2m1x16_sr(y, p.w);
        } else {
            codes = e2m1x16_rn(y);
        }
        *reinterpret_cast<uint2*>(out.codes + r * (C / 2) + col / 2) = codes;
        if (out.scales) out.scales[r * bpr + bk] = (uint8_t)sb;
        if (out.scales_mma) out.scales_mma[mma_sf_offset(r, bk, nkb)] = (uint8_t)sb;
    };
    uint32_t bufa[B::WORDS], bufb[B::WORDS];
    int64_t ra, ka, rb, kb;
    bool oka = fetch(warp0, bufa, ra, ka), okb;
    for (int64_t seg = warp0; seg < nseg; seg += 2 * nwarps) {
        okb = fetch(seg + nwarps, bufb, rb, kb);
        if (oka) encode(bufa, ra, ka);
        if (seg + nwarps >= nseg) break;
        oka = fetch(seg + 2 * nwarps, bufa, ra, ka);
        if (okb) encode(bufb, rb, kb);
    }
}

// Column operand (x^T: 1x16 blocks along the rows of x, the RHT along the same rows)
// of one bf16 patch at (r0, c0): two columns at a time with packed arithmetic.
template <bool SR, bool RHT>
__device__ __forceinline__ void encode_col_patch_bf16(const uint4 (&v)[16], int64_t r0, int64_t c0, int64_t R,
                                                      uint32_t sign_mask, bool fold, const float* eb_table,
                                                      float s_enc, const PhiloxKey& key, uint32_t sr_offset,
                                                      const QOut& out, int64_t nkb) {
    const float quarter = RHT ? 0.25f : 1.0f;
    float2 t[4][16];
    unpack_patch_bf16<false>(v, sign_mask, t);
    // Operand rows c0 + j (j < 8): codes R/2 bytes apart, canonical scales R/16 apart,
    // Philox groups R/16 apart (R % 16 == 0, r0 % 16 == 0), tensor-core scales 16 bytes
    // apart (c0 % 8 == 0 keeps c0 + j inside one group of 32 operand rows).
    const int64_t hr = R / 2, sr = R / 16;
    uint8_t* cdst = out.codes + c0 * hr + r0 / 2;
    uint8_t* sdst = out.scales ? out.scales + c0 * sr + r0 / 16 : nullptr;
    uint8_t* mdst = out.scales_mma ? out.scales_mma + mma_sf_offset(c0, r0 / 16, nkb) : nullptr;
    uint64_t grp = (uint64_t)(c0 * sr + r0 / 16);
#pragma unroll
    for (int k = 0; k < 4; ++k) {                    // operand rows c0 + 2k, c0 + 2k + 1
        if constexpr (RHT) hadamard16_x2(t[k]);
        float m0, m1;
        col_pair_abs_max(t[k], m0, m1);
        const uint32_t sb0 = block_scale_code(__fmul_rn(fabsf(m0), quarter), s_enc);
        const uint32_t sb1 = block_scale_code(__fmul_rn(fabsf(m1), quarter), s_enc);
        float2 eb = make_float2(eb_table[sb0], eb_table[sb1]);
        if (fold) eb = __fmul2_rn(eb, make_float2(quarter, quarter));
        float y0[16], y1[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float2 u = t[k][i];
            if (!fold) u = __fmul2_rn(u, make_float2(0.25f, 0.25f));
            u = __fmul2_rn(u, eb);
            y0[i] = u.x;
            y1[i] = u.y;
        }
        uint2 codes0, codes1;
        if constexpr (SR) {
            const Philox4 p0 = sr_philox(key, 1u, sr_offset, grp);
            const Philox4 p1 = sr_philox(key, 1u, sr_offset, grp + (uint64_t)sr);
            codes0 = e2m1x16_sr(y0, p0.w);
            codes1 = e2m1x16_sr(y1, p1.w);
        } else {
            codes0 = e2m1x16_rn(y0);
            codes1 = e2m1x16_rn(y1);
        }
        *reinterpret_cast<uint2*>(cdst) = codes0;
        *reinterpret_cast<uint2*>(cdst + hr) = codes1;
        if (sdst) {
            sdst[0] = (uint8_t)sb0;
            sdst[sr] = (uint8_t)sb1;
            sdst += 2 * sr;
        }
        if (mdst) {
            mdst[0] = (uint8_t)sb0;
            mdst[16] = (uint8_t)sb1;
            mdst += 32;
        }
        cdst += 2 * hr;
        grp += 2 * (uint64_t)sr;
    }
}

// ---------------------------------------------------------------------------
// Pass 2, 1x16 blocks along columns (operand x^T), optional RHT along rows.
// ---------------------------------------------------------------------------
template <typename T, bool SR, bool RHT, bool SQR = false>
__global__ void __launch_bounds__(kPatchThreads, kPatchCtasPerSm) encode_col_kernel(const T* __restrict__ x, int64_t R, int64_t C,
                                                              int64_t ldx, const uint32_t* __restrict__ partials,
                                                              int nparts, QOut out, const PhiloxKey sr_key,
                                                              uint32_t sr_offset, uint64_t rht_seed,
                                                              uint32_t* dev_status) {
    pdl_launch_dependents();
    pdl_wait();
    constexpr int VEC = Vec<T>::N;
    const uint32_t sign_mask = RHT ? rht_sign_mask(rht_seed) : 0u;
    const Scales sc = tensor_scales(partials, nparts, out.s_dec, dev_status);
    const PhiloxKey& key = sr_key;
    const int64_t tiles_c = (C + 8 * VEC - 1) / (8 * VEC);
    const int64_t tiles = ((R + 63) / 64) * tiles_c;
    const int64_t nkb = (R + 255) / 256;             // operand cols = R
    const int64_t warp0 = (int64_t)blockIdx.x * (kPatchThreads / 32) + (threadIdx.x >> 5);
    const int64_t nwarps = (int64_t)gridDim.x * (kPatchThreads / 32);
    if constexpr (sizeof(T) == 2) {
        // the quarter of the transform folds into e_b when the smallest e_b (code 126) stays exact
        const bool fold = !RHT || __fmul_rn(g_eb_table[126], 0.25f) >= FLT_MIN;
        PatchPipe<T> pp(x, ldx, R, C, warp0, nwarps, tiles, tiles_c, patch_smem);
        while (pp.next()) {
            if (!pp.ok) continue;
            uint4 v[16];
            pp.read(v);
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = pre16<T, SQR>(v[i]);
            encode_col_patch_bf16<SR, RHT>(v, pp.r0, pp.c0, R, sign_mask, fold, g_eb_table, sc.s_enc, key, sr_offset,
                                           out, nkb);
        }
        return;
    }
    PatchPipe<T> pp(x, ldx, R, C, warp0, nwarps, tiles, tiles_c, patch_smem);
    while (pp.next()) {
        if (!pp.ok) continue;
        const int64_t r0 = pp.r0, c0 = pp.c0;
        uint4 v[16];
        pp.read(v);
        float t[VEC][16];
        unpack_patch<T>(v, t);
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            if constexpr (RHT) rht16(t[j], sign_mask);
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(t[j][i]));
            const uint32_t sb = block_scale_code(amax, sc.s_enc);
            const float e_b = g_eb_table[sb];
            const int64_t c = c0 + j;                // operand row
            const float2 eb = make_float2(e_b, e_b);
            float y[16];
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
                const float2 v = __fmul2_rn(make_float2(t[j][i], t[j][i + 1]), eb);
                y[i] = v.x;
                y[i + 1] = v.y;
            }
            uint2 codes;
            if constexpr (SR) {
                const Philox4 p = sr_philox(key, 1u, sr_offset, (uint64_t)(c * R + r0) >> 4);   // r0 % 16 == 0
                codes = e2m1x16_sr(y, p.w);
            } else {
                codes = e2m1x16_rn(y);
            }
            *reinterpret_cast<uint2*>(out.codes + c * (R / 2) + r0 / 2) = codes;
            const int64_t s = r0 / 16;
            if (out.scales) out.scales[c * (R / 16) + s] = (uint8_t)sb;
            if (out.scales_mma) out.scales_mma[mma_sf_offset(c, s, nkb)] = (uint8_t)sb;
        }
    }
}

// ---------------------------------------------------------------------------
// Pass 2 of a dual quantization of bf16 x (the row operand, and the column operand
// with the RHT along rows) in one read of x.  Each patch, once in shared memory, is
// encoded as the column operand exactly as encode_col_kernel does, then as the row
// operand: lanes 2j and 2j + 1 hold the two 8-column halves of the same 16-column
// blocks of 16 rows, so lane 2j + h takes rows 8h .. 8h + 7 of those blocks and reads
// both halves back from the pair's slots.  Per element the arithmetic is that of the
// two single-operand kernels.
// ---------------------------------------------------------------------------
template <bool SR, bool SQR>
__global__ void __launch_bounds__(kPatchThreads, kPatchCtasPerSm) encode_dual_kernel(
    const uint16_t* __restrict__ x, int64_t R, int64_t C, int64_t ldx, const uint32_t* __restrict__ part_row,
    const uint32_t* __restrict__ part_col, int nparts, QOut out_row, QOut out_col, const PhiloxKey key_row,
    const PhiloxKey key_col, uint32_t off_row, uint32_t off_col, uint64_t rht_seed, uint32_t* dev_status) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ float eb_row[128];
    const uint32_t sign_mask = rht_sign_mask(rht_seed);
    const Scales s_row = tensor_scales(part_row, nparts, out_row.s_dec, dev_status, eb_row);
    const Scales s_col = tensor_scales(part_col, nparts, out_col.s_dec, dev_status);
    const int64_t tiles_c = (C + 63) / 64;
    const int64_t tiles = ((R + 63) / 64) * tiles_c;
    const int64_t nkb_col = (R + 255) / 256, nkb_row = (C + 255) / 256;
    const int lane = threadIdx.x & 31, half = lane & 1;
    const int warp = threadIdx.x >> 5;
    const int64_t warp0 = (int64_t)blockIdx.x * (kPatchThreads / 32) + warp;
    const int64_t nwarps = (int64_t)gridDim.x * (kPatchThreads / 32);
    const bool fold = __fmul_rn(g_eb_table[126], 0.25f) >= FLT_MIN;
    // this lane pair's two 16-byte chunks of a row, slot 0
    const uint32_t pair_base = smem_addr(patch_smem) + (uint32_t)(warp * 2 * kPatchSlotBytes + (lane & ~1) * 16);
    PatchPipe<uint16_t> pp(x, ldx, R, C, warp0, nwarps, tiles, tiles_c, patch_smem);
    while (pp.next()) {
        __syncwarp();                                // the partner lane's copy has landed too
        if (pp.ok) {
            {
                uint4 v[16];
                pp.read(v);
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = pre16<uint16_t, SQR>(v[i]);
                encode_col_patch_bf16<SR, true>(v, pp.r0, pp.c0, R, sign_mask, fold, g_eb_table, s_col.s_enc, key_col,
                                                off_col, out_col, nkb_col);
            }
            // rows r0 + 8h + i: the tensor-core scale offset steps by 16 per row (no carry out
            // of the row's low five bits, as r0 % 16 == 0 and 8h + i < 16)
            RowDst d = row_dst(out_row, pp.r0 + half * 8, pp.c0 & ~(int64_t)15, C, nkb_row);
            const uint32_t base = pair_base + pp.rslot * kPatchSlotBytes + (uint32_t)(half * 8 * 512);
#pragma unroll 2
            for (int i = 0; i < 8; ++i) {
                uint32_t w[8];
                asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%8];\n\t"
                             "ld.shared.v4.u32 {%4, %5, %6, %7}, [%8+16];"
                             : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
                             : "r"(base + i * 512) : "memory");
                if constexpr (SQR) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) w[k] = sqrelu_bf16x2(w[k]);
                }
                encode_row_block_bf16<SR>(w, d, s_row.s_enc, eb_row, key_row, off_row);
                d.codes += C / 2;
                if (d.scale) d.scale += C / 16;
                if (d.scale_mma) d.scale_mma += 16;
                d.group += (uint64_t)(C / 16);
            }
        }
        __syncwarp();                                // done with the partner's slot before it is refilled
    }
}

// ---------------------------------------------------------------------------
// Pass 2, 16x16 tiles (weights): writes W and W^T codes from one tile scale.
// ---------------------------------------------------------------------------
template <typename T, bool SR>
__global__ void __launch_bounds__(kPatchThreads, kAmaxCtasPerSm) encode_2d_kernel(const T* __restrict__ x, int64_t R, int64_t C,
                                                             int64_t ldx, const uint32_t* __restrict__ partials,
                                                             int nparts, QOut out, const PhiloxKey sr_key,
                                                             uint32_t sr_offset, uint32_t* dev_status) {
    pdl_launch_dependents();
    pdl_wait();
    constexpr int VEC = Vec<T>::N;
    constexpr int LPT = 16 / VEC;                    // lanes per 16-column tile
    const Scales sc = tensor_scales(partials, nparts, out.s_dec, dev_status);
    const PhiloxKey& key = sr_key;
    const int lane = threadIdx.x & 31, cc = lane & 7;
    const int64_t tiles_c = (C + 8 * VEC - 1) / (8 * VEC);
    const int64_t tiles = ((R + 63) / 64) * tiles_c;
    const int64_t nkb = (C + 255) / 256, nkb_t = (R + 255) / 256;
    const int64_t warp0 = (int64_t)blockIdx.x * (kPatchThreads / 32) + (threadIdx.x >> 5);
    const int64_t nwarps = (int64_t)gridDim.x * (kPatchThreads / 32);
    PatchPipe<T, kAmaxAhead> pp(x, ldx, R, C, warp0, nwarps, tiles, tiles_c, patch_smem);
    if constexpr (sizeof(T) == 2) {
        // bf16: tile maxima on the packed words, then row by row from shared memory; the
        // W^T codes come from two 8 x 8 nibble transposes of the 16 row words.
        while (pp.next()) {
            const int64_t r0 = pp.r0, c0 = pp.c0;
            uint32_t am = 0u;                        // every lane takes part in the shuffle
            if (pp.ok) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const uint4 q = pp.read_row(i);
                    am = max_abs_bf16x2(am, max_abs_bf16x2(max_abs_bf16x2(q.x, q.y), max_abs_bf16x2(q.z, q.w)));
                }
            }
            float amax = __uint_as_float(bf16x2_abs_max_bits(am));
            amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));      // the tile's other 8 columns
            const bool ok = pp.ok;
            uint32_t sb = 0u;                        // lanes without a patch: 0, the padding value
            if (ok) {
                sb = block_scale_code_bf16(amax, sc.s_enc);
                const float2 eb = make_float2(g_eb_table[sb], g_eb_table[sb]);
                uint32_t lo[8], hi[8];                   // row words: rows 0-7, 8-15
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const uint4 q = pp.read_row(i);
                    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
                    float y[8];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float2 u = __fmul2_rn(make_float2(bf16_lo(w[j]), bf16_hi(w[j])), eb);
                        y[2 * j] = u.x;
                        y[2 * j + 1] = u.y;
                    }
                    uint32_t packed;
                    if constexpr (SR) {
                        const uint64_t idx0 = (uint64_t)((r0 + i) * C + c0);      // c0 % 8 == 0
                        const Philox4 p = sr_philox(key, 0u, sr_offset, idx0 >> 4);
                        const bool upper = (idx0 & 8) != 0;
                        packed = e2m1x4_sr(y[0], y[1], y[2], y[3], upper ? p.w[2] : p.w[0]) |
                                 (e2m1x4_sr(y[4], y[5], y[6], y[7], upper ? p.w[3] : p.w[1]) << 16);
                    } else {
                        packed = e2m1x8_rn(y);
                    }
                    *reinterpret_cast<uint32_t*>(out.codes + (r0 + i) * (C / 2) + c0 / 2) = packed;
                    if (i < 8) lo[i] = packed;
                    else hi[i - 8] = packed;
                }
                if (out.codes_t) {
                    transpose_nibbles8(lo);
                    transpose_nibbles8(hi);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        *reinterpret_cast<uint2*>(out.codes_t + (c0 + j) * (R / 2) + r0 / 2) = make_uint2(lo[j], hi[j]);
                }
                if ((cc & 1) == 0 && out.scales) out.scales[(r0 / 16) * (C / 16) + c0 / 16] = (uint8_t)sb;
            }
            // Tile-layout scales as 32-bit words (four adjacent scale columns of one row), so a
            // lane stores two words instead of sixteen bytes; every lane takes part in the shuffles.
            const int rg = lane >> 3;
            if (out.scales_mma) {
                // scale columns c0/16 of the lanes cc = 0, 2, 4, 6 of this row group; rows r0 + cc, r0 + cc + 8
                uint32_t w = 0u;
#pragma unroll
                for (int k = 0; k < 4; ++k) w |= __shfl_sync(0xFFFFFFFFu, sb, (lane & 24) | (2 * k)) << (8 * k);
                const bool base_ok = __shfl_sync(0xFFFFFFFFu, ok ? 1u : 0u, lane & 24) != 0u;
                if (base_ok) {
                    const int64_t s0 = (c0 - cc * 8) / 16;              // a multiple of 4
                    *reinterpret_cast<uint32_t*>(out.scales_mma + mma_sf_offset(r0 + cc, s0, nkb)) = w;
                    *reinterpret_cast<uint32_t*>(out.scales_mma + mma_sf_offset(r0 + cc + 8, s0, nkb)) = w;
                }
            }
            if (out.scales_mma_t) {
                // W^T rows = this 16-column block's columns; scale columns r0/16 of the row groups 0..3
                uint32_t w = 0u;
#pragma unroll
                for (int k = 0; k < 4; ++k) w |= __shfl_sync(0xFFFFFFFFu, sb, (k << 3) | (cc & 6)) << (8 * k);
                const bool base_ok = __shfl_sync(0xFFFFFFFFu, ok ? 1u : 0u, cc & 6) != 0u;
                if (base_ok) {
                    const int64_t st0 = (r0 - rg * 16) / 16;            // a multiple of 4
                    const int64_t cb = c0 - (cc & 1) * 8;                // the block's first column
                    const int64_t j = (cc & 1) * 8 + rg * 2;
                    *reinterpret_cast<uint32_t*>(out.scales_mma_t + mma_sf_offset(cb + j, st0, nkb_t)) = w;
                    *reinterpret_cast<uint32_t*>(out.scales_mma_t + mma_sf_offset(cb + j + 1, st0, nkb_t)) = w;
                }
            }
        }
    } else {
        while (pp.next()) {
            const int64_t r0 = pp.r0, c0 = pp.c0;
            // every lane takes part in the shuffles; invalid ones contribute 0
            const bool valid = pp.ok;
            float t[VEC][16];
            float amax = 0.0f;
            if (valid) {
                uint4 v[16];
                pp.read(v);
                unpack_patch<T>(v, t);
                float cm[VEC];
    #pragma unroll
                for (int j = 0; j < VEC; ++j) cm[j] = abs_max16(t[j]);
    #pragma unroll
                for (int s = VEC / 2; s >= 1; s >>= 1)
    #pragma unroll
                    for (int j = 0; j < s; ++j) cm[j] = fmaxf(cm[j], cm[j + s]);
                amax = cm[0];
            }
    #pragma unroll
            for (int o = 1; o < LPT; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
            if (!valid) continue;
            const uint32_t sb = sizeof(T) == 2 ? block_scale_code_bf16(amax, sc.s_enc) : block_scale_code(amax, sc.s_enc);
            const float e_b = g_eb_table[sb];
            // Encode row by row (W); the W^T codes are the same nibbles, transposed in registers.
            uint32_t lo_t[VEC], hi_t[VEC];
    #pragma unroll
            for (int j = 0; j < VEC; ++j) { lo_t[j] = 0u; hi_t[j] = 0u; }
    #pragma unroll
            for (int i = 0; i < 16; ++i) {
                float y[VEC];
    #pragma unroll
                for (int j = 0; j < VEC; ++j) y[j] = __fmul_rn(t[j][i], e_b);
                uint32_t packed;
                if constexpr (SR) {
                    // elements idx0 .. idx0+VEC-1 use words ((idx0 >> 2) & 3) .. of their 16-element call
                    const uint64_t idx0 = (uint64_t)((r0 + i) * C + c0);
                    const Philox4 p = sr_philox(key, 0u, sr_offset, idx0 >> 4);
                    if constexpr (VEC == 8) {
                        const bool hi = (idx0 & 8) != 0;
                        packed = e2m1x4_sr(y[0], y[1], y[2], y[3], hi ? p.w[2] : p.w[0]) |
                                 (e2m1x4_sr(y[4], y[5], y[6], y[7], hi ? p.w[3] : p.w[1]) << 16);
                    } else {
                        const uint32_t k = (uint32_t)(idx0 >> 2) & 3u;
                        const uint32_t word = k == 0 ? p.w[0] : k == 1 ? p.w[1] : k == 2 ? p.w[2] : p.w[3];
                        packed = e2m1x4_sr(y[0], y[1], y[2], y[3], word);
                    }
                } else {
                    if constexpr (VEC == 8) packed = e2m1x8_rn(y);
                    else packed = e2m1x4_rn(y);
                }
                uint8_t* dst = out.codes + (r0 + i) * (C / 2) + c0 / 2;
                if constexpr (VEC == 8) *reinterpret_cast<uint32_t*>(dst) = packed;
                else *reinterpret_cast<uint16_t*>(dst) = (uint16_t)packed;
    #pragma unroll
                for (int j = 0; j < VEC; ++j) {
                    const uint32_t nib = (packed >> (4 * j)) & 0xFu;
                    if (i < 8) lo_t[j] |= nib << (4 * i);
                    else hi_t[j] |= nib << (4 * (i - 8));
                }
            }
            if (out.codes_t) {
    #pragma unroll
                for (int j = 0; j < VEC; ++j)
                    *reinterpret_cast<uint2*>(out.codes_t + (c0 + j) * (R / 2) + r0 / 2) = make_uint2(lo_t[j], hi_t[j]);
            }
            if ((cc % LPT) == 0) {
                const int64_t s = c0 / 16, st = r0 / 16;
                if (out.scales) out.scales[st * (C / 16) + s] = (uint8_t)sb;
                if (out.scales_mma)
                    for (int i = 0; i < 16; ++i) out.scales_mma[mma_sf_offset(r0 + i, s, nkb)] = (uint8_t)sb;
                if (out.scales_mma_t)
                    for (int j = 0; j < 16; ++j) out.scales_mma_t[mma_sf_offset(c0 + j, st, nkb_t)] = (uint8_t)sb;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
}  // namespace nvfp4

using namespace nvfp4;

extern "C" size_t nvfp4_scales_mma_bytes(int64_t rows, int64_t cols) {
    if (rows <= 0 || cols <= 0) return 0;
    return (size_t)((rows + 127) / 128) * (size_t)((cols + 255) / 256) * 2048u;
}

extern "C" size_t nvfp4_quantize_workspace_bytes(int64_t, int64_t, const nvfp4_qparams*) {
    return (size_t)kMaxPartials * sizeof(uint32_t);
}

namespace nvfp4 {

namespace {

// Host-side argument checks shared by the single and the dual quantization.
nvfp4_status check_quantize_args(const void* x, int32_t x_dtype, int64_t R, int64_t C, int64_t ldx,
                                 const nvfp4_qparams* p, const nvfp4_qtensor* out) {
    if (!p || !out || !out->s_dec) return NVFP4_ERR_INVALID_ARG;
    if (x_dtype != NVFP4_F32 && x_dtype != NVFP4_BF16) return NVFP4_ERR_INVALID_ARG;
    if (p->block < NVFP4_BLOCK_1X16_ROW || p->block > NVFP4_BLOCK_16X16) return NVFP4_ERR_INVALID_ARG;
    if (p->round != NVFP4_ROUND_RNE && p->round != NVFP4_ROUND_SR) return NVFP4_ERR_INVALID_ARG;
    if (p->rht && p->block != NVFP4_BLOCK_1X16_COL) return NVFP4_ERR_INVALID_ARG;
    if (R < 0 || C < 0 || ldx < C) return NVFP4_ERR_SHAPE;
    const bool col = p->block == NVFP4_BLOCK_1X16_COL;
    const int64_t rows = col ? C : R, cols = col ? R : C;
    if (out->rows != rows || out->cols != cols) return NVFP4_ERR_SHAPE;
    if (C % 16 != 0) return NVFP4_ERR_SHAPE;
    if ((col || p->block == NVFP4_BLOCK_16X16) && R % 16 != 0) return NVFP4_ERR_SHAPE;
    // the kernels address the tensor-core scale layout with 32-bit offsets
    if (nvfp4_scales_mma_bytes(rows, cols) >= (1ull << 32) || nvfp4_scales_mma_bytes(cols, rows) >= (1ull << 32))
        return NVFP4_ERR_SHAPE;
    const size_t esz = x_dtype == NVFP4_BF16 ? 2 : 4;
    const bool empty = (R == 0 || C == 0);
    if (!empty) {
        if (!x || !out->codes) return NVFP4_ERR_INVALID_ARG;
        if (!out->scales && !out->scales_mma) return NVFP4_ERR_INVALID_ARG;
        if (!aligned16(x) || ((size_t)ldx * esz) % 16 != 0 || !aligned16(out->codes)) return NVFP4_ERR_ALIGNMENT;
        if (p->block == NVFP4_BLOCK_16X16 && out->codes_t && !aligned16(out->codes_t)) return NVFP4_ERR_ALIGNMENT;
        if ((out->scales_mma && !aligned16(out->scales_mma)) ||
            (p->block == NVFP4_BLOCK_16X16 && out->scales_mma_t && !aligned16(out->scales_mma_t)))
            return NVFP4_ERR_ALIGNMENT;
    }
    return NVFP4_OK;
}

// CTAs of one kernel resident on an SM at once (registers and shared memory),
// looked up once per kernel and device.
template <typename K>
int resident_per_sm(K* kern, int threads, size_t smem) {
    static std::mutex mu;
    static std::map<std::pair<int, const void*>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    std::lock_guard<std::mutex> lk(mu);
    const auto key = std::make_pair(dev, reinterpret_cast<const void*>(kern));
    const auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, smem) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 1;
    }
    n = std::max(n, 1);
    cache[key] = n;
    return n;
}

// Launch a grid-stride kernel of kThreads threads with one wave of resident CTAs
// (the SM count times the kernel's occupancy), or fewer when the work is smaller;
// *grid = the CTAs launched.
template <typename K, typename... Args>
cudaError_t launch_resident(K* kern, int64_t work_ctas, int sms, int* grid, cudaStream_t stream, Args... args) {
    const int64_t wave = (int64_t)sms * resident_per_sm(kern, kThreads, 0);
    *grid = (int)std::max<int64_t>(1, std::min<int64_t>(std::min<int64_t>(wave, work_ctas), kMaxPartials));
    return launch_pdl(kern, dim3(*grid), dim3(kThreads), 0, stream, args...);
}

// Grid of the patch kernels: one CTA (eight warps) per SM at most, one warp per
// 64 x (8 * 16 B) tile at least.
int patch_grid(int sms, int64_t R, int64_t C, bool is16, int ctas_per_sm = kPatchCtasPerSm) {
    const int vec = is16 ? 8 : 4;
    const int64_t tiles = (R == 0 || C == 0) ? 0 : ((R + 63) / 64) * ((C + 8 * vec - 1) / (8 * vec));
    const int64_t g = std::max<int64_t>(1, std::min<int64_t>((int64_t)sms * ctas_per_sm,
                                                             (tiles + kPatchThreads / 32 - 1) / (kPatchThreads / 32)));
    return (int)std::min<int64_t>(g, kMaxPartials);
}

// The patch kernels' dynamic shared memory (the cp.async double buffer), allowed once
// per kernel and device.
template <typename K>
cudaError_t allow_patch_smem(K* kern, int bytes = kPatchSmemBytes) {
    static std::mutex mu;
    static std::set<std::pair<int, const void*>> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(mu);
    const auto key = std::make_pair(dev, reinterpret_cast<const void*>(kern));
    if (done.count(key)) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.insert(key);
    return e;
}

template <typename K, typename... Args>
cudaError_t launch_patch(K* kern, int grid, cudaStream_t stream, Args... args) {
    const cudaError_t e = allow_patch_smem(kern);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(kPatchThreads), kPatchSmemBytes, stream, args...);
}
// The maxima passes and the 16x16 encoder: kAmaxAhead copies in flight per warp (more shared
// memory, fewer CTAs).
template <typename K, typename... Args>
cudaError_t launch_patch_amax(K* kern, int grid, cudaStream_t stream, Args... args) {
    const cudaError_t e = allow_patch_smem(kern, kAmaxSmemBytes);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(kPatchThreads), kAmaxSmemBytes, stream, args...);
}

// Pass 1 for one quantization: per-CTA partial maxima of |x| or |RHT(x)|; *g1 = their count.
cudaError_t amax_pass(const void* x, bool is16, int64_t R, int64_t C, int64_t ldx, bool rht, uint64_t rht_seed,
                      uint32_t* partials, int sms, int* g1, cudaStream_t stream, bool sqr = false) {
    const int64_t chunks = (R == 0 || C == 0) ? 0 : R * (C / (is16 ? 8 : 4));
    if (rht) {
        *g1 = patch_grid(sms, R, C, is16, kAmaxCtasPerSm);
        return is16 ? launch_patch_amax(amax_rht_kernel<uint16_t>, *g1, stream, (const uint16_t*)x, R, C, ldx, rht_seed, partials)
                    : launch_patch_amax(amax_rht_kernel<float>, *g1, stream, (const float*)x, R, C, ldx, rht_seed, partials);
    }
    const int64_t work = (chunks + kThreads * 4 - 1) / (kThreads * 4);
    const uint16_t* xb = (const uint16_t*)x;
    if (ldx == C) {
        if (is16 && sqr) return launch_resident(amax_flat_kernel<uint16_t, true>, work, sms, g1, stream, xb, chunks, partials);
        if (is16) return launch_resident(amax_flat_kernel<uint16_t>, work, sms, g1, stream, xb, chunks, partials);
        return launch_resident(amax_flat_kernel<float>, work, sms, g1, stream, (const float*)x, chunks, partials);
    }
    if (is16 && sqr) return launch_resident(amax_kernel<uint16_t, true>, work, sms, g1, stream, xb, R, C, ldx, partials);
    if (is16) return launch_resident(amax_kernel<uint16_t>, work, sms, g1, stream, xb, R, C, ldx, partials);
    return launch_resident(amax_kernel<float>, work, sms, g1, stream, (const float*)x, R, C, ldx, partials);
}

// The kernels' view of an output, with the padding of its tensor-core scale layout
// (rows to 128, scale columns to 16) zeroed.
nvfp4_status prepare_output(const nvfp4_qparams* p, const nvfp4_qtensor* out, int64_t R, int64_t C, QOut* q,
                            cudaStream_t stream) {
    const bool col = p->block == NVFP4_BLOCK_1X16_COL;
    const int64_t rows = col ? C : R, cols = col ? R : C;
    *q = QOut{out->codes, out->scales, out->scales_mma,
              p->block == NVFP4_BLOCK_16X16 ? out->codes_t : nullptr,
              p->block == NVFP4_BLOCK_16X16 ? out->scales_mma_t : nullptr, out->s_dec};
    if (R == 0 || C == 0) return NVFP4_OK;
    if (q->scales_mma && (rows % 128 != 0 || cols % 256 != 0))
        if (cudaMemsetAsync(q->scales_mma, 0, nvfp4_scales_mma_bytes(rows, cols), stream) != cudaSuccess)
            return NVFP4_ERR_CUDA;
    if (q->scales_mma_t && (cols % 128 != 0 || rows % 256 != 0))
        if (cudaMemsetAsync(q->scales_mma_t, 0, nvfp4_scales_mma_bytes(cols, rows), stream) != cudaSuccess)
            return NVFP4_ERR_CUDA;
    return NVFP4_OK;
}

// Pass 2 for one quantization, given the pass-1 partials (g1 of them).
nvfp4_status encode_pass(const void* x, int32_t x_dtype, int64_t R, int64_t C, int64_t ldx, const nvfp4_qparams* p,
                         const nvfp4_qtensor* out, const uint32_t* partials, int g1, int sms, uint32_t* dev_status,
                         cudaStream_t stream, bool sqr = false) {
    const bool empty = (R == 0 || C == 0);
    const bool is16 = x_dtype == NVFP4_BF16;
    const size_t esz = is16 ? 2 : 4;
    const uint64_t rs = p->rht_seed;
    QOut q;
    const nvfp4_status st = prepare_output(p, out, R, C, &q, stream);
    if (st != NVFP4_OK) return st;

    const bool sr = p->round == NVFP4_ROUND_SR;
    const int64_t row_warps = empty ? 0 : R * ((C / 16 + 31) / 32);
    const int64_t row_ctas = (row_warps + 7) / 8;
    int g_row = 0;
    const int g_patch = patch_grid(sms, R, C, is16);
    const int g_deep = patch_grid(sms, R, C, is16, kAmaxCtasPerSm);
    // 32-byte loads when every 16-element block starts on a 32-byte boundary
    const int v8 = ((reinterpret_cast<uintptr_t>(x) & 31u) == 0 && ((size_t)ldx * esz) % 32 == 0) ? 1 : 0;
    const PhiloxKey ss = philox_key(p->sr_seed);
    const uint32_t so = p->sr_offset;
    cudaError_t e = cudaSuccess;
#define NVFP4_LAUNCH_T(T)                                                                                  \
    do {                                                                                                   \
        const T* xt = (const T*)x;                                                                         \
        if (p->block == NVFP4_BLOCK_1X16_ROW) {                                                            \
            if (sr) e = launch_resident(encode_row_kernel<T, true>, row_ctas, sms, &g_row, stream, xt, R, C, ldx, partials, g1, q, ss, so, v8, dev_status); \
            else e = launch_resident(encode_row_kernel<T, false>, row_ctas, sms, &g_row, stream, xt, R, C, ldx, partials, g1, q, ss, so, v8, dev_status); \
        } else if (p->block == NVFP4_BLOCK_1X16_COL) {                                                     \
            if (sr && p->rht) e = launch_patch(encode_col_kernel<T, true, true>, g_patch, stream, xt, R, C, ldx, partials, g1, q, ss, so, rs, dev_status); \
            else if (sr) e = launch_patch(encode_col_kernel<T, true, false>, g_patch, stream, xt, R, C, ldx, partials, g1, q, ss, so, rs, dev_status); \
            else if (p->rht) e = launch_patch(encode_col_kernel<T, false, true>, g_patch, stream, xt, R, C, ldx, partials, g1, q, ss, so, rs, dev_status); \
            else e = launch_patch(encode_col_kernel<T, false, false>, g_patch, stream, xt, R, C, ldx, partials, g1, q, ss, so, rs, dev_status); \
        } else {                                                                                           \
            if (sr) e = launch_patch_amax(encode_2d_kernel<T, true>, g_deep, stream, xt, R, C, ldx, partials, g1, q, ss, so, dev_status); \
            else e = launch_patch_amax(encode_2d_kernel<T, false>, g_deep, stream, xt, R, C, ldx, partials, g1, q, ss, so, dev_status); \
        }                                                                                                  \
    } while (0)
    if (is16 && sqr) {
        // bf16 with the squared-ReLU load transform (row and column operands only)
        const uint16_t* xt = (const uint16_t*)x;
        if (p->block == NVFP4_BLOCK_1X16_ROW) {
            if (sr) e = launch_resident(encode_row_kernel<uint16_t, true, true>, row_ctas, sms, &g_row, stream, xt, R, C, ldx, partials, g1, q, ss, so, v8, dev_status);
            else e = launch_resident(encode_row_kernel<uint16_t, false, true>, row_ctas, sms, &g_row, stream, xt, R, C, ldx, partials, g1, q, ss, so, v8, dev_status);
        } else if (p->block == NVFP4_BLOCK_1X16_COL) {
            if (sr && p->rht) e = launch_patch(encode_col_kernel<uint16_t, true, true, true>, g_patch, stream, xt, R, C, ldx, partials, g1, q, ss, so, rs, dev_status);
            else if (sr) e = launch_patch(encode_col_kernel<uint16_t, true, false, true>, g_patch, stream, xt, R, C, ldx, partials, g1, q, ss, so, rs, dev_status);
            else if (p->rht) e = launch_patch(encode_col_kernel<uint16_t, false, true, true>, g_patch, stream, xt, R, C, ldx, partials, g1, q, ss, so, rs, dev_status);
            else e = launch_patch(encode_col_kernel<uint16_t, false, false, true>, g_patch, stream, xt, R, C, ldx, partials, g1, q, ss, so, rs, dev_status);
        } else {
            return NVFP4_ERR_UNSUPPORTED;
        }
    } else if (is16) {
        NVFP4_LAUNCH_T(uint16_t);
    } else {
        NVFP4_LAUNCH_T(float);
    }
#undef NVFP4_LAUNCH_T
    if (e != cudaSuccess) return NVFP4_ERR_CUDA;
    return NVFP4_OK;
}

}  // namespace

nvfp4_status quantize_impl(const void* x, int32_t x_dtype, int64_t R, int64_t C, int64_t ldx,
                           const nvfp4_qparams* p, const nvfp4_qtensor* out, void* ws, size_t ws_bytes,
                           uint32_t* dev_status, cudaStream_t stream) {
    nvfp4_status st = check_quantize_args(x, x_dtype, R, C, ldx, p, out);
    if (st != NVFP4_OK) return st;
    if (!ws || ws_bytes < (size_t)kMaxPartials * sizeof(uint32_t) || !aligned16(ws)) return NVFP4_ERR_WORKSPACE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return NVFP4_ERR_CUDA;
    const int sms = sm_count(dev);
    if (sms <= 0) return NVFP4_ERR_CUDA;
    const bool is16 = x_dtype == NVFP4_BF16;
    uint32_t* partials = static_cast<uint32_t*>(ws);
    int g1 = 0;
    if (amax_pass(x, is16, R, C, ldx, p->rht != 0, p->rht_seed, partials, sms, &g1, stream) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    return encode_pass(x, x_dtype, R, C, ldx, p, out, partials, g1, sms, dev_status, stream);
}

// Whether a dual quantization takes the fused encode (one read of x for both operands):
// bf16 x, a non-empty tensor, the RHT column operand and one rounding mode for both.
bool dual_fused(int32_t x_dtype, int64_t R, int64_t C, const nvfp4_qparams* p_row, const nvfp4_qparams* p_col) {
    return x_dtype == NVFP4_BF16 && R > 0 && C > 0 && p_col->rht && p_row->round == p_col->round;
}

// Pass 2 of a dual quantization that dual_fused accepts: one encode_dual_kernel launch.
nvfp4_status encode_dual_pass(const void* x, int64_t R, int64_t C, int64_t ldx, const nvfp4_qparams* p_row,
                              const nvfp4_qtensor* out_row, const nvfp4_qparams* p_col, const nvfp4_qtensor* out_col,
                              const uint32_t* part_row, const uint32_t* part_col, int g1, int sms,
                              uint32_t* dev_status, cudaStream_t stream, bool sqr) {
    QOut qr, qc;
    nvfp4_status st = prepare_output(p_row, out_row, R, C, &qr, stream);
    if (st != NVFP4_OK) return st;
    st = prepare_output(p_col, out_col, R, C, &qc, stream);
    if (st != NVFP4_OK) return st;
    const int g = patch_grid(sms, R, C, true);
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    auto launch = [&](auto* kern) {
        return launch_patch(kern, g, stream, xb, R, C, ldx, part_row, part_col, g1, qr, qc, philox_key(p_row->sr_seed),
                            philox_key(p_col->sr_seed), p_row->sr_offset, p_col->sr_offset, p_col->rht_seed, dev_status);
    };
    const bool sr = p_row->round == NVFP4_ROUND_SR;
    const cudaError_t e = sr ? (sqr ? launch(encode_dual_kernel<true, true>) : launch(encode_dual_kernel<true, false>))
                             : (sqr ? launch(encode_dual_kernel<false, true>) : launch(encode_dual_kernel<false, false>));
    return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

nvfp4_status quantize_dual_impl(const void* x, int32_t x_dtype, int64_t R, int64_t C, int64_t ldx,
                                const nvfp4_qparams* p_row, const nvfp4_qtensor* out_row,
                                const nvfp4_qparams* p_col, const nvfp4_qtensor* out_col, void* ws,
                                size_t ws_bytes, uint32_t* dev_status, cudaStream_t stream, bool sqr = false) {
    if (!p_row || !p_col) return NVFP4_ERR_INVALID_ARG;
    if (sqr && x_dtype != NVFP4_BF16) return NVFP4_ERR_UNSUPPORTED;
    if (p_row->block != NVFP4_BLOCK_1X16_ROW || p_col->block != NVFP4_BLOCK_1X16_COL) return NVFP4_ERR_INVALID_ARG;
    nvfp4_status st = check_quantize_args(x, x_dtype, R, C, ldx, p_row, out_row);
    if (st != NVFP4_OK) return st;
    st = check_quantize_args(x, x_dtype, R, C, ldx, p_col, out_col);
    if (st != NVFP4_OK) return st;
    if (!ws || ws_bytes < 2 * (size_t)kMaxPartials * sizeof(uint32_t) || !aligned16(ws)) return NVFP4_ERR_WORKSPACE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return NVFP4_ERR_CUDA;
    const int sms = sm_count(dev);
    if (sms <= 0) return NVFP4_ERR_CUDA;
    const bool is16 = x_dtype == NVFP4_BF16;
    uint32_t* part_plain = static_cast<uint32_t*>(ws);
    uint32_t* part_col = part_plain + kMaxPartials;
    int g1 = 0;
    if (p_col->rht) {
        // one read of x for both tensor amaxes
        g1 = patch_grid(sms, R, C, is16, kAmaxCtasPerSm);
        const cudaError_t e = !is16
            ? launch_patch_amax(amax_dual_kernel<float>, g1, stream, (const float*)x, R, C, ldx, p_col->rht_seed, part_plain, part_col)
            : sqr ? launch_patch_amax(amax_dual_kernel<uint16_t, true>, g1, stream, (const uint16_t*)x, R, C, ldx, p_col->rht_seed, part_plain, part_col)
                  : launch_patch_amax(amax_dual_kernel<uint16_t>, g1, stream, (const uint16_t*)x, R, C, ldx, p_col->rht_seed, part_plain, part_col);
        if (e != cudaSuccess) return NVFP4_ERR_CUDA;
    } else {
        // without the RHT both operands share the plain amax
        if (amax_pass(x, is16, R, C, ldx, false, 0, part_plain, sms, &g1, stream, sqr) != cudaSuccess) return NVFP4_ERR_CUDA;
        part_col = part_plain;
    }
    if (dual_fused(x_dtype, R, C, p_row, p_col))
        return encode_dual_pass(x, R, C, ldx, p_row, out_row, p_col, out_col, part_plain, part_col, g1, sms, dev_status,
                                stream, sqr);
    st = encode_pass(x, x_dtype, R, C, ldx, p_row, out_row, part_plain, g1, sms, dev_status, stream, sqr);
    if (st != NVFP4_OK) return st;
    return encode_pass(x, x_dtype, R, C, ldx, p_col, out_col, part_col, g1, sms, dev_status, stream, sqr);
}

}  // namespace nvfp4

extern "C" nvfp4_status nvfp4_quantize(const void* x, int32_t x_dtype, int64_t R, int64_t C, int64_t ldx,
                                       const nvfp4_qparams* params, const nvfp4_qtensor* out,
                                       void* workspace, size_t workspace_bytes, uint32_t* dev_status,
                                       void* stream) {
    return nvfp4::quantize_impl(x, x_dtype, R, C, ldx, params, out, workspace, workspace_bytes, dev_status,
                                static_cast<cudaStream_t>(stream));
}

extern "C" nvfp4_status nvfp4_quantize_dual_sqrelu(const void* h, int32_t h_dtype, int64_t R, int64_t C, int64_t ldh,
                                                   const nvfp4_qparams* params_row, const nvfp4_qtensor* out_row,
                                                   const nvfp4_qparams* params_col, const nvfp4_qtensor* out_col,
                                                   void* workspace, size_t workspace_bytes, uint32_t* dev_status,
                                                   void* stream) {
    return nvfp4::quantize_dual_impl(h, h_dtype, R, C, ldh, params_row, out_row, params_col, out_col, workspace,
                                     workspace_bytes, dev_status, static_cast<cudaStream_t>(stream), true);
}

namespace nvfp4 {
// The dual quantization with the tensor maxima already known (left by the GEMM epilogue that
// produced x): only the two encode passes run.  BF16 x; with sqr, of relu(x)^2.
static nvfp4_status quantize_dual_premax_impl(const void* x, int32_t x_dtype, int64_t R, int64_t C, int64_t ldx,
                                              const nvfp4_qparams* p_row, const nvfp4_qtensor* out_row,
                                              const nvfp4_qparams* p_col, const nvfp4_qtensor* out_col,
                                              const uint32_t* maxima, size_t maxima_bytes, uint32_t* dev_status,
                                              cudaStream_t stream, bool sqr) {
    if (!p_row || !p_col || !maxima) return NVFP4_ERR_INVALID_ARG;
    // two halves of `parts` partial maxima each (what nvfp4_sqrelu_maxima_bytes sizes)
    const size_t parts = maxima_bytes / (2 * sizeof(uint32_t));
    if (parts == 0 || parts > (1u << 30)) return NVFP4_ERR_WORKSPACE;
    if (x_dtype != NVFP4_BF16) return NVFP4_ERR_UNSUPPORTED;
    if (p_row->block != NVFP4_BLOCK_1X16_ROW || p_col->block != NVFP4_BLOCK_1X16_COL) return NVFP4_ERR_INVALID_ARG;
    nvfp4_status st = check_quantize_args(x, x_dtype, R, C, ldx, p_row, out_row);
    if (st != NVFP4_OK) return st;
    st = check_quantize_args(x, x_dtype, R, C, ldx, p_col, out_col);
    if (st != NVFP4_OK) return st;
    if ((reinterpret_cast<uintptr_t>(maxima) & 3u) != 0) return NVFP4_ERR_ALIGNMENT;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return NVFP4_ERR_CUDA;
    const int sms = sm_count(dev);
    if (sms <= 0) return NVFP4_ERR_CUDA;
    const uint32_t* part_col = p_col->rht ? maxima + parts : maxima;
    if (dual_fused(x_dtype, R, C, p_row, p_col))
        return encode_dual_pass(x, R, C, ldx, p_row, out_row, p_col, out_col, maxima, part_col, (int)parts, sms,
                                dev_status, stream, sqr);
    st = encode_pass(x, x_dtype, R, C, ldx, p_row, out_row, maxima, (int)parts, sms, dev_status, stream, sqr);
    if (st != NVFP4_OK) return st;
    return encode_pass(x, x_dtype, R, C, ldx, p_col, out_col, part_col, (int)parts, sms, dev_status, stream, sqr);
}
}  // namespace nvfp4

extern "C" nvfp4_status nvfp4_quantize_dual_sqrelu_premax(const void* h, int32_t h_dtype, int64_t R, int64_t C,
                                                          int64_t ldh, const nvfp4_qparams* params_row,
                                                          const nvfp4_qtensor* out_row, const nvfp4_qparams* params_col,
                                                          const nvfp4_qtensor* out_col, const uint32_t* maxima,
                                                          size_t maxima_bytes, uint32_t* dev_status, void* stream) {
    return nvfp4::quantize_dual_premax_impl(h, h_dtype, R, C, ldh, params_row, out_row, params_col, out_col, maxima,
                                            maxima_bytes, dev_status, static_cast<cudaStream_t>(stream), true);
}

extern "C" nvfp4_status nvfp4_quantize_dual_premax(const void* x, int32_t x_dtype, int64_t R, int64_t C, int64_t ldx,
                                                   const nvfp4_qparams* params_row, const nvfp4_qtensor* out_row,
                                                   const nvfp4_qparams* params_col, const nvfp4_qtensor* out_col,
                                                   const uint32_t* maxima, size_t maxima_bytes, uint32_t* dev_status,
                                                   void* stream) {
    return nvfp4::quantize_dual_premax_impl(x, x_dtype, R, C, ldx, params_row, out_row, params_col, out_col, maxima,
                                            maxima_bytes, dev_status, static_cast<cudaStream_t>(stream), false);
}

extern "C" size_t nvfp4_quantize_dual_workspace_bytes(int64_t, int64_t) {
    return 2 * (size_t)kMaxPartials * sizeof(uint32_t);
}

extern "C" nvfp4_status nvfp4_quantize_dual(const void* x, int32_t x_dtype, int64_t R, int64_t C, int64_t ldx,
                                            const nvfp4_qparams* params_row, const nvfp4_qtensor* out_row,
                                            const nvfp4_qparams* params_col, const nvfp4_qtensor* out_col,
                                            void* workspace, size_t workspace_bytes, uint32_t* dev_status,
                                            void* stream) {
    return nvfp4::quantize_dual_impl(x, x_dtype, R, C, ldx, params_row, out_row, params_col, out_col, workspace,
                                     workspace_bytes, dev_status, static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
// Allocation-free quantize.  Same kernels and results as nvfp4_quantize, but
// the amax pass's partial maxima go to a file-scope device array instead of a
// caller-provided workspace.  For callers that can pass their input and output
// buffers but cannot obtain one more device buffer: a plug-in that only sees
// the tensors its host framework planned, or code that runs where allocating
// would re-enter or break the caller's allocator.
// ---------------------------------------------------------------------------
namespace nvfp4 {
namespace {

// The scratch: one partial maximum per amax CTA, kMaxPartials (4096) of them,
// 16 KB.  Every device that loads this library keeps it until the process exits.
// Host code must not pass the symbol itself to a kernel: on the host it is only
// a stand-in, so its device address is looked up with cudaGetSymbolAddress.
static __device__ __align__(256) uint32_t g_noalloc_partials[kMaxPartials];

std::mutex g_noalloc_mutex;

// The scratch's address is a property of the CUDA context that loaded this library's module,
// not of the device: after cudaDeviceReset (or a primary context that is released and created
// again) the module is loaded anew and the array may move.  So the cache is keyed on the
// context's process-unique id (cuCtxGetId), and a new context gets a fresh lookup.
struct NoallocEntry { unsigned long long ctx_id; void* addr; };
NoallocEntry g_noalloc_cache[16];
int g_noalloc_used = 0, g_noalloc_next = 0;

// Process-unique id of the calling thread's current context; 0 when there is none yet (or
// the driver entry points are unavailable).
unsigned long long current_ctx_id() {
    static PFN_cuCtxGetCurrent_v4000 get_cur = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void* f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_cur = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
    });
    CUcontext ctx = nullptr;
    if (!get_cur || !get_id || get_cur(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    unsigned long long id = 0;
    return get_id(ctx, &id) == CUDA_SUCCESS ? id : 0;
}

// Device address of the scratch in the current context, looked up once per context (the
// lookup also creates the device's primary context if none is current yet) and cached.
nvfp4_status noalloc_scratch(void** addr) {
    std::lock_guard<std::mutex> lk(g_noalloc_mutex);
    unsigned long long id = current_ctx_id();
    if (id != 0)
        for (int i = 0; i < g_noalloc_used; ++i)
            if (g_noalloc_cache[i].ctx_id == id) { *addr = g_noalloc_cache[i].addr; return NVFP4_OK; }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_partials) != cudaSuccess || !p) return NVFP4_ERR_CUDA;
    id = current_ctx_id();
    if (id != 0) {                       // remember it (the oldest entry makes room)
        g_noalloc_cache[g_noalloc_next] = NoallocEntry{id, p};
        g_noalloc_next = (g_noalloc_next + 1) % 16;
        g_noalloc_used = std::min(g_noalloc_used + 1, 16);
    }
    *addr = p;
    return NVFP4_OK;
}

}  // namespace
}  // namespace nvfp4

extern "C" nvfp4_status nvfp4_quantize_noalloc(const void* x, int32_t x_dtype, int64_t R, int64_t C, int64_t ldx,
                                               const nvfp4_qparams* params, const nvfp4_qtensor* out,
                                               uint32_t* dev_status, void* stream) {
    if (!params) return NVFP4_ERR_INVALID_ARG;
    if (nvfp4_quantize_workspace_bytes(R, C, params) > sizeof(nvfp4::g_noalloc_partials)) return NVFP4_ERR_WORKSPACE;
    void* scratch = nullptr;
    const nvfp4_status st = nvfp4::noalloc_scratch(&scratch);
    if (st != NVFP4_OK) return st;
    return nvfp4::quantize_impl(x, x_dtype, R, C, ldx, params, out, scratch, sizeof(nvfp4::g_noalloc_partials),
                                dev_status, static_cast<cudaStream_t>(stream));
}
