// mx.cu -- MXFP4 quantization (sm_103a), the 4-bit microscaling format the NVFP4
// recipe is compared against (news page "NVIDIA NVFP4 paper: 4-bit pretrain hits
// FP8 parity (12B, 10T tokens)", zubnet.ai, ¶3: at 8B parameters MXFP4 trails
// NVFP4 in loss and needs about a third more tokens to match it).
//
// The format is the OCP Microscaling one (the page names it, not its rules):
// blocks of 32 consecutive elements share one UE8M0 scale X = 2^(code - 127);
// code = floor(log2(amax_b)) - 2 + 127, clamped to [0, 254], puts the block's
// largest magnitude in [4, 8) = the top E2M1 binade; each element is
// e2m1_rne_sat(x / X).  There is no tensor-wide scale and no stochastic rounding.
//
// Kernels (both HBM-bound, one pass over the input):
//   mx_row_kernel<T>  one thread per 32-element block along a row: two or four
//                     32-byte streaming loads, the block maximum, the scale
//                     code from the exponent field, 16 bytes of codes;
//   mx_col_kernel<T>  blocks down the columns (the operand x^T): a CTA stages a
//                     64 x 128 tile in shared memory with coalesced 16-byte loads,
//                     then each thread walks one column (two blocks) and writes
//                     32 contiguous bytes of x^T's codes.
// Scales go to the canonical row-major array and/or the tensor-core tile layout
// the MXFP4 GEMM reads (1 KB tiles of 128 rows x 8 scales, see include/nvfp4.h).
#include <cuda_runtime.h>
#include <cstdint>

#include "device_common.cuh"
#include "host_common.h"

namespace nvfp4 {
namespace mx {

constexpr int kRowThreads = 256;
constexpr int kColRows = 64, kColCols = 128;          // col kernel tile: two blocks per column

// Scale code of a block from its largest magnitude (a non-negative float): the
// biased exponent field minus 2 for normal amax, clamped below at 0 (zero and
// subnormal maxima, whose log2 is below -126, clamp there too).
__device__ __forceinline__ uint32_t mx_scale_code(float amax) {
    const int e = (int)(__float_as_uint(amax) >> 23) - 2;
    return (uint32_t)max(e, 0);
}

// 1 / X = 2^(127 - code), code <= 252 for finite input so the result is a normal float.
__device__ __forceinline__ float mx_inv_scale(uint32_t code) { return __uint_as_float((254u - code) << 23); }

// Byte offset of (row r, scale column s) in the 1 KB-tile layout, nkt tiles per 128-row block.
__host__ __device__ __forceinline__ size_t mx_mma_offset(int64_t r, int64_t s, int64_t nkt) {
    return ((size_t)((r >> 7) * nkt + (s >> 3)) << 10) | ((size_t)((s >> 2) & 1) << 9) | ((size_t)(r & 31) << 4) |
           ((size_t)((r >> 5) & 3) << 2) | (size_t)(s & 3);
}

template <typename T> struct Block32;
template <> struct Block32<uint16_t> {                  // bf16: 64 bytes
    __device__ __forceinline__ static void load(const uint16_t* p, float (&v)[32]) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t w[8];
            ld_stream32(p + 16 * h, w);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                v[16 * h + 2 * i] = bf16_lo(w[i]);
                v[16 * h + 2 * i + 1] = bf16_hi(w[i]);
            }
        }
    }
};
template <> struct Block32<float> {                     // fp32: 128 bytes
    __device__ __forceinline__ static void load(const float* p, float (&v)[32]) {
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            uint32_t w[8];
            ld_stream32(p + 8 * h, w);
#pragma unroll
            for (int i = 0; i < 8; ++i) v[8 * h + i] = __uint_as_float(w[i]);
        }
    }
};

// 32 values of one block -> scale code and 16 bytes of codes (element 2j low nibble of byte j).
__device__ __forceinline__ uint4 mx_encode32(float (&v)[32], uint32_t& code) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    code = mx_scale_code(amax);
    const float inv = mx_inv_scale(code);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __fmul_rn(v[i], inv);      // exact: a power of two (or one rounding
                                                                    // of a far-below-0.25 subnormal)
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) w[q] = e2m1x8_rn(*reinterpret_cast<const float (*)[8]>(&v[8 * q]));
    return make_uint4(w[0], w[1], w[2], w[3]);
}

template <typename T>
__global__ void __launch_bounds__(kRowThreads)
mx_row_kernel(const T* __restrict__ x, int64_t ldx, int R, int C, int64_t nkt, uint8_t* __restrict__ codes,
              uint8_t* __restrict__ scales, uint8_t* __restrict__ scales_mma) {
    pdl_launch_dependents();
    pdl_wait();
    const int nb = C >> 5;
    const int64_t total = (int64_t)R * nb;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / nb;
        const int s = (int)(i - r * nb);
        float v[32];
        Block32<T>::load(x + r * ldx + 32 * s, v);
        uint32_t code;
        const uint4 c = mx_encode32(v, code);
        *reinterpret_cast<uint4*>(codes + r * (C >> 1) + 16 * s) = c;
        if (scales) scales[i] = (uint8_t)code;
        if (scales_mma) scales_mma[mx_mma_offset(r, s, nkt)] = (uint8_t)code;
    }
}

// x [R, C] -> x^T's codes [C, R/2] and scales [C, R/32].  Grid: (ceil(C/128), ceil(R/64)).
template <typename T>
__global__ void __launch_bounds__(kColCols)
mx_col_kernel(const T* __restrict__ x, int64_t ldx, int R, int C, int64_t nkt, uint8_t* __restrict__ codes_t,
              uint8_t* __restrict__ scales, uint8_t* __restrict__ scales_mma) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ __align__(16) T tile[kColRows][kColCols];
    constexpr int kChunk = 16 / sizeof(T);                     // elements per 16-byte load
    constexpr int kChunksPerRow = kColCols / kChunk;
    const int c0 = blockIdx.x * kColCols, r0 = blockIdx.y * kColRows;
    const int rows = min(kColRows, R - r0);                    // 32 or 64 (R is a multiple of 32)
    const bool full_cols = c0 + kColCols <= C;
    for (int k = threadIdx.x; k < kColRows * kChunksPerRow; k += kColCols) {
        const int r = k / kChunksPerRow, ch = k % kChunksPerRow;
        if (r >= rows) break;
        const int c = c0 + ch * kChunk;
        const T* src = x + (int64_t)(r0 + r) * ldx + c;
        if (full_cols || c + kChunk <= C) {
            *reinterpret_cast<uint4*>(&tile[r][ch * kChunk]) = ld_stream(src);
        } else {                                               // the ragged right edge: element loads
#pragma unroll
            for (int e = 0; e < kChunk; ++e) tile[r][ch * kChunk + e] = c + e < C ? src[e] : T(0);
        }
    }
    __syncthreads();
    const int c = c0 + threadIdx.x;
    if (c >= C) return;
    const int64_t ncodes = R >> 1, nsc = R >> 5;
    for (int b = 0; b < rows / 32; ++b) {
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            if constexpr (sizeof(T) == 2)
                v[i] = __uint_as_float((uint32_t)tile[32 * b + i][threadIdx.x] << 16);
            else
                v[i] = tile[32 * b + i][threadIdx.x];
        }
        uint32_t code;
        const uint4 q = mx_encode32(v, code);
        const int s = (r0 >> 5) + b;
        *reinterpret_cast<uint4*>(codes_t + (int64_t)c * ncodes + 16 * s) = q;
        if (scales) scales[(int64_t)c * nsc + s] = (uint8_t)code;
        if (scales_mma) scales_mma[mx_mma_offset(c, s, nkt)] = (uint8_t)code;
    }
}

template <typename K>
int grid_for(K kernel, int threads, int64_t work, int dev) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    const int64_t need = (work + threads - 1) / threads;
    return (int)std::max<int64_t>(1, std::min<int64_t>(need, (int64_t)per_sm * sm_count(dev)));
}

}  // namespace mx
}  // namespace nvfp4

using namespace nvfp4;

extern "C" size_t nvfp4_mx_scales_mma_bytes(int64_t rows, int64_t cols) {
    if (rows < 0 || cols < 0) return 0;
    return (size_t)((rows + 127) / 128) * (size_t)((cols + 255) / 256) * 1024u;
}

extern "C" nvfp4_status nvfp4_mx_quantize(const void* x, int32_t x_dtype, int64_t R, int64_t C, int64_t ldx,
                                          int32_t col, const nvfp4_qtensor* out, void* stream_) {
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    if (!x || !out || !out->codes) return NVFP4_ERR_INVALID_ARG;
    if (x_dtype != NVFP4_F32 && x_dtype != NVFP4_BF16) return NVFP4_ERR_INVALID_ARG;
    if (col != 0 && col != 1) return NVFP4_ERR_INVALID_ARG;
    if (R < 0 || C < 0 || ldx < C) return NVFP4_ERR_SHAPE;
    const int64_t rows = col ? C : R, cols = col ? R : C;       // the quantized operand's logical shape
    if (out->rows != rows || out->cols != cols) return NVFP4_ERR_SHAPE;
    if (cols % 32 != 0 || R > (1ll << 31) - 1 || C > (1ll << 31) - 1) return NVFP4_ERR_SHAPE;
    const size_t esz = x_dtype == NVFP4_BF16 ? 2 : 4;
    // the row kernel loads 32-byte pieces, the col kernel 16-byte ones
    const uintptr_t need = col ? 16 : 32;
    if ((reinterpret_cast<uintptr_t>(x) % need) != 0 || ((size_t)ldx * esz) % need != 0 || !aligned16(out->codes))
        return NVFP4_ERR_ALIGNMENT;
    if (col && (R + mx::kColRows - 1) / mx::kColRows > 65535) return NVFP4_ERR_SHAPE;   // grid.y of the col kernel
    if (R == 0 || C == 0) return NVFP4_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return NVFP4_ERR_CUDA;
    const int64_t nkt = (cols + 255) / 256;
    // padding rows and scale columns of the tile layout hold code 0 (never 0xFF, the NaN code)
    if (out->scales_mma && (rows % 128 != 0 || cols % 256 != 0))
        if (cudaMemsetAsync(out->scales_mma, 0, nvfp4_mx_scales_mma_bytes(rows, cols), stream) != cudaSuccess)
            return NVFP4_ERR_CUDA;
    cudaError_t e = cudaSuccess;
    if (!col) {
        const int64_t work = R * (C / 32);
        if (x_dtype == NVFP4_BF16) {
            auto k = mx::mx_row_kernel<uint16_t>;
            e = launch_pdl(k, dim3(mx::grid_for(k, mx::kRowThreads, work, dev)), dim3(mx::kRowThreads), 0, stream,
                           static_cast<const uint16_t*>(x), ldx, (int)R, (int)C, nkt, out->codes, out->scales,
                           out->scales_mma);
        } else {
            auto k = mx::mx_row_kernel<float>;
            e = launch_pdl(k, dim3(mx::grid_for(k, mx::kRowThreads, work, dev)), dim3(mx::kRowThreads), 0, stream,
                           static_cast<const float*>(x), ldx, (int)R, (int)C, nkt, out->codes, out->scales,
                           out->scales_mma);
        }
    } else {
        // x walks the column tiles (neighbouring CTAs read neighbouring pieces of the same rows)
        const int64_t row_tiles = (R + mx::kColRows - 1) / mx::kColRows;
        const dim3 grid((unsigned)((C + mx::kColCols - 1) / mx::kColCols), (unsigned)row_tiles);
        if (x_dtype == NVFP4_BF16)
            e = launch_pdl(mx::mx_col_kernel<uint16_t>, grid, dim3(mx::kColCols), 0, stream,
                           static_cast<const uint16_t*>(x), ldx, (int)R, (int)C, nkt, out->codes, out->scales,
                           out->scales_mma);
        else
            e = launch_pdl(mx::mx_col_kernel<float>, grid, dim3(mx::kColCols), 0, stream, static_cast<const float*>(x),
                           ldx, (int)R, (int)C, nkt, out->codes, out->scales, out->scales_mma);
    }
    return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}
