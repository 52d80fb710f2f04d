// linear.cu -- the NVFP4 linear layer's three GEMMs, each a quantize + GEMM on
// the caller's stream (news page "NVIDIA NVFP4 paper: 4-bit pretrain hits FP8
// parity (12B, 10T tokens)", ¶2):
//   Fprop  Y  = X . W^T     X 1x16 RNE along K,       W 16x16 (2D) RNE
//   Dgrad  dX = dY . W      dY 1x16 SR along N,       W^T from the same 2D quantization
//   Wgrad  dW = dY^T . X    dY^T and X^T 1x16 along M after the 16x16 RHT (one
//                           shared sign vector); dY^T SR, X^T RNE
// The quantized activations and gradients live in the caller's workspace:
//   [partials 16 KB][slot A: codes, tile scales, s_dec][slot B: same]
#include <cuda_runtime.h>
#include <algorithm>
#include <cstdint>

#include "host_common.h"

namespace nvfp4 {
namespace {

constexpr size_t kPartialBytes = 4096 * sizeof(uint32_t);

inline size_t up16(size_t v) { return (v + 15) & ~size_t(15); }

struct Slot { uint8_t* codes; uint8_t* scales_mma; float* s_dec; };

inline size_t slot_bytes(int64_t rows, int64_t cols) {
    return up16((size_t)rows * (size_t)cols / 2) + up16(nvfp4_scales_mma_bytes(rows, cols)) + 16;
}

// Slot A holds X (Fprop, [M, K]), dY (Dgrad, [M, N]) or dY^T (Wgrad, [N, M]); the
// tile-layout scales pad rows to 128 and columns to 256, so the orientations differ.
inline size_t slot_a_bytes(int64_t M, int64_t N, int64_t K) {
    return std::max(std::max(slot_bytes(M, K), slot_bytes(M, N)), slot_bytes(N, M));
}

inline Slot carve(uint8_t*& p, int64_t rows, int64_t cols) {
    Slot s;
    s.codes = p;
    p += up16((size_t)rows * (size_t)cols / 2);
    s.scales_mma = p;
    p += up16(nvfp4_scales_mma_bytes(rows, cols));
    s.s_dec = reinterpret_cast<float*>(p);
    p += 16;
    return s;
}

inline nvfp4_qtensor as_q(const Slot& s, int64_t rows, int64_t cols) {
    nvfp4_qtensor q{};
    q.codes = s.codes;
    q.scales_mma = s.scales_mma;
    q.s_dec = s.s_dec;
    q.rows = rows;
    q.cols = cols;
    return q;
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" size_t nvfp4_linear_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    if (M < 0 || N < 0 || K < 0) return 0;
    return kPartialBytes + slot_a_bytes(M, N, K) + slot_bytes(K, M) + 64;
}

extern "C" nvfp4_status nvfp4_linear_fprop(const void* X, int32_t x_dtype, int64_t M, int64_t K, int64_t ldx,
                                           const nvfp4_qtensor* Wq, void* Y, int32_t y_dtype, int64_t ldy,
                                           void* workspace, size_t workspace_bytes, uint32_t* dev_status,
                                           void* stream) {
    if (!Wq) return NVFP4_ERR_INVALID_ARG;
    if (Wq->cols != K) return NVFP4_ERR_SHAPE;
    const int64_t N = Wq->rows;
    if (!workspace || workspace_bytes < nvfp4_linear_workspace_bytes(M, N, K)) return NVFP4_ERR_WORKSPACE;
    uint8_t* p = static_cast<uint8_t*>(workspace);
    void* partials = p;
    p += kPartialBytes;
    const Slot xs = carve(p, M, K);
    nvfp4_qtensor xq = as_q(xs, M, K);
    nvfp4_qparams qp{NVFP4_BLOCK_1X16_ROW, NVFP4_ROUND_RNE, 0, 0u, 0ull, 0ull};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    nvfp4_status st = quantize_impl(X, x_dtype, M, K, ldx, &qp, &xq, partials, kPartialBytes, dev_status, s);
    if (st != NVFP4_OK) return st;
    return gemm_impl(&xq, Wq, Y, y_dtype, ldy, dev_status, s);
}

extern "C" nvfp4_status nvfp4_linear_dgrad(const void* dY, int32_t dy_dtype, int64_t M, int64_t N, int64_t lddy,
                                           const nvfp4_qtensor* Wq, uint64_t sr_seed, uint32_t sr_offset,
                                           void* dX, int32_t dx_dtype, int64_t lddx,
                                           void* workspace, size_t workspace_bytes, uint32_t* dev_status,
                                           void* stream) {
    if (!Wq || !Wq->codes_t || !Wq->scales_mma_t) return NVFP4_ERR_INVALID_ARG;
    if (Wq->rows != N) return NVFP4_ERR_SHAPE;
    const int64_t K = Wq->cols;
    if (!workspace || workspace_bytes < nvfp4_linear_workspace_bytes(M, N, K)) return NVFP4_ERR_WORKSPACE;
    uint8_t* p = static_cast<uint8_t*>(workspace);
    void* partials = p;
    p += kPartialBytes;
    const Slot ds = carve(p, M, N);
    nvfp4_qtensor dyq = as_q(ds, M, N);
    nvfp4_qtensor wt{};
    wt.codes = Wq->codes_t;
    wt.scales_mma = Wq->scales_mma_t;
    wt.s_dec = Wq->s_dec;
    wt.rows = K;
    wt.cols = N;
    nvfp4_qparams qp{NVFP4_BLOCK_1X16_ROW, NVFP4_ROUND_SR, 0, sr_offset, sr_seed, 0ull};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    nvfp4_status st = quantize_impl(dY, dy_dtype, M, N, lddy, &qp, &dyq, partials, kPartialBytes, dev_status, s);
    if (st != NVFP4_OK) return st;
    return gemm_impl(&dyq, &wt, dX, dx_dtype, lddx, dev_status, s);
}

extern "C" nvfp4_status nvfp4_linear_wgrad(const void* dY, int32_t dy_dtype, int64_t lddy,
                                           const void* X, int32_t x_dtype, int64_t ldx,
                                           int64_t M, int64_t N, int64_t K,
                                           uint64_t sr_seed, uint32_t sr_offset, uint64_t rht_seed,
                                           void* dW, int32_t dw_dtype, int64_t lddw,
                                           void* workspace, size_t workspace_bytes, uint32_t* dev_status,
                                           void* stream) {
    if (!workspace || workspace_bytes < nvfp4_linear_workspace_bytes(M, N, K)) return NVFP4_ERR_WORKSPACE;
    uint8_t* p = static_cast<uint8_t*>(workspace);
    void* partials = p;
    p += kPartialBytes;
    uint8_t* pa = p;
    const Slot ds = carve(pa, N, M);                 // dY^T: [N, M]
    p += slot_a_bytes(M, N, K);
    const Slot xs = carve(p, K, M);                  // X^T: [K, M]
    nvfp4_qtensor dyq = as_q(ds, N, M), xq = as_q(xs, K, M);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    nvfp4_qparams qd{NVFP4_BLOCK_1X16_COL, NVFP4_ROUND_SR, 1, sr_offset, sr_seed, rht_seed};
    nvfp4_status st = quantize_impl(dY, dy_dtype, M, N, lddy, &qd, &dyq, partials, kPartialBytes, dev_status, s);
    if (st != NVFP4_OK) return st;
    nvfp4_qparams qx{NVFP4_BLOCK_1X16_COL, NVFP4_ROUND_RNE, 1, 0u, 0ull, rht_seed};
    st = quantize_impl(X, x_dtype, M, K, ldx, &qx, &xq, partials, kPartialBytes, dev_status, s);
    if (st != NVFP4_OK) return st;
    return gemm_impl(&dyq, &xq, dW, dw_dtype, lddw, dev_status, s);
}
