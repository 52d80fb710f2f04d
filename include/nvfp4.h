/*
 * nvfp4.h -- C ABI of the GB300 (sm_103a) NVFP4 quantized linear layer.
 *
 * The method is the one summarised on the news page "NVIDIA NVFP4 paper: 4-bit
 * pretrain hits FP8 parity (12B, 10T tokens)" (zubnet.ai), cited as [page ¶n]:
 *   ¶2: E2M1 elements in 16-element blocks with an E4M3 scale per block and an
 *       FP32 per-tensor scale; 2D block scaling for weights; a 16x16 Random
 *       Hadamard Transform with random +-1 signs on the Wgrad inputs only;
 *       stochastic rounding on gradients only.
 *   ¶1, ¶3: the GEMMs run on Blackwell tensor cores.
 * Where the page is silent this library fixes one reading:
 *   tensor scale   s_enc = 2688 / amax_t (1 if amax_t = 0, clamped to FLT_MAX),
 *                  s_dec = 1 / s_enc (the stored FP32 per-tensor scale);
 *   block scale    S_b = e4m3_rne_satfinite((amax_b / 6) * s_enc);
 *   element        y = x * RN(s_enc / S_b), E2M1 round-to-nearest-even (ties to
 *                  the even code) or stochastic as Blackwell's conversion does
 *                  it (round up iff p + R * 2^-16 >= 1, p the position of |y|
 *                  between its grid neighbours, R 16 Philox4x32-10 bits); the
 *                  sign of x is kept (-0 -> 8);
 *   RHT            y = (1/4) H16 diag(s) v per 16-chunk along the token axis,
 *                  stages h = 1, 2, 4, 8, one sign vector s per call
 *                  (bit j of word 0 of Philox(key = rht_seed, counter = 0));
 *   SR bits        element i (row-major in the operand's logical [rows, cols])
 *                  draws on word ((i >> 2) & 3) of Philox(key = sr_seed,
 *                  counter = (i >> 4, stream, sr_offset)), stream 1 for column
 *                  quantization, 0 otherwise; with A = bits 16-23 : 0-7 and
 *                  B = bits 24-31 : 8-15 of the word, i % 4 = 0, 1, 2, 3 takes
 *                  A, A bit-reversed, B, B bit-reversed (how the four-wide
 *                  stochastic-rounding conversion splits one word).
 *
 * Conventions for every call below:
 *   - pointers are DEVICE pointers unless stated; `stream` is a cudaStream_t;
 *   - every call is asynchronous on `stream`, never allocates, never syncs
 *     (except nvfp4_status_query);
 *   - the caller owns every buffer;
 *   - host-side argument errors return a status and launch nothing;
 *   - device-side errors (a non-finite tensor, a pipeline wait that timed out)
 *     are written to *dev_status (a uint32 the caller zeroes once) and read back
 *     with nvfp4_status_query; after an error the outputs are unspecified.
 */
#ifndef NVFP4_GB300_H
#define NVFP4_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define NVFP4_API __attribute__((visibility("default")))
#else
#define NVFP4_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    NVFP4_OK = 0,
    NVFP4_ERR_INVALID_ARG = 1,   /* null pointer, bad enum, inconsistent operands */
    NVFP4_ERR_SHAPE = 2,         /* a dimension breaks the block or tile rules */
    NVFP4_ERR_ALIGNMENT = 3,     /* pointer or pitch not 16-byte aligned */
    NVFP4_ERR_WORKSPACE = 4,     /* workspace missing or too small */
    NVFP4_ERR_UNSUPPORTED = 5,   /* valid request this build does not implement */
    NVFP4_ERR_CUDA = 6,          /* a CUDA runtime call failed (launch, no device) */
    NVFP4_ERR_NONFINITE = 7,     /* device: the tensor amax was Inf or NaN */
    NVFP4_ERR_TIMEOUT = 8        /* device: a bounded pipeline wait ran out */
} nvfp4_status;

typedef enum { NVFP4_F32 = 0, NVFP4_BF16 = 1 } nvfp4_dtype;
typedef enum { NVFP4_ROUND_RNE = 0, NVFP4_ROUND_SR = 1 } nvfp4_round;
typedef enum {
    NVFP4_BLOCK_1X16_ROW = 0,    /* activations / Fprop & Dgrad gradients [page ¶2] */
    NVFP4_BLOCK_1X16_COL = 1,    /* Wgrad operands: blocks along the token axis */
    NVFP4_BLOCK_16X16 = 2        /* weights: 2D 16x16 tiles [page ¶2] */
} nvfp4_block;

/* Quantization parameters.  `rht` is only valid with NVFP4_BLOCK_1X16_COL. */
typedef struct {
    int32_t block;               /* nvfp4_block */
    int32_t round;               /* nvfp4_round */
    int32_t rht;                 /* 1: apply the 16x16 RHT (Wgrad inputs) */
    uint32_t sr_offset;          /* Philox counter word 3 for SR */
    uint64_t sr_seed;            /* Philox key for SR */
    uint64_t rht_seed;           /* Philox key for the RHT sign vector */
} nvfp4_qparams;

/*
 * A quantized operand of logical shape [rows, cols], 16-element blocks along cols.
 *   codes        [rows, cols/2] bytes, row pitch cols/2: element 2j in the low
 *                nibble of byte j, element 2j+1 in the high nibble.
 *   scales       canonical E4M3 block scales, row-major: [rows, cols/16]; for
 *                NVFP4_BLOCK_16X16 the tile grid [rows/16, cols/16].  May be NULL.
 *   scales_mma   the same scales in the tensor-core tile layout the GEMM reads:
 *                ceil(rows/128) x ceil(cols/256) tiles of 2048 bytes, tile
 *                (rb, kb) at byte ((rb * ceil(cols/256)) + kb) * 2048; inside a
 *                tile, the scale of row r, scale-column s (s = k/16) sits at
 *                ((s/4)%4)*512 + (r%32)*16 + ((r%128)/32)*4 + s%4.  Padding rows
 *                and scale-columns hold 0.  nvfp4_scales_mma_bytes() gives the
 *                size.  May be NULL (then the operand cannot feed nvfp4_gemm).
 *   s_dec        one float: the FP32 per-tensor decode scale.  Always written.
 *   codes_t,     NVFP4_BLOCK_16X16 only (else ignored): the transposed operand
 *   scales_mma_t [cols, rows/2] codes and its tile-layout scales, so that W and
 *                W^T share one quantized representation [page ¶2].  NULL: skip.
 * Dequantized value: e2m1(code) * e4m3(scale) * s_dec.
 */
typedef struct {
    uint8_t* codes;
    uint8_t* scales;
    uint8_t* scales_mma;
    float* s_dec;
    uint8_t* codes_t;
    uint8_t* scales_mma_t;
    int64_t rows;
    int64_t cols;
} nvfp4_qtensor;

/* Bytes of a tile-layout scale buffer for an operand of logical [rows, cols]. */
NVFP4_API size_t nvfp4_scales_mma_bytes(int64_t rows, int64_t cols);

/* Workspace bytes nvfp4_quantize needs (device memory, any contents, 16-byte
   aligned): the per-CTA partial maxima of the tensor amax pass. */
NVFP4_API size_t nvfp4_quantize_workspace_bytes(int64_t R, int64_t C, const nvfp4_qparams* params);

/*
 * nvfp4_quantize -- quantize x [R, C] (row pitch ldx elements, F32 or BF16).
 *   1X16_ROW : operand x,   out->rows = R, out->cols = C; C % 16 == 0.
 *   1X16_COL : operand x^T, out->rows = C, out->cols = R; R % 16 == 0, C % 16 == 0;
 *              with params->rht the RHT runs along R before everything else.
 *   16X16    : operand x,   out->rows = R, out->cols = C; R, C % 16 == 0.
 * Two passes over x: the tensor amax (after the RHT where it applies) and the
 * encode.  x, the output buffers and ldx*sizeof(elem) must be 16-byte aligned.
 * R == 0 or C == 0 is valid: only s_dec (= 1) is written.
 */
NVFP4_API nvfp4_status nvfp4_quantize(const void* x, int32_t x_dtype, int64_t R, int64_t C, int64_t ldx,
                            const nvfp4_qparams* params, const nvfp4_qtensor* out,
                            void* workspace, size_t workspace_bytes, uint32_t* dev_status,
                            void* stream);

/* Workspace bytes nvfp4_quantize_dual needs (two sets of amax partial maxima). */
NVFP4_API size_t nvfp4_quantize_dual_workspace_bytes(int64_t R, int64_t C);

/*
 * nvfp4_quantize_dual -- both quantizations a tensor needs in training, from
 * one amax read: the 1X16_ROW operand (params_row, out_row: [R, C]) and the
 * 1X16_COL operand (params_col, out_col: [C, R], with or without the RHT).  With
 * the RHT the single amax pass computes |x| and |RHT(x)| maxima together, and for
 * BF16 x with one rounding mode for both operands a single encode pass writes both
 * (x is read twice in all); results are identical to two nvfp4_quantize calls with
 * the same parameters.
 * Used for X (Fprop operand + the Wgrad operand saved for the backward pass) and
 * for dY (Dgrad + Wgrad operands).  Same argument rules as nvfp4_quantize.
 */
NVFP4_API nvfp4_status nvfp4_quantize_dual(const void* x, int32_t x_dtype, int64_t R, int64_t C, int64_t ldx,
                                           const nvfp4_qparams* params_row, const nvfp4_qtensor* out_row,
                                           const nvfp4_qparams* params_col, const nvfp4_qtensor* out_col,
                                           void* workspace, size_t workspace_bytes, uint32_t* dev_status,
                                           void* stream);

/*
 * nvfp4_quantize_dual_sqrelu -- nvfp4_quantize_dual of A = relu(H)^2 (the squared
 * ReLU of an MLP block, applied element by element to bf16 H: max(h, 0)^2 in fp32,
 * rounded to bf16) without A ever being stored: every pass applies the activation to
 * H as it is loaded.  Results are identical to nvfp4_sqrelu_forward followed by
 * nvfp4_quantize_dual.  BF16 input only (else NVFP4_ERR_UNSUPPORTED); arguments as
 * for nvfp4_quantize_dual, with H, its row pitch ldh and its shape [R, C].  Not on
 * the page, whose MLP activation is unspecified: a fusion of the block's two steps.
 */
NVFP4_API nvfp4_status nvfp4_quantize_dual_sqrelu(const void* h, int32_t h_dtype, int64_t R, int64_t C, int64_t ldh,
                                                  const nvfp4_qparams* params_row, const nvfp4_qtensor* out_row,
                                                  const nvfp4_qparams* params_col, const nvfp4_qtensor* out_col,
                                                  void* workspace, size_t workspace_bytes, uint32_t* dev_status,
                                                  void* stream);

/*
 * nvfp4_quantize_noalloc -- nvfp4_quantize without a workspace argument; it
 * allocates nothing.  The page describes no such call: it exists for callers
 * that can hand over their input and output buffers but cannot obtain one more
 * device buffer -- a plug-in that only sees the tensors its host framework
 * planned, or code running where an allocation would re-enter or break the
 * caller's allocator.
 *   Scratch: the amax pass's per-CTA partial maxima live in a static device
 *   array of 4096 uint32 (16 KB) inside this library, held on every device that
 *   loads the library until the process exits.  Calls needing more scratch than
 *   that are rejected with NVFP4_ERR_WORKSPACE (the amax grid is capped at 4096
 *   CTAs, so no tensor size needs more).
 *   Set-up: the first call in a CUDA context (normally a device's primary
 *   context) looks up the array's device address there (cudaGetSymbolAddress)
 *   and caches it under that context's id; make that first call before any
 *   stream capture.  A context created later (after cudaDeviceReset, say) gets
 *   its own lookup on its first call.
 *   Sharing: every call uses the same array; each amax CTA overwrites its own
 *   slot before the encode pass reads it, so nothing needs clearing between
 *   calls, but calls that overlap on the GPU (different streams, concurrently)
 *   race on the array and give wrong results.
 * Arguments, layouts, results and errors are otherwise those of nvfp4_quantize.
 */
NVFP4_API nvfp4_status nvfp4_quantize_noalloc(const void* x, int32_t x_dtype, int64_t R, int64_t C, int64_t ldx,
                                              const nvfp4_qparams* params, const nvfp4_qtensor* out,
                                              uint32_t* dev_status, void* stream);

/*
 * nvfp4_gemm -- D[M, N] = s_dec(A) * s_dec(B) * sum_k qA[m,k]*SA[m,k/16] * qB[n,k]*SB[n,k/16]
 * on the tcgen05 block-scaled FP4 tensor cores (fp32 accumulation in TMEM).
 *   A: [M, K] quantized along K (codes + scales_mma); B: [N, K] likewise.
 *   D: F32 or BF16, row pitch ldd elements (ldd >= N).
 * Rules: A->cols == B->cols == K, K % 32 == 0, M, N >= 1; codes 16-byte aligned.
 * M and N need not be tile multiples (edges are masked).
 */
NVFP4_API nvfp4_status nvfp4_gemm(const nvfp4_qtensor* A, const nvfp4_qtensor* B, void* D, int32_t d_dtype,
                        int64_t ldd, uint32_t* dev_status, void* stream);

/*
 * Bytes of the workspace nvfp4_gemm_ws uses on CUDA device `device` (partial sums for one
 * 256 x 256 fp32 tile per pair of multiprocessors, and a few counters); 0 if the device cannot
 * be queried.
 */
NVFP4_API size_t nvfp4_gemm_workspace_bytes(int32_t device);

/*
 * nvfp4_gemm_ws -- nvfp4_gemm that may balance the last, partial wave of output tiles over all
 * multiprocessors: when the tiles do not divide evenly among the SM pairs, the tiles of the
 * last wave are cut in two along K, computed by different SM pairs, whose fp32 partial sums
 * meet in `workspace` (an order-free sum of two; whichever half finishes second stores the
 * tile, and no SM waits for another).  NVFP4 operands, BF16 output through the CTA-pair
 * kernel; otherwise the call is nvfp4_gemm.  Results are deterministic; the split tiles' sums
 * are grouped differently from nvfp4_gemm's (a different fp32 rounding, well inside the GEMM's
 * error bound), the other tiles are identical to nvfp4_gemm's.  Same arguments as nvfp4_gemm,
 * plus: workspace -- device memory of at least nvfp4_gemm_workspace_bytes(current device)
 * bytes (else NVFP4_ERR_WORKSPACE), 16-byte aligned, zero-filled before its first use; every
 * call leaves it as the next call needs it, unless the call reports an error on dev_status, after
 * which it must be zero-filled again.  Calls that may run concurrently (other streams) need
 * workspaces of their own.  workspace NULL: exactly nvfp4_gemm.  Not on the page: a scheduling
 * choice for the page's three GEMMs [page ¶2, ¶3].
 */
NVFP4_API nvfp4_status nvfp4_gemm_ws(const nvfp4_qtensor* A, const nvfp4_qtensor* B, void* D, int32_t d_dtype,
                                     int64_t ldd, void* workspace, size_t workspace_bytes, uint32_t* dev_status,
                                     void* stream);

/*
 * nvfp4_gemm_sqrelu_bwd -- the Dgrad GEMM of a squared-ReLU MLP with the activation's
 * backward in its epilogue: with dA = bf16(s_dec(A) s_dec(B) sum_k qA qB) (what nvfp4_gemm
 * stores in BF16), D[m, n] = bf16(dA[m, n] * (H[m, n] > 0 ? 2 H[m, n] : +0)) in fp32 --
 * bit for bit nvfp4_gemm (CTA-pair kernel, BF16) followed by nvfp4_sqrelu_backward, without
 * writing and re-reading dA.  H and D: BF16 [M, N], row pitches ldh, ldd >= N elements,
 * bases and pitches 16-byte aligned (else NVFP4_ERR_ALIGNMENT).  A, B as for nvfp4_gemm.
 * Not on the page (its MLP activation is unspecified): a fusion of two steps of the MLP
 * block built around the page's Dgrad GEMM [page ¶2, ¶3].
 */
NVFP4_API nvfp4_status nvfp4_gemm_sqrelu_bwd(const nvfp4_qtensor* A, const nvfp4_qtensor* B, const void* H,
                                             int64_t ldh, void* D, int64_t ldd, uint32_t* dev_status,
                                             void* stream);

/*
 * nvfp4_gemm_sqrelu_bwd_maxima -- nvfp4_gemm_sqrelu_bwd whose epilogue also leaves the two
 * tensor maxima the dual quantization of its output dH needs (max|dH| and max|RHT(dH)| along
 * rows with the RHT sign vector of rht_seed), as nvfp4_gemm_sqrelu_maxima does for relu(H)^2;
 * nvfp4_quantize_dual_premax then quantizes dH without an amax read.  dH is identical to
 * nvfp4_gemm_sqrelu_bwd's.  Additional rules: maxima non-NULL, 4-byte aligned, maxima_bytes at
 * least nvfp4_sqrelu_maxima_bytes(current device) (else NVFP4_ERR_WORKSPACE); M % 16 == 0 and
 * N % 16 == 0.
 */
NVFP4_API nvfp4_status nvfp4_gemm_sqrelu_bwd_maxima(const nvfp4_qtensor* A, const nvfp4_qtensor* B, const void* H,
                                                    int64_t ldh, void* D, int64_t ldd, uint64_t rht_seed,
                                                    uint32_t* maxima, size_t maxima_bytes, uint32_t* dev_status,
                                                    void* stream);

/*
 * Bytes of the partial-maxima buffer the *_maxima GEMMs write on CUDA device `device`: two
 * halves (|x|, then |RHT(x)| / 4) of one uint32 partial per epilogue warp, eight warps per CTA
 * and at most one CTA per multiprocessor, so 2 * 8 * (multiprocessor count) * 4 bytes.  0 if the
 * device cannot be queried.  A buffer of B bytes is read as two halves of B / 8 partials.
 */
NVFP4_API size_t nvfp4_sqrelu_maxima_bytes(int32_t device);

/*
 * nvfp4_gemm_sqrelu_maxima -- the first GEMM of a squared-ReLU MLP with the next
 * quantization's tensor maxima in its epilogue: H = bf16(s_dec(A) s_dec(B) sum_k qA qB),
 * stored exactly as nvfp4_gemm (CTA-pair kernel, BF16) stores it, and, for A = relu(H)^2
 * as nvfp4_quantize_dual_sqrelu forms it, max|A| and max|RHT(A)| along rows (the RHT sign
 * vector of rht_seed) as partial maxima in `maxima` (maxima_bytes of device memory, at least
 * nvfp4_sqrelu_maxima_bytes(current device), else NVFP4_ERR_WORKSPACE; 4-byte aligned;
 * contents on entry ignored: the call writes every partial).  nvfp4_quantize_dual_sqrelu_premax
 * then needs no amax pass over H.  H: BF16 [M, N], pitch ldh >= N, base and pitch 16-byte
 * aligned; M % 16 == 0 and N % 16 == 0.  A, B as for nvfp4_gemm.  Not on the page: the tensor
 * amax of the next quantization [page ¶2: the FP32 per-tensor scale] taken where the tensor is
 * produced instead of in a pass of its own.
 */
NVFP4_API nvfp4_status nvfp4_gemm_sqrelu_maxima(const nvfp4_qtensor* A, const nvfp4_qtensor* B, void* H,
                                                int64_t ldh, uint64_t rht_seed, uint32_t* maxima,
                                                size_t maxima_bytes, uint32_t* dev_status, void* stream);

/*
 * nvfp4_quantize_dual_sqrelu_premax -- nvfp4_quantize_dual_sqrelu of H using the maxima that
 * nvfp4_gemm_sqrelu_maxima left for this same H (with rht_seed == params_col->rht_seed when
 * params_col->rht is set): only the two encode passes run, and the results are identical to
 * nvfp4_quantize_dual_sqrelu's.  BF16 H only (else NVFP4_ERR_UNSUPPORTED); no workspace;
 * maxima_bytes is the size the GEMM was given (two halves of maxima_bytes / 8 partials;
 * NVFP4_ERR_WORKSPACE if that is 0); other arguments as for nvfp4_quantize_dual_sqrelu.
 */
NVFP4_API nvfp4_status nvfp4_quantize_dual_sqrelu_premax(const void* h, int32_t h_dtype, int64_t R, int64_t C,
                                                         int64_t ldh, const nvfp4_qparams* params_row,
                                                         const nvfp4_qtensor* out_row,
                                                         const nvfp4_qparams* params_col,
                                                         const nvfp4_qtensor* out_col, const uint32_t* maxima,
                                                         size_t maxima_bytes, uint32_t* dev_status, void* stream);

/*
 * nvfp4_quantize_dual_premax -- nvfp4_quantize_dual of x using the maxima that
 * nvfp4_gemm_sqrelu_bwd_maxima left for this same x (rht_seed == params_col->rht_seed when
 * params_col->rht is set): only the two encode passes run; results identical to
 * nvfp4_quantize_dual's.  BF16 x only (else NVFP4_ERR_UNSUPPORTED); no workspace; maxima_bytes
 * as for nvfp4_quantize_dual_sqrelu_premax.
 */
NVFP4_API nvfp4_status nvfp4_quantize_dual_premax(const void* x, int32_t x_dtype, int64_t R, int64_t C, int64_t ldx,
                                                  const nvfp4_qparams* params_row, const nvfp4_qtensor* out_row,
                                                  const nvfp4_qparams* params_col, const nvfp4_qtensor* out_col,
                                                  const uint32_t* maxima, size_t maxima_bytes, uint32_t* dev_status,
                                                  void* stream);

/*
 * MXFP4 -- the earlier 4-bit microscaling format the page compares NVFP4 with
 * [page ¶3: at 8B parameters MXFP4 trails NVFP4 in loss and needs ~36% more
 * tokens].  The page gives no rules for it; these follow the OCP Microscaling
 * format: blocks of 32 elements along the quantized axis, one UE8M0 scale per
 * block X = 2^(code - 127) with code = floor(log2(amax_b)) - 2 + 127 clamped
 * to [0, 254] (0 for an all-zero block), element code = e2m1_rne_sat(x / X),
 * no tensor scale, no stochastic rounding.  Dequantized value: e2m1(code) * X.
 *
 * The operand uses nvfp4_qtensor with these meanings (s_dec, codes_t and
 * scales_mma_t are ignored):
 *   codes       [rows, cols/2] bytes, as for NVFP4;
 *   scales      UE8M0 codes, row-major [rows, cols/32].  May be NULL;
 *   scales_mma  the tile layout the MXFP4 GEMM reads: ceil(rows/128) x
 *               ceil(cols/256) tiles of 1024 bytes, tile (rb, kb) at byte
 *               ((rb * ceil(cols/256)) + kb) * 1024; inside a tile, row r,
 *               scale-column s (s = k/32) at ((s/4)%2)*512 + (r%32)*16 +
 *               ((r%128)/32)*4 + s%4.  Padding holds 0.  May be NULL.
 */
NVFP4_API size_t nvfp4_mx_scales_mma_bytes(int64_t rows, int64_t cols);

/*
 * nvfp4_mx_quantize -- MXFP4 quantization of x [R, C] (row pitch ldx elements,
 * F32 or BF16).  col = 0: blocks along C, the operand is [R, C]; col = 1:
 * blocks along R, the operand is x^T [C, R] (out->rows = C, out->cols = R).
 * Rules: the operand's cols % 32 == 0; x and its row pitch 32-byte aligned
 * (col = 0) or 16-byte aligned (col = 1); codes 16-byte aligned; with col = 1,
 * R <= 65535 * 64.  Non-finite input gives unspecified codes.  Asynchronous on
 * `stream`; nothing is allocated.
 */
NVFP4_API nvfp4_status nvfp4_mx_quantize(const void* x, int32_t x_dtype, int64_t R, int64_t C, int64_t ldx,
                                         int32_t col, const nvfp4_qtensor* out, void* stream);

/*
 * nvfp4_mx_gemm -- D[M, N] = sum_k qA[m,k]*XA[m,k/32] * qB[n,k]*XB[n,k/32] with
 * MXFP4 operands (scales_mma required) on the tcgen05 block-scaled FP4 tensor
 * cores (scale_vec::2X, UE8M0 scales, fp32 accumulation), CTA-pair kernel.
 * D: BF16 only (F32 gives NVFP4_ERR_UNSUPPORTED), base and pitch ldd 16-byte
 * aligned.  Other rules as for nvfp4_gemm.
 */
NVFP4_API nvfp4_status nvfp4_mx_gemm(const nvfp4_qtensor* A, const nvfp4_qtensor* B, void* D, int32_t d_dtype,
                                     int64_t ldd, uint32_t* dev_status, void* stream);

/* Workspace bytes for the three linear-layer calls below with these sizes. */
NVFP4_API size_t nvfp4_linear_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * Fprop [page ¶2]: Y[M, N] = X[M, K] . W^T.  X (F32/BF16, pitch ldx) is
 * quantized 1x16 along K with RNE; Wq is the 16X16-quantized weight ([N, K]).
 */
NVFP4_API nvfp4_status nvfp4_linear_fprop(const void* X, int32_t x_dtype, int64_t M, int64_t K, int64_t ldx,
                                const nvfp4_qtensor* Wq, void* Y, int32_t y_dtype, int64_t ldy,
                                void* workspace, size_t workspace_bytes, uint32_t* dev_status,
                                void* stream);

/*
 * Dgrad [page ¶2]: dX[M, K] = dY[M, N] . W.  dY is quantized 1x16 along N with
 * stochastic rounding (sr_seed, sr_offset); the weight operand is W^T from the
 * same 16X16 quantization (Wq->codes_t and Wq->scales_mma_t must be set).
 */
NVFP4_API nvfp4_status nvfp4_linear_dgrad(const void* dY, int32_t dy_dtype, int64_t M, int64_t N, int64_t lddy,
                                const nvfp4_qtensor* Wq, uint64_t sr_seed, uint32_t sr_offset,
                                void* dX, int32_t dx_dtype, int64_t lddx,
                                void* workspace, size_t workspace_bytes, uint32_t* dev_status,
                                void* stream);

/*
 * Wgrad [page ¶2]: dW[N, K] = dY^T . X.  Both operands are quantized 1x16 along
 * the token axis M after the 16x16 RHT with one shared sign vector (rht_seed);
 * dY^T with stochastic rounding (sr_seed, sr_offset), X^T with RNE.  M % 16 == 0.
 */
NVFP4_API nvfp4_status nvfp4_linear_wgrad(const void* dY, int32_t dy_dtype, int64_t lddy,
                                const void* X, int32_t x_dtype, int64_t ldx,
                                int64_t M, int64_t N, int64_t K,
                                uint64_t sr_seed, uint32_t sr_offset, uint64_t rht_seed,
                                void* dW, int32_t dw_dtype, int64_t lddw,
                                void* workspace, size_t workspace_bytes, uint32_t* dev_status,
                                void* stream);

/*
 * Squared-ReLU of the dense MLP block the NVFP4 linear layers sit in (the page's
 * model is a hybrid; the MLP block around them is the plain dense case).  bf16
 * [n] contiguous buffers, n % 8 == 0, 16-byte aligned; fp32 arithmetic rounded
 * to nearest-even bf16:  a = relu(h)^2;  dh = da * (2 * relu(h)).
 */
NVFP4_API nvfp4_status nvfp4_sqrelu_forward(const void* h, void* a, int64_t n, void* stream);
NVFP4_API nvfp4_status nvfp4_sqrelu_backward(const void* h, const void* da, void* dh, int64_t n, void* stream);

/* Synchronises `stream`, reads *dev_status and returns it as a status. */
NVFP4_API nvfp4_status nvfp4_status_query(const uint32_t* dev_status, void* stream);

/* Static string for a status code. */
NVFP4_API const char* nvfp4_status_string(int32_t status);

/* Upper bound, in nanoseconds, of every bounded pipeline wait in the GEMM
   (default 2e9).  Process-wide; for tests that exercise the timeout path. */
NVFP4_API void nvfp4_set_wait_timeout_ns(uint64_t ns);

/*
 * Diagnostics (not on the hot path).  They run the exact device routines the
 * kernels use, so tests can pin them element by element.
 *   nvfp4_debug_e4m3: out[i] = block-scale cast of v[i] (RNE, saturating).
 *   nvfp4_debug_e2m1: out[i] = E2M1 code of y[i]; round = RNE or SR (with the
 *                     16-bit random value R = r16[i], through the kernels'
 *                     stochastic-rounding conversion); for RNE, hw = 1 uses the
 *                     hardware conversion instead of the software rule.
 *   nvfp4_debug_philox: out[4*i..] = Philox4x32-10(ctr[4*i..], key) words.
 *   nvfp4_selftest_wait_timeout: one CTA waits on an mbarrier nobody arrives
 *                     at, bounded by timeout_ns; sets *dev_status to
 *                     NVFP4_ERR_TIMEOUT and returns normally.
 */
NVFP4_API nvfp4_status nvfp4_debug_e4m3(const float* v, int64_t n, uint8_t* out, void* stream);
NVFP4_API nvfp4_status nvfp4_debug_e2m1(const float* y, const uint32_t* r16, int64_t n, int32_t round, int32_t hw,
                              uint8_t* out, void* stream);
NVFP4_API nvfp4_status nvfp4_debug_philox(const uint32_t* ctr, int64_t n, uint64_t key, uint32_t* out, void* stream);
NVFP4_API nvfp4_status nvfp4_selftest_wait_timeout(uint64_t timeout_ns, uint32_t* dev_status, void* stream);
/* GEMM kernel choice, process-wide, for tests: 0 = automatic (the CTA-pair
   kernel for bf16 outputs with at least one 256 x 256 tile per SM pair, else
   the single-CTA kernel), 1 = always single-CTA, 2 = CTA-pair wherever its
   epilogue applies (bf16, 16-byte aligned output). */
NVFP4_API void nvfp4_gemm_force_path(int32_t path);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_GB300_H */
