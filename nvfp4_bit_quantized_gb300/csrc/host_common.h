// host_common.h -- host-side helpers shared by the C-ABI translation units.
#pragma once

#include <algorithm>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/nvfp4.h"

namespace nvfp4 {

// Partial maxima a producing GEMM epilogue leaves for the quantizer (nvfp4_gemm_sqrelu_maxima):
// one per epilogue warp (eight per CTA, at most one CTA per SM), for |A| then for |RHT(A)| / 4.
// A buffer of B bytes holds two halves of B / 8 partials each.
constexpr int kMaximaWarpsPerCta = 8;

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launches a library kernel with programmatic stream serialization: it may be scheduled while
// the previous kernel in the stream drains, overlapping its launch and prologue with that
// kernel's tail.  Every kernel of the library lets its successor launch at once
// (griddepcontrol.launch_dependents) and waits for its predecessor to complete, with its
// writes visible (griddepcontrol.wait), before it reads or writes global memory; after a
// kernel launched without the attribute the wait returns at once.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Multiprocessor count of `dev`, cached (152 on GB300).
int sm_count(int dev);

// Process-wide bound of the GEMM's pipeline waits, in ns.
uint64_t wait_timeout_ns();

nvfp4_status quantize_impl(const void* x, int32_t x_dtype, int64_t R, int64_t C, int64_t ldx,
                           const nvfp4_qparams* p, const nvfp4_qtensor* out, void* ws, size_t ws_bytes,
                           uint32_t* dev_status, cudaStream_t stream);

// ws: optional split-tail workspace (nvfp4_gemm_ws), NULL for tile-by-tile work.
nvfp4_status gemm_impl(const nvfp4_qtensor* A, const nvfp4_qtensor* B, void* D, int32_t d_dtype, int64_t ldd,
                       uint32_t* dev_status, cudaStream_t stream, void* ws = nullptr, size_t ws_bytes = 0);

}  // namespace nvfp4
