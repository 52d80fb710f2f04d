// activation.cu -- squared-ReLU for the dense MLP block around the NVFP4 linear
// layers (bf16 in / out, fp32 arithmetic, round-to-nearest-even to bf16):
//   forward   a  = relu(h)^2
//   backward  dh = da * (2 * relu(h))
// with relu(h) = h if h > 0 else +0 (so signed zeros are reproducible).
// Memory-bound elementwise kernels with 16-byte accesses.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "device_common.cuh"
#include "host_common.h"

namespace nvfp4 {
namespace {

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__global__ void sqrelu_fwd_kernel(const uint4* __restrict__ h, uint4* __restrict__ a, int64_t n8) {
    pdl_launch_dependents();
    pdl_wait();
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 v = ld_stream(h + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float l = bf16_lo(w[k]), u = bf16_hi(w[k]);
            const float lo = l > 0.0f ? l : 0.0f, hi = u > 0.0f ? u : 0.0f;
            o[k] = pack_bf16x2(__fmul_rn(lo, lo), __fmul_rn(hi, hi));
        }
        a[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

__global__ void sqrelu_bwd_kernel(const uint4* __restrict__ h, const uint4* __restrict__ da, uint4* __restrict__ dh,
                                  int64_t n8) {
    pdl_launch_dependents();
    pdl_wait();
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 hv = ld_stream(h + i), gv = ld_stream(da + i);
        const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float l = bf16_lo(hw[k]), u = bf16_hi(hw[k]);
            const float tlo = l > 0.0f ? __fmul_rn(2.0f, l) : 0.0f, thi = u > 0.0f ? __fmul_rn(2.0f, u) : 0.0f;
            o[k] = pack_bf16x2(__fmul_rn(bf16_lo(gw[k]), tlo), __fmul_rn(bf16_hi(gw[k]), thi));
        }
        dh[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

int grid_for(int64_t n8) {
    int dev = 0;
    cudaGetDevice(&dev);
    const int64_t g = std::min<int64_t>((n8 + 255) / 256, (int64_t)sm_count(dev) * 8);
    return (int)std::max<int64_t>(1, g);
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" nvfp4_status nvfp4_sqrelu_forward(const void* h, void* a, int64_t n, void* stream) {
    if (n < 0 || n % 8 != 0) return NVFP4_ERR_SHAPE;
    if (n == 0) return NVFP4_OK;
    if (!h || !a) return NVFP4_ERR_INVALID_ARG;
    if (!aligned16(h) || !aligned16(a)) return NVFP4_ERR_ALIGNMENT;
    const cudaError_t e = launch_pdl(sqrelu_fwd_kernel, dim3(grid_for(n / 8)), dim3(256), 0,
                                     static_cast<cudaStream_t>(stream), static_cast<const uint4*>(h),
                                     static_cast<uint4*>(a), n / 8);
    return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

extern "C" nvfp4_status nvfp4_sqrelu_backward(const void* h, const void* da, void* dh, int64_t n, void* stream) {
    if (n < 0 || n % 8 != 0) return NVFP4_ERR_SHAPE;
    if (n == 0) return NVFP4_OK;
    if (!h || !da || !dh) return NVFP4_ERR_INVALID_ARG;
    if (!aligned16(h) || !aligned16(da) || !aligned16(dh)) return NVFP4_ERR_ALIGNMENT;
    const cudaError_t e = launch_pdl(sqrelu_bwd_kernel, dim3(grid_for(n / 8)), dim3(256), 0,
                                     static_cast<cudaStream_t>(stream), static_cast<const uint4*>(h),
                                     static_cast<const uint4*>(da), static_cast<uint4*>(dh), n / 8);
    return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}
