// capi.cu -- status handling, process-wide settings, diagnostics and the
// bounded-wait self-test of the NVFP4 library.
#include <cuda_runtime.h>
#include <atomic>
#include <cstdint>
#include <mutex>

#include "device_common.cuh"
#include "host_common.h"

namespace nvfp4 {

namespace {
std::atomic<uint64_t> g_timeout_ns{2000000000ull};
std::mutex g_sm_mutex;
int g_sm_cache[64] = {0};
}  // namespace

int sm_count(int dev) {
    if (dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lk(g_sm_mutex);
    if (g_sm_cache[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        g_sm_cache[dev] = v;
    }
    return g_sm_cache[dev];
}

uint64_t wait_timeout_ns() { return g_timeout_ns.load(); }

__global__ void debug_e4m3_kernel(const float* v, int64_t n, uint8_t* out) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        out[i] = (uint8_t)e4m3_rn_sat(v[i]);
}

__global__ void debug_e2m1_kernel(const float* y, const uint32_t* r16, int64_t n, int round, int hw, uint8_t* out) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        uint32_t c;
        if (round == NVFP4_ROUND_SR) {
            // value 0 of the four-wide conversion draws R from bits 16-23 : bits 0-7
            const uint32_t r = r16[i] & 0xFFFFu;
            c = e2m1x4_sr(y[i], 0.0f, 0.0f, 0.0f, ((r >> 8) << 16) | (r & 0xFFu)) & 0xFu;
        }
        else if (hw) c = e2m1x2_hw(0.0f, y[i]) & 0xFu;
        else c = e2m1_rne_sw(y[i]);
        out[i] = (uint8_t)c;
    }
}

__global__ void debug_philox_kernel(const uint32_t* ctr, int64_t n, uint64_t key, uint32_t* out) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const Philox4 p = philox4x32_10(ctr[4 * i], ctr[4 * i + 1], ctr[4 * i + 2], ctr[4 * i + 3],
                                        (uint32_t)key, (uint32_t)(key >> 32));
        for (int k = 0; k < 4; ++k) out[4 * i + k] = p.w[k];
    }
}

// One thread waits on a barrier that expects one arrival nobody makes.
__global__ void selftest_wait_kernel(uint64_t timeout_ns, uint32_t* dev_status) {
    __shared__ uint64_t bar;
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait_bounded(&bar, 0u, timeout_ns, &abort_flag, dev_status);
    __syncthreads();
}

inline int grid_for(int64_t n) {
    int64_t g = (n + 255) / 256;
    return (int)std::max<int64_t>(1, std::min<int64_t>(g, 4096));
}

}  // namespace nvfp4

using namespace nvfp4;

extern "C" const char* nvfp4_status_string(int32_t s) {
    switch (s) {
        case NVFP4_OK: return "ok";
        case NVFP4_ERR_INVALID_ARG: return "invalid argument";
        case NVFP4_ERR_SHAPE: return "shape breaks the block or tile rules";
        case NVFP4_ERR_ALIGNMENT: return "pointer or pitch not 16-byte aligned";
        case NVFP4_ERR_WORKSPACE: return "workspace missing or too small";
        case NVFP4_ERR_UNSUPPORTED: return "unsupported";
        case NVFP4_ERR_CUDA: return "CUDA runtime error";
        case NVFP4_ERR_NONFINITE: return "non-finite tensor amax";
        case NVFP4_ERR_TIMEOUT: return "bounded pipeline wait timed out";
        default: return "unknown status";
    }
}

extern "C" nvfp4_status nvfp4_status_query(const uint32_t* dev_status, void* stream) {
    if (!dev_status) return NVFP4_ERR_INVALID_ARG;
    uint32_t h = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&h, dev_status, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess) return NVFP4_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return NVFP4_ERR_CUDA;
    return static_cast<nvfp4_status>(h);
}

extern "C" void nvfp4_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns ? ns : 1ull); }

extern "C" nvfp4_status nvfp4_debug_e4m3(const float* v, int64_t n, uint8_t* out, void* stream) {
    if (n < 0 || (n > 0 && (!v || !out))) return NVFP4_ERR_INVALID_ARG;
    if (n == 0) return NVFP4_OK;
    debug_e4m3_kernel<<<grid_for(n), 256, 0, static_cast<cudaStream_t>(stream)>>>(v, n, out);
    return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

extern "C" nvfp4_status nvfp4_debug_e2m1(const float* y, const uint32_t* r16, int64_t n, int32_t round, int32_t hw,
                                         uint8_t* out, void* stream) {
    if (n < 0 || (n > 0 && (!y || !out))) return NVFP4_ERR_INVALID_ARG;
    if (round == NVFP4_ROUND_SR && n > 0 && !r16) return NVFP4_ERR_INVALID_ARG;
    if (n == 0) return NVFP4_OK;
    debug_e2m1_kernel<<<grid_for(n), 256, 0, static_cast<cudaStream_t>(stream)>>>(y, r16, n, round, hw, out);
    return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

extern "C" nvfp4_status nvfp4_debug_philox(const uint32_t* ctr, int64_t n, uint64_t key, uint32_t* out, void* stream) {
    if (n < 0 || (n > 0 && (!ctr || !out))) return NVFP4_ERR_INVALID_ARG;
    if (n == 0) return NVFP4_OK;
    debug_philox_kernel<<<grid_for(n), 256, 0, static_cast<cudaStream_t>(stream)>>>(ctr, n, key, out);
    return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

extern "C" nvfp4_status nvfp4_selftest_wait_timeout(uint64_t timeout_ns, uint32_t* dev_status, void* stream) {
    if (!dev_status) return NVFP4_ERR_INVALID_ARG;
    if (timeout_ns == 0 || timeout_ns > 10000000000ull) return NVFP4_ERR_INVALID_ARG;
    selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(timeout_ns, dev_status);
    return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}
