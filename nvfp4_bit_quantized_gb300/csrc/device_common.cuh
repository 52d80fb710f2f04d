// device_common.cuh -- device-side building blocks of the NVFP4 quantizers and GEMM
// (sm_103a): bf16 unpacking, the E4M3 block-scale cast, E2M1 element encoding
// (round-to-nearest-even and stochastic), the squared ReLU on packed bf16, Philox4x32-10,
// the 16-point Hadamard butterflies, and bounded mbarrier waits.
//
// Method: news page "NVIDIA NVFP4 paper: 4-bit pretrain hits FP8 parity (12B,
// 10T tokens)" (zubnet.ai), ¶2.  The readings this file implements where the
// page is silent are listed in include/nvfp4.h.
#pragma once

#include <cstdint>
#include <cfloat>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include "../../include/nvfp4.h"

namespace nvfp4 {

// ----------------------------------------------------------------------------
// Device status word: the first error wins.
// ----------------------------------------------------------------------------
__device__ __forceinline__ void set_status(uint32_t* dev_status, uint32_t code) {
    if (dev_status) atomicCAS(dev_status, 0u, code);
}

// ----------------------------------------------------------------------------
// bf16 / fp32 element access.  A 16-byte chunk holds 8 bf16 or 4 fp32 values.
// ----------------------------------------------------------------------------
// Programmatic dependent launch (see launch_pdl): the successor kernel may launch now, and
// this kernel waits until its predecessor has completed and its writes are visible.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// 32-byte streaming load (the address must be 32-byte aligned).
__device__ __forceinline__ void ld_stream32(const void* p, uint32_t (&w)[8]) {
    asm volatile("ld.global.nc.L1::no_allocate.v8.u32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
                 : "l"(p));
}

template <typename T> struct Vec;
template <> struct Vec<uint16_t> {           // bf16 bits
    static constexpr int N = 8;
    __device__ __forceinline__ static void unpack(const uint4& v, float* f) {
        f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
        f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
    }
};
template <> struct Vec<float> {
    static constexpr int N = 4;
    __device__ __forceinline__ static void unpack(const uint4& v, float* f) {
        f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
    }
};

// ----------------------------------------------------------------------------
// Tensor and block scales (readings: s_enc = 2688 / amax_t; S_b = e4m3(amax_b/6 * s_enc);
// e_b = s_enc / S_b).  Every operation is one IEEE fp32 op with round-to-nearest.
// ----------------------------------------------------------------------------
__device__ __forceinline__ float tensor_s_enc(float amax_t) {
    if (amax_t == 0.0f) return 1.0f;
    return fminf(__fdiv_rn(2688.0f, amax_t), FLT_MAX);
}

// E4M3 cast with round-to-nearest-even and saturation to +-448 (cvt.rn.satfinite).
__device__ __forceinline__ uint32_t e4m3_rn_sat(float v) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
    return r & 0xFFu;                         // second source lands in the low byte
}

// Exact E4M3 -> fp32 via the hardware e4m3 -> f16 conversion.
__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
    uint32_t h2;
    uint16_t in = (uint16_t)code;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// RN(a / 6) by the published correction step for division by a reciprocal
// (P. Markstein, "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Dev. 34, 1990; for a divisor known in advance, N. Brisebarre,
// J.-M. Muller, S. K. Raina, IEEE Trans. Computers 53(8), 2004): q0 = RN(a * RN(1/6)),
// the exact remainder r = a - 6 q0 from one fma, q = RN(q0 + r * RN(1/6)).  Three
// instructions instead of the general division.  The result is the correctly rounded
// quotient for every positive finite bf16 value and for every fp32 a >= 6 * 2^-126
// (a normal quotient); below that the quotient is subnormal and the step can miss by
// one unit, so div6_rn falls back to the IEEE division there.  Both claims are checked
// in exact arithmetic on the host, over every bf16 value and every fp32 significand.
__device__ __forceinline__ float div6_correction(float a) {
    const float inv6 = __uint_as_float(0x3E2AAAABu);        // RN(1/6)
    const float q0 = __fmul_rn(a, inv6);
    const float r = __fmaf_rn(-q0, 6.0f, a);
    return __fmaf_rn(r, inv6, q0);
}
__device__ __forceinline__ float div6_rn(float a) {
    return a >= 0x1.8p-124f ? div6_correction(a) : __fdiv_rn(a, 6.0f);   // 0x1.8p-124 = 6 * 2^-126
}

__device__ __forceinline__ uint32_t block_scale_code(float amax_b, float s_enc) {
    return e4m3_rn_sat(__fmul_rn(div6_rn(amax_b), s_enc));
}
__device__ __forceinline__ uint32_t block_scale_code_bf16(float amax_b, float s_enc) {
    return e4m3_rn_sat(__fmul_rn(div6_correction(amax_b), s_enc));
}

__device__ __forceinline__ float block_multiplier(uint32_t sb_code, float s_enc) {
    float sb = e4m3_to_f32(sb_code);
    if (sb == 0.0f) return 0.0f;
    return fminf(__fdiv_rn(s_enc, sb), FLT_MAX);
}

// ----------------------------------------------------------------------------
// E2M1 element encode.
// Round-to-nearest-even: count the grid midpoints below |y|; at a midpoint the
// even code wins (strict '>' where the lower code is even, '>=' where the upper
// one is).  |y| > 5 saturates to code 7 (6.0).  The sign bit is that of y.
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t e2m1_rne_sw(float y) {
    float a = fabsf(y);
    uint32_t c = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) +
                 (a > 2.5f) + (a >= 3.5f) + (a > 5.0f);
    return c | ((__float_as_uint(y) >> 28) & 8u);
}

// Hardware conversion of two fp32 values to an E2M1 pair (first source in the
// high nibble).  cvt.rn.satfinite.e2m1x2 rounds to nearest-even, saturates to 6
// and keeps the sign of zero: exactly the rule above (pinned against the oracle
// element by element), so the kernels use it.
__device__ __forceinline__ uint32_t e2m1x2_hw(float hi, float lo) {
    uint32_t out;
    asm("{\n\t.reg .b8 t;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
        "cvt.u32.u8 %0, t;\n\t}"
        : "=r"(out) : "f"(hi), "f"(lo));
    return out;
}

// Eight values -> eight E2M1 codes, element k in nibble k (hardware conversion).
__device__ __forceinline__ uint32_t e2m1x8_rn(const float (&y)[8]) {
    uint32_t out;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(out)
        : "f"(y[0]), "f"(y[1]), "f"(y[2]), "f"(y[3]), "f"(y[4]), "f"(y[5]), "f"(y[6]), "f"(y[7]));
    return out;
}

// Sixteen values -> 64 bits of codes (round to nearest even).
__device__ __forceinline__ uint2 e2m1x16_rn(const float (&y)[16]) {
    return make_uint2(e2m1x8_rn(*reinterpret_cast<const float (*)[8]>(&y[0])),
                      e2m1x8_rn(*reinterpret_cast<const float (*)[8]>(&y[8])));
}

// Four values -> four codes in the low 16 bits.
__device__ __forceinline__ uint32_t e2m1x4_rn(const float (&y)[4]) {
    uint32_t out;
    asm("{\n\t.reg .b8 b0, b1;\n\t.reg .b16 h;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "mov.b16 h, {b0, b1};\n\t"
        "cvt.u32.u16 %0, h;\n\t}"
        : "=r"(out) : "f"(y[0]), "f"(y[1]), "f"(y[2]), "f"(y[3]));
    return out;
}

// Stochastic rounding of four values to E2M1 codes with Blackwell's conversion
// (cvt.rs.satfinite.e2m1x4.f32), value k in nibble k.  The rule, pinned element
// by element against the oracle: |y| goes up to the next grid point iff
// p + R * 2^-16 >= 1, p its position between the two neighbours, R a 16-bit
// random value; |y| >= 6 saturates; the sign of y is kept.  The conversion takes
// the four R from one 32-bit word: with A = bits 16-23 : bits 0-7 and
// B = bits 24-31 : bits 8-15, value 0 uses A, value 1 A bit-reversed, value 2 B,
// value 3 B bit-reversed -- the layout the SR random bits are defined in.
__device__ __forceinline__ uint32_t e2m1x4_sr(float y0, float y1, float y2, float y3, uint32_t rbits) {
    uint16_t d;
    asm("cvt.rs.satfinite.e2m1x4.f32 %0, {%1, %2, %3, %4}, %5;"      // first source -> top nibble
        : "=h"(d) : "f"(y3), "f"(y2), "f"(y1), "f"(y0), "r"(rbits));
    return d;
}

// Sixteen values -> 64 bits of codes, stochastic rounding with the four words of one Philox call.
__device__ __forceinline__ uint2 e2m1x16_sr(const float (&y)[16], const uint32_t (&w)[4]) {
    return make_uint2(e2m1x4_sr(y[0], y[1], y[2], y[3], w[0]) | (e2m1x4_sr(y[4], y[5], y[6], y[7], w[1]) << 16),
                      e2m1x4_sr(y[8], y[9], y[10], y[11], w[2]) | (e2m1x4_sr(y[12], y[13], y[14], y[15], w[3]) << 16));
}

// ----------------------------------------------------------------------------
// Packed bf16 / fp32x2 helpers shared by the quantizers and the GEMM epilogue.
// ----------------------------------------------------------------------------
// Squared ReLU of two packed bf16 values, rounded back to bf16: relu(h)^2 in fp32, one
// rounding to bf16 (max(h, 0) squares to +0 for h <= 0, -0 and NaN alike).  The MLP's
// activation, applied to H as it is loaded, so A = relu(H)^2 is quantized without being
// stored (SQR kernels).
__device__ __forceinline__ uint32_t sqrelu_bf16x2(uint32_t w) {
    const float2 r = make_float2(fmaxf(__uint_as_float(w << 16), 0.0f), fmaxf(__uint_as_float(w & 0xFFFF0000u), 0.0f));
    const __nv_bfloat162 b = __float22bfloat162_rn(__fmul2_rn(r, r));
    return *reinterpret_cast<const uint32_t*>(&b);
}

// The 16-point Hadamard butterflies of two columns at once, unnormalised (the 1/4 of
// the transform is applied by the caller): h = 1, 2, 4, 8, lower index first,
// (t_i, t_{i+h}) <- (t_i + t_{i+h}, t_i - t_{i+h}), each one fp32 RN operation.
__device__ __forceinline__ void hadamard16_x2(float2 (&t)[16]) {
    const float2 neg1 = make_float2(-1.0f, -1.0f);
#pragma unroll
    for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if ((i & h) == 0) {
                const float2 a = t[i], b = t[i + h];
                t[i] = __fadd2_rn(a, b);
                t[i + h] = __ffma2_rn(b, neg1, a);           // a - b, one rounding
            }
        }
    }
}


// ----------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of two 32x32->64
// multiplies and xors on a 4-word counter, with a 2-word key advanced by the
// Weyl increments between rounds.
// ----------------------------------------------------------------------------
struct Philox4 { uint32_t w[4]; };

// The ten round keys.  The quantizers get them as a kernel parameter, computed on the host, so
// each round's xor reads its key straight from the parameter bank.
struct PhiloxKey { uint32_t k0[10], k1[10]; };

__host__ __device__ __forceinline__ PhiloxKey philox_key(uint64_t seed) {
    PhiloxKey k;
    uint32_t a = (uint32_t)seed, b = (uint32_t)(seed >> 32);
#pragma unroll
    for (int i = 0; i < 10; ++i) { k.k0[i] = a; k.k1[i] = b; a += 0x9E3779B9u; b += 0xBB67AE85u; }
    return k;
}

__device__ __forceinline__ Philox4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                                 const PhiloxKey& key) {
#pragma unroll
    for (int i = 0; i < 10; ++i) {
        // low and high halves of the two 32x32 products as separate multiplies
        // (measured slightly faster than one 64-bit product each)
        const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
        const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
        const uint32_t n0 = hi1 ^ c1 ^ key.k0[i];
        const uint32_t n2 = hi0 ^ c3 ^ key.k1[i];
        c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
    }
    Philox4 r;
    r.w[0] = c0; r.w[1] = c1; r.w[2] = c2; r.w[3] = c3;
    return r;
}

__device__ __forceinline__ Philox4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                                 uint32_t k0, uint32_t k1) {
    return philox4x32_10(c0, c1, c2, c3, philox_key(((uint64_t)k1 << 32) | k0));
}

// The random bits of elements 16g .. 16g+15 come from one call with counter
// (lo32 g, hi32 g, stream, offset); word k serves elements 16g+4k .. 16g+4k+3.
__device__ __forceinline__ Philox4 sr_philox(const PhiloxKey& key, uint32_t stream, uint32_t offset, uint64_t group) {
    return philox4x32_10((uint32_t)group, (uint32_t)(group >> 32), stream, offset, key);
}

// RHT sign vector: s_j = -1 iff bit j of word 0 of Philox(key = seed, counter = 0).
__device__ __forceinline__ uint32_t rht_sign_mask(uint64_t seed) {
    return philox4x32_10(0u, 0u, 0u, 0u, (uint32_t)seed, (uint32_t)(seed >> 32)).w[0] & 0xFFFFu;
}

// ----------------------------------------------------------------------------
// 16-point randomized Hadamard: t = s .* v; butterflies h = 1, 2, 4, 8 with
// (t_i, t_{i+h}) <- (t_i + t_{i+h}, t_i - t_{i+h}); y = t / 4.
// ----------------------------------------------------------------------------
__device__ __forceinline__ void rht16(float* t, uint32_t sign_mask) {
#pragma unroll
    for (int j = 0; j < 16; ++j) t[j] = ((sign_mask >> j) & 1u) ? -t[j] : t[j];
#pragma unroll
    for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if ((i & h) == 0) {
                const float a = t[i], b = t[i + h];
                t[i] = __fadd_rn(a, b);
                t[i + h] = __fsub_rn(a, b);
            }
        }
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) t[j] = __fmul_rn(t[j], 0.25f);
}

// ----------------------------------------------------------------------------
// Shared-memory mbarrier helpers with bounded waits.
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for the phase with parity `parity` of `bar` to complete.  Gives up when
// *abort becomes non-zero (another role gave up; abort may be null) or after
// timeout_ns; on a timeout it records NVFP4_ERR_TIMEOUT and raises *abort.
// Returns true on success.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t timeout_ns,
                                                  volatile uint32_t* abort, uint32_t* dev_status) {
    const uint32_t a = smem_addr(bar);
    if (mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(a, parity)) return true;
        if ((it & 63u) == 0) {
            if (abort && *abort) return false;
            if (global_ns() - t0 > timeout_ns) {
                set_status(dev_status, NVFP4_ERR_TIMEOUT);
                if (abort) *abort = 1u;
                return false;
            }
        }
    }
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_addr(bar)), "r"(bytes) : "memory");
}

}  // namespace nvfp4
