// Device encoders for the block formats of the MoE step (MXFP8: E4M3 + E8M0 per 32;
// MXFP4: E2M1 + E8M0 per 32; NVFP4: E2M1 + E4M3 per 16 with an fp32 global scale). All arithmetic that decides a
// code is IEEE fp32 with explicit rounding (no contraction), so the codes equal those
// of any other exact fp32 implementation of the same rule.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

namespace moe {

// Round-to-nearest-even, saturating E4M3 of two values: returns (hi << 8) | lo.
__device__ __forceinline__ uint16_t e4m3x2(float hi, float lo) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ uint8_t e4m3(float v) { return (uint8_t)(e4m3x2(0.0f, v) & 0xFF); }

// Round-to-nearest-even, saturating E2M1 of two values: returns (hi << 4) | lo.
__device__ __forceinline__ uint8_t e2m1x2(float hi, float lo) {
    uint32_t r;
    asm("{\n\t.reg .b8 q;\n\tcvt.rn.satfinite.e2m1x2.f32 q, %1, %2;\n\tcvt.u32.u8 %0, q;\n\t}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return (uint8_t)r;
}

// Exact fp32 value of an E4M3 byte (NaN pattern not produced here).
__device__ __forceinline__ float e4m3_to_f32(uint8_t b) {
    const uint32_t e = (b >> 3) & 15u, m = b & 7u;
    float v = (e == 0) ? (float)m * 0.001953125f : __uint_as_float(((e + 120u) << 23) | (m << 20));
    return (b & 0x80) ? -v : v;
}

// Exact 2^p for p in [-127, 127] (2^-127 is an fp32 subnormal).
__device__ __forceinline__ float exp2_int(int p) {
    return (p >= -126) ? __uint_as_float((uint32_t)(p + 127) << 23) : __uint_as_float(0x00400000u);
}

// MXFP8 block exponent: the smallest e in [-127, 127] with amax <= 448 * 2^e
// (448 = 1.75 * 2^8): e = E - 8, plus one when amax's significand exceeds 1.75.
__device__ __forceinline__ int mx_exponent(float amax) {
    if (!(amax > 0.0f)) return -127;
    const uint32_t u = __float_as_uint(amax);
    int E = (int)((u >> 23) & 0xFF) - 127;
    int e = E - 8 + (((u & 0x7FFFFFu) > 0x600000u) ? 1 : 0);
    if ((u >> 23) == 0) e = -127;  // subnormal amax
    return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// MXFP4 block exponent: the smallest e in [-127, 127] with amax <= 6 * 2^e (6 = 1.5 * 2^2):
// e = E - 2, plus one when amax's significand exceeds 1.5.
__device__ __forceinline__ int mx4_exponent(float amax) {
    if (!(amax > 0.0f)) return -127;
    const uint32_t u = __float_as_uint(amax);
    int E = (int)((u >> 23) & 0xFF) - 127;
    int e = E - 2 + (((u & 0x7FFFFFu) > 0x400000u) ? 1 : 0);
    if ((u >> 23) == 0) e = -127;  // subnormal amax
    return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// NVFP4 block scale byte: E4M3(amax / (6 * gs)).
__device__ __forceinline__ uint8_t nv_scale(float amax, float gs) {
    return e4m3(__fdiv_rn(amax, __fmul_rn(6.0f, gs)));
}

}  // namespace moe
