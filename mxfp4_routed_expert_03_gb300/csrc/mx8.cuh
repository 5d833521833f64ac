// Two-term MXFP8 (E4M3) split of activations, used as the B operand of the
// block-scaled tensor-core GEMMs.
//
// A block of 32 values v (one E8M0 scale each term) is written as
//   v ~= hi * 2^s_hi + lo * 2^s_lo,   hi, lo in E4M3,
// where s_hi is the smallest exponent with max|v| / 2^s_hi <= 448 (E4M3's
// largest finite value, so nothing saturates), hi = RN_e4m3(v / 2^s_hi), and
// lo quantises the exact residual v - hi * 2^s_hi the same way. Two E4M3
// terms carry about 8 significant bits, the precision of bf16, which keeps
// the tensor-core path within the layer's output tolerance while the weights
// stay E2M1.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace mx8 {

// Exponent s with amax / 2^s <= 448 and s minimal (amax > 0 finite); clamped
// to the E8M0 range [-127, 127]. amax == 0 gives -127.
__device__ __forceinline__ int scale_exp(float amax) {
    uint32_t b = __float_as_uint(amax);
    int e = (int)((b >> 23) & 0xFF);
    if (e == 0) return -127;                 // zero or fp32 subnormal: smallest scale
    if (e == 255) return 127;                // inf / nan: largest scale
    int E = e - 127;                         // amax = 1.m * 2^E
    int s = (b & 0x7FFFFF) > 0x600000 ? E - 7 : E - 8;  // 448 = 1.75 * 2^8
    return s < -127 ? -127 : (s > 127 ? 127 : s);
}

__device__ __forceinline__ float exp2i(int s) {  // 2^s for s in [-127, 127]
    if (s >= -126) return __uint_as_float((uint32_t)(s + 127) << 23);
    return __uint_as_float(0x00400000u);          // 2^-127
}

// Round two fp32 values to E4M3 (satfinite), packed: a in the low byte.
__device__ __forceinline__ uint32_t to_e4m3x2(float a, float b) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
    return r;
}

// Decode two packed E4M3 (low byte first) to fp32.
__device__ __forceinline__ float2 from_e4m3x2(uint32_t v) {
    uint32_t h;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}"
        : "=r"(h)
        : "r"(v));
    __half2 hh = *reinterpret_cast<__half2 *>(&h);
    return __half22float2(hh);
}

}  // namespace mx8

// MXFP4 activations (the FP4 x FP4 mode): E2M1 elements with one E8M0 scale
// per 32 values, converted as OCP MX v1.0 specifies (section 6.3): the scale
// is 2^(floor(log2(amax)) - 2), 2 being the largest exponent of E2M1, and
// each element v / scale rounds to the nearest E2M1 value, ties to even,
// magnitudes above 6 clamped to 6.
namespace mx4 {

// floor(log2(amax)) - 2 for amax > 0 finite, clamped to the E8M0 range
// [-127, 127]; -127 for zero.
__device__ __forceinline__ int scale_exp(float amax) {
    const uint32_t b = __float_as_uint(amax);
    const int e = (int)((b >> 23) & 0xFF);
    const uint32_t mant = b & 0x7FFFFF;
    int fl;
    if (e == 255) return 127;
    if (e == 0) {
        if (mant == 0) return -127;
        fl = (31 - __clz((int)mant)) - 149;  // subnormal: leading bit of the mantissa
    } else {
        fl = e - 127;
    }
    const int s = fl - 2;
    return s < -127 ? -127 : (s > 127 ? 127 : s);
}

// Two fp32 values to one byte of E2M1 codes (round to nearest even,
// saturating): lo in the low nibble, hi in the high nibble.
__device__ __forceinline__ uint32_t to_e2m1x2(float lo, float hi) {
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r;
}

}  // namespace mx4
