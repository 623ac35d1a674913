// convert.cuh -- exact element conversions of the integer routes, shared by
// the operand-conversion kernels (convert.cu) and the GEMM kernel's in-ring
// conversion (gemm_tc.cu).
//   s8 in [-128, 127] -> binary16 (11-bit significand: exact up to 2048)
//   s4 in [-8, 7]     -> E4M3 (4-bit significand: exact up to 16)
#pragma once

#include <cstdint>

#include <cuda_fp16.h>

namespace ptc {

// ---------------------------------------------------------------- s8 -> f16
// Four int8 lanes -> four binary16 lanes without a conversion per element:
// flipping the sign bit maps v to u = v + 128 in [0, 255]; the binary16 with
// bit pattern 0x6400 | u is exactly 1024 + u (exponent 2^10, unit spacing);
// subtracting 1152 = 1024 + 128 leaves v exactly.
__device__ __forceinline__ void s8x4_to_f16x4(uint32_t x, uint32_t &lo, uint32_t &hi) {
    const uint32_t u = x ^ 0x80808080u;
    const uint32_t p01 = __byte_perm(u, 0x64646464u, 0x4140);
    const uint32_t p23 = __byte_perm(u, 0x64646464u, 0x4342);
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
    const __half2 r01 = __hsub2(*reinterpret_cast<const __half2 *>(&p01), bias);
    const __half2 r23 = __hsub2(*reinterpret_cast<const __half2 *>(&p23), bias);
    lo = *reinterpret_cast<const uint32_t *>(&r01);
    hi = *reinterpret_cast<const uint32_t *>(&r23);
}

__device__ __forceinline__ uint16_t s8_to_f16_bits(int8_t v) {
    return __half_as_ushort(__int2half_rn(static_cast<int>(v)));
}

// ---------------------------------------------------------------- s4 -> e4m3
// E4M3 (sign, 4 exponent bits with bias 7, 3 fraction bits) encoding of a
// small integer, from the format's definition: |v| = 2^e * (1 + f/8).
__host__ __device__ constexpr uint32_t e4m3_of_int(int v) {
    const uint32_t sign = v < 0 ? 0x80u : 0u;
    const int a = v < 0 ? -v : v;
    if (a == 0) return sign;
    int e = 0;
    while ((a >> (e + 1)) != 0) ++e;            // e = floor(log2 a)
    const uint32_t frac = uint32_t((a << 3) >> e) - 8u;  // exact for a <= 15
    return sign | (uint32_t(e + 7) << 3) | frac;
}

// Byte i of the four lookup words is the E4M3 encoding of the two's-complement
// nibble i (0..7 -> 0..7, 8..15 -> -8..-1).
__host__ __device__ constexpr uint32_t lut_word(int first) {
    uint32_t w = 0;
    for (int i = 0; i < 4; ++i) {
        const int nib = first + i;
        w |= e4m3_of_int(nib >= 8 ? nib - 16 : nib) << (8 * i);
    }
    return w;
}
inline constexpr uint32_t LUT0 = lut_word(0), LUT1 = lut_word(4), LUT2 = lut_word(8), LUT3 = lut_word(12);
static_assert(e4m3_of_int(1) == 0x38 && e4m3_of_int(7) == 0x4E && e4m3_of_int(-8) == 0xD0,
              "E4M3 encoding");

// Eight packed s4 (a 32-bit word, element j in bits 4j..4j+3) -> eight E4M3
// bytes (lo: elements 0-3, hi: 4-7).  PRMT looks each nibble's low three bits
// up in the positive (0..7) and the negative (-8..-1) half-tables, and a third
// PRMT takes byte j from the negative result when bit 3 of nibble j is set
// (selector j, or j + 4: that bit shifted to bit 2).  Eleven instructions per
// eight values; no selector has bit 3 set, so PRMT never replicates a sign.
__device__ __forceinline__ void s4x8_to_e4m3x8(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t idx = w & 0x77777777u;
    const uint32_t sel = ((w >> 1) & 0x44444444u) | 0x32103210u;
    lo = __byte_perm(__byte_perm(LUT0, LUT1, idx), __byte_perm(LUT2, LUT3, idx), sel);
    hi = __byte_perm(__byte_perm(LUT0, LUT1, idx >> 16), __byte_perm(LUT2, LUT3, idx >> 16), sel >> 16);
}

__device__ __forceinline__ uint8_t s4_to_e4m3_byte(uint32_t nib) {
    uint32_t lo, hi;
    s4x8_to_e4m3x8(nib & 0xFu, lo, hi);
    return static_cast<uint8_t>(lo & 0xFFu);
}

// Sixteen s8 (one 16-byte vector, element j in byte j) -> sixteen binary16
// (two 16-byte vectors: elements 0-7, 8-15).
__device__ __forceinline__ void cvt_s8_f16_x16(const uint4 &x, uint4 &o0, uint4 &o1) {
    s8x4_to_f16x4(x.x, o0.x, o0.y);
    s8x4_to_f16x4(x.y, o0.z, o0.w);
    s8x4_to_f16x4(x.z, o1.x, o1.y);
    s8x4_to_f16x4(x.w, o1.z, o1.w);
}

// Thirty-two packed s4 (one 16-byte vector, element 2b in the low nibble of
// byte b, 2b + 1 in its high nibble) -> thirty-two E4M3 bytes (two vectors).
__device__ __forceinline__ void cvt_s4_e4m3_x32(const uint4 &x, uint4 &o0, uint4 &o1) {
    s4x8_to_e4m3x8(x.x, o0.x, o0.y);
    s4x8_to_e4m3x8(x.y, o0.z, o0.w);
    s4x8_to_e4m3x8(x.z, o1.x, o1.y);
    s4x8_to_e4m3x8(x.w, o1.z, o1.w);
}

}  // namespace ptc
