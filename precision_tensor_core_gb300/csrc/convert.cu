// convert.cu -- operand preparation for the integer routes.
//
// sm_103a offers no integer tcgen05 MMA, so the INT8 and INT4 products of
// "Hand-Written PTX Tensor-Core GEMM Kernels: A Multi-Precision Study on
// NVIDIA L4" (sections IV-B and IV-C) run on floating-point tensor-core kinds
// whose input formats hold every integer operand exactly:
//   s8 in [-128, 127] -> binary16 (11-bit significand: exact up to 2048)
//   s4 in [-8, 7]     -> E4M3 (4-bit significand: exact up to 16)
// These kernels rewrite A (row-major) and B (column-major, i.e. rows of K)
// into dense workspace rows of the MMA's input type, K contiguous.  They are
// streaming, HBM-bound kernels: 16-byte loads and stores, a grid-stride loop
// over (row, 16-byte vector) pairs, and scalar code only for the ragged end
// of a row, so no byte past a row's last element is read.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace ptc {
namespace {

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

// Converts rows [0, rows_a) of A and then rows [0, rows_b) of B, cols
// elements each, in one grid-stride pass over (row, 16-element vector) pairs.
// Each thread takes UNROLL vectors per pass and issues all their loads before
// converting, so that several 16-byte loads per thread are in flight.
constexpr int UNROLL = 4;

__global__ void s8_to_f16_kernel(const int8_t *__restrict__ src_a, int64_t lds_a, int rows_a,
                                 const int8_t *__restrict__ src_b, int64_t lds_b, int rows_b,
                                 int cols, uint16_t *__restrict__ dst_a, uint16_t *__restrict__ dst_b,
                                 int64_t ldd) {
    const int vpr = (cols + 15) / 16;  // 16-element vectors per row
    const int64_t total = int64_t(rows_a + rows_b) * vpr;
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t base = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; base < total;
         base += stride * UNROLL) {
        uint4 x[UNROLL];
        const int8_t *s[UNROLL];
        uint16_t *d[UNROLL];
        int c0[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t i = base + u * stride;
            s[u] = nullptr;
            if (i >= total) continue;
            int64_t r = i / vpr;
            c0[u] = int(i - r * vpr) * 16;
            if (r < rows_a) {
                s[u] = src_a + r * lds_a + c0[u];
                d[u] = dst_a + r * ldd + c0[u];
            } else {
                r -= rows_a;
                s[u] = src_b + r * lds_b + c0[u];
                d[u] = dst_b + r * ldd + c0[u];
            }
            if (c0[u] + 16 <= cols) x[u] = __ldcs(reinterpret_cast<const uint4 *>(s[u]));
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            if (s[u] == nullptr) continue;
            if (c0[u] + 16 <= cols) {
                uint4 o0, o1;
                s8x4_to_f16x4(x[u].x, o0.x, o0.y);
                s8x4_to_f16x4(x[u].y, o0.z, o0.w);
                s8x4_to_f16x4(x[u].z, o1.x, o1.y);
                s8x4_to_f16x4(x[u].w, o1.z, o1.w);
                reinterpret_cast<uint4 *>(d[u])[0] = o0;
                reinterpret_cast<uint4 *>(d[u])[1] = o1;
            } else {
                for (int j = 0; j < cols - c0[u]; ++j) d[u][j] = s8_to_f16_bits(s[u][j]);
            }
        }
    }
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
constexpr uint32_t LUT0 = lut_word(0), LUT1 = lut_word(4), LUT2 = lut_word(8), LUT3 = lut_word(12);
static_assert(e4m3_of_int(1) == 0x38 && e4m3_of_int(7) == 0x4E && e4m3_of_int(-8) == 0xD0,
              "E4M3 encoding");

// Four packed s4 (16 bits, element j in bits 4j..4j+3) -> four E4M3 bytes.
// The nibbles are exactly the byte selectors of PRMT: the low three bits pick
// a byte of the 8-entry half-table, bit 3 picks the half.
__device__ __forceinline__ uint32_t s4x4_to_e4m3x4(uint32_t sel16) {
    const uint32_t idx = sel16 & 0x7777u;
    const uint32_t pos = __byte_perm(LUT0, LUT1, idx);
    const uint32_t neg = __byte_perm(LUT2, LUT3, idx);
    const uint32_t t = (sel16 >> 3) & 0x1111u;  // bit 3 of each nibble at bit 4j
    const uint32_t m = ((t & 1u) | ((t & 0x10u) << 4) | ((t & 0x100u) << 8) | ((t & 0x1000u) << 12)) * 0xFFu;
    return (pos & ~m) | (neg & m);
}

__device__ __forceinline__ uint8_t s4_to_e4m3_byte(uint32_t nib) {
    return static_cast<uint8_t>(s4x4_to_e4m3x4(nib & 0xFu) & 0xFFu);
}

// As s8_to_f16_kernel: rows of A, then rows of B, 32-element vectors.
__global__ void s4_to_e4m3_kernel(const uint8_t *__restrict__ src_a, int64_t lds_a, int rows_a,
                                  const uint8_t *__restrict__ src_b, int64_t lds_b, int rows_b,
                                  int cols, uint8_t *__restrict__ dst_a, uint8_t *__restrict__ dst_b,
                                  int64_t ldd) {
    const int vpr = (cols + 31) / 32;  // 32-element (16-byte packed) vectors per row
    const int64_t total = int64_t(rows_a + rows_b) * vpr;
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t base = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; base < total;
         base += stride * UNROLL) {
        uint4 x[UNROLL];
        const uint8_t *s[UNROLL];
        uint8_t *d[UNROLL];
        int c0[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t i = base + u * stride;
            s[u] = nullptr;
            if (i >= total) continue;
            int64_t r = i / vpr;
            c0[u] = int(i - r * vpr) * 32;
            if (r < rows_a) {
                s[u] = src_a + r * lds_a + c0[u] / 2;
                d[u] = dst_a + r * ldd + c0[u];
            } else {
                r -= rows_a;
                s[u] = src_b + r * lds_b + c0[u] / 2;
                d[u] = dst_b + r * ldd + c0[u];
            }
            if (c0[u] + 32 <= cols) x[u] = __ldcs(reinterpret_cast<const uint4 *>(s[u]));
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            if (s[u] == nullptr) continue;
            if (c0[u] + 32 <= cols) {
                const uint32_t w[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
                uint32_t o[8];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    o[2 * q] = s4x4_to_e4m3x4(w[q] & 0xFFFFu);
                    o[2 * q + 1] = s4x4_to_e4m3x4(w[q] >> 16);
                }
                reinterpret_cast<uint4 *>(d[u])[0] = make_uint4(o[0], o[1], o[2], o[3]);
                reinterpret_cast<uint4 *>(d[u])[1] = make_uint4(o[4], o[5], o[6], o[7]);
            } else {
                for (int j = 0; j < cols - c0[u]; ++j) {
                    const uint32_t b = s[u][j >> 1];
                    d[u][j] = s4_to_e4m3_byte((j & 1) ? (b >> 4) : b);
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_s8_to_f16(const int8_t *src, int64_t lds, int rows, int cols, uint16_t *dst,
                             int64_t ldd, int grid, cudaStream_t stream) {
    s8_to_f16_kernel<<<grid, 256, 0, stream>>>(src, lds, rows, src, lds, 0, cols, dst, dst, ldd);
    return cudaGetLastError();
}

cudaError_t launch_s8_to_f16_pair(const int8_t *a, int64_t lda, int rows_a, const int8_t *b,
                                  int64_t ldb, int rows_b, int cols, uint16_t *dst_a, uint16_t *dst_b,
                                  int64_t ldd, int grid, cudaStream_t stream) {
    s8_to_f16_kernel<<<grid, 256, 0, stream>>>(a, lda, rows_a, b, ldb, rows_b, cols, dst_a, dst_b, ldd);
    return cudaGetLastError();
}

cudaError_t launch_s4_to_e4m3_pair(const uint8_t *a, int64_t lda, int rows_a, const uint8_t *b,
                                   int64_t ldb, int rows_b, int cols, uint8_t *dst_a, uint8_t *dst_b,
                                   int64_t ldd, int grid, cudaStream_t stream) {
    s4_to_e4m3_kernel<<<grid, 256, 0, stream>>>(a, lda, rows_a, b, ldb, rows_b, cols, dst_a, dst_b, ldd);
    return cudaGetLastError();
}

}  // namespace ptc
