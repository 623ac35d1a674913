// baseline.cu -- the paper's own kernel families, run on GB300 as same-precision
// baselines for its speedup definitions.
//
// "Hand-Written PTX Tensor-Core GEMM Kernels: A Multi-Precision Study on
// NVIDIA L4" compares, per precision, a double-buffered WMMA kernel with
// hand-written PTX kernels (section III-A: a shared configuration of 16 x 16
// warp tiles, four in X and two in Y, eight warps per block; cp.async 16-byte
// staging into two shared-memory buffers, Listing 1; mma.sync m16n8k16 /
// m16n8k32 / m16n8k64 on register fragments, Listing 2).  These kernels
// restate that design for sm_103a with the legacy warp-level tensor-core
// instructions; they are comparison points for the tcgen05 kernels, not the
// library's fast path.
//
// Fragments of the mma.sync kernels come either from scalar 32-bit shared
// loads packed by hand (the *_MMA variants) or from ldmatrix (*_LDM: A as four
// 8 x 8 b16 matrices with .x4, B as two with .x2; the FP16 kernel's row-major
// B tile is transposed by the load), the fragment path of the paper's fastest
// INT8 / INT4 kernels (section IV-B/IV-C, Table VI; Listing 2 loads A with
// ldmatrix.x4 and B with .x2 before each m16n8k64).
//
// Block: 256 threads = 8 warps, block tile 32 (M) x 64 (N), warp (wy, wx)
// owns rows 16 wy .. +15 and columns 16 wx .. +15.  Per stage 64 bytes of K
// per operand row (32 FP16, 64 INT8 or 128 INT4 values), rows padded by 16
// bytes; stage kt+1 is copied with cp.async while stage kt is computed.
// Shapes must be multiples of the block tile and of the stage depth.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <mma.h>

#include <cstdint>

#include "internal.h"

namespace ptc {
namespace {

using namespace nvcuda;

constexpr int BM = 32, BN = 64, THREADS = 256;
constexpr int ROWB = 64;         // K bytes per operand row per stage
constexpr int PITCH = ROWB + 16; // padded shared-memory row pitch in bytes

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Shared-memory stage: A 32 rows, B either 64 N-rows of K (integer operands,
// column-major B) or KB K-rows of 64 N values (FP16 B, row-major).
template <Variant V>
struct Shape;

// Per-variant constants: K values per stage and the tile layouts.
//   row layout:    operand rows of 64 bytes at PITCH (80 bytes)
//   sliced layout: the 64 bytes of a row in four 16-byte K slices, slice s of
//                  row r at s * rows * 32 + r * 32 (32-byte aligned fragment
//                  starts for the integer WMMA shapes, whose K step is 16 bytes)
template <int KVALS, bool B_ROWMAJOR, bool SLICED>
struct StageShape {
    static constexpr int K = KVALS;
    static constexpr bool B_RM = B_ROWMAJOR;
    static constexpr bool SL = SLICED;
    static_assert(!(B_RM && SL), "row-major B tiles are never sliced");
    static constexpr int A_BYTES = SLICED ? 4 * BM * 32 : BM * PITCH;
    // FP16 B row-major: K rows of 64 halves (128 bytes) padded by 16 bytes.
    static constexpr int B_PITCH = B_ROWMAJOR ? (BN * 2 + 16) : PITCH;
    static constexpr int B_BYTES = SLICED ? 4 * BN * 32 : (B_ROWMAJOR ? KVALS * B_PITCH : BN * PITCH);
    static constexpr int BYTES = A_BYTES + B_BYTES;
};

template <> struct Shape<BASE_F16_WMMA> : StageShape<32, true, false> {};
template <> struct Shape<BASE_F16_MMA> : StageShape<32, true, false> {};
template <> struct Shape<BASE_S8_WMMA> : StageShape<64, false, true> {};
template <> struct Shape<BASE_S8_MMA> : StageShape<64, false, false> {};
template <> struct Shape<BASE_S4_WMMA> : StageShape<128, false, true> {};
template <> struct Shape<BASE_S4_MMA> : StageShape<128, false, false> {};
template <> struct Shape<BASE_F16_LDM> : StageShape<32, true, false> {};
template <> struct Shape<BASE_S8_LDM> : StageShape<64, false, false> {};
template <> struct Shape<BASE_S4_LDM> : StageShape<128, false, false> {};

// Copies stage kt of the block's A rows and B tile into shared memory.
// lda_b / ldb_b are row pitches in bytes of the global operands.
template <Variant V>
__device__ __forceinline__ void load_stage(uint8_t *sa, uint8_t *sb, const uint8_t *A, int64_t lda_b,
                                           const uint8_t *B, int64_t ldb_b, int m0, int n0, int kt) {
    using S = Shape<V>;
    const int t = threadIdx.x;
    // A: 32 rows x 64 bytes = 128 chunks of 16 bytes.
    if (t < BM * (ROWB / 16)) {
        const int r = t / (ROWB / 16), c = t % (ROWB / 16);
        uint8_t *dst = S::SL ? sa + c * (BM * 32) + r * 32 : sa + r * PITCH + c * 16;
        cp_async16(dst, A + int64_t(m0 + r) * lda_b + int64_t(kt) * ROWB + c * 16);
    }
    if constexpr (S::SL) {
        const int r = t / (ROWB / 16), c = t % (ROWB / 16);
        cp_async16(sb + c * (BN * 32) + r * 32, B + int64_t(n0 + r) * ldb_b + int64_t(kt) * ROWB + c * 16);
    } else if constexpr (S::B_RM) {
        // FP16 B row-major: 32 K-rows x 128 bytes = 256 chunks.
        const int r = t / 8, c = t % 8;
        cp_async16(sb + r * S::B_PITCH + c * 16, B + int64_t(kt * S::K + r) * ldb_b + int64_t(n0) * 2 + c * 16);
    } else {
        // Integer B column-major: 64 N-rows x 64 bytes = 256 chunks.
        const int r = t / (ROWB / 16), c = t % (ROWB / 16);
        cp_async16(sb + r * PITCH + c * 16, B + int64_t(n0 + r) * ldb_b + int64_t(kt) * ROWB + c * 16);
    }
}

__device__ __forceinline__ uint32_t ld32(const uint8_t *p) { return *reinterpret_cast<const uint32_t *>(p); }

// ldmatrix: lane t supplies the address of row t % 8 of 8 x 8 b16 matrix t / 8
// (16 contiguous bytes); register i of lane t receives the 32 bits at row
// t / 4, columns 2 (t % 4) .. +1 of matrix i (.trans: of its transpose).
__device__ __forceinline__ void ldm_x4(const uint8_t *row, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(row));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(a));
}
__device__ __forceinline__ void ldm_x2(const uint8_t *row, uint32_t &r0, uint32_t &r1) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(row));
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(a));
}
__device__ __forceinline__ void ldm_x2_trans(const uint8_t *row, uint32_t &r0, uint32_t &r1) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(row));
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(a));
}

// A fragment of one 16 x 16-byte slice (bytes kb .. kb + 31 of the warp's 16
// rows at PITCH): matrices rows 0-7 / 8-15 x bytes 0-15 / 16-31, which is the
// register order a0..a3 of m16n8k16 (FP16), m16n8k32 (s8) and m16n8k64 (s4).
__device__ __forceinline__ void ldm_a(const uint8_t *sa, int kb, int lane, uint32_t (&a)[4]) {
    const int r = (lane & 7) + 8 * ((lane >> 3) & 1);
    ldm_x4(sa + r * PITCH + kb + 16 * (lane >> 4), a[0], a[1], a[2], a[3]);
}

template <Variant V>
__global__ void __launch_bounds__(THREADS)
    baseline_kernel(const uint8_t *A, int64_t lda_b, const uint8_t *B, int64_t ldb_b, void *C, int64_t ldc,
                    int K) {
    using S = Shape<V>;
    __shared__ __align__(128) uint8_t smem[2][S::BYTES];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int wy = warp / 4, wx = warp % 4;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    const int kt_n = K / S::K;
    constexpr bool INT_C = !(V == BASE_F16_WMMA || V == BASE_F16_MMA || V == BASE_F16_LDM);

    // Accumulators: WMMA fragments, or mma.sync registers for two n8 tiles.
    wmma::fragment<wmma::accumulator, 16, 16, 16, float> acc_f;
    wmma::fragment<wmma::accumulator, 16, 16, 16, int> acc_i;
    wmma::fragment<wmma::accumulator, 8, 8, 32, int> acc_4[2][2];
    float cf[2][4] = {};
    int ci[2][4] = {};
    if constexpr (V == BASE_F16_WMMA) wmma::fill_fragment(acc_f, 0.0f);
    if constexpr (V == BASE_S8_WMMA) wmma::fill_fragment(acc_i, 0);
    if constexpr (V == BASE_S4_WMMA) {
        for (int i = 0; i < 2; ++i)
            for (int j = 0; j < 2; ++j) wmma::fill_fragment(acc_4[i][j], 0);
    }
    const int g = lane >> 2, tq = lane & 3;  // mma.sync fragment coordinates

    load_stage<V>(smem[0], smem[0] + S::A_BYTES, A, lda_b, B, ldb_b, m0, n0, 0);
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();
    for (int kt = 0; kt < kt_n; ++kt) {
        const int buf = kt & 1;
        if (kt + 1 < kt_n) {
            load_stage<V>(smem[buf ^ 1], smem[buf ^ 1] + S::A_BYTES, A, lda_b, B, ldb_b, m0, n0, kt + 1);
            cp_async_commit();
        }
        // This warp's 16 A rows (row layout); the sliced layout indexes per slice.
        const uint8_t *sa = smem[buf] + (S::SL ? 0 : wy * 16 * PITCH);
        const uint8_t *sb = smem[buf] + S::A_BYTES;
        if constexpr (V == BASE_F16_WMMA) {
#pragma unroll
            for (int k = 0; k < S::K; k += 16) {
                wmma::fragment<wmma::matrix_a, 16, 16, 16, half, wmma::row_major> fa;
                wmma::fragment<wmma::matrix_b, 16, 16, 16, half, wmma::row_major> fb;
                wmma::load_matrix_sync(fa, reinterpret_cast<const half *>(sa) + k, PITCH / 2);
                wmma::load_matrix_sync(fb, reinterpret_cast<const half *>(sb + k * S::B_PITCH) + wx * 16,
                                       S::B_PITCH / 2);
                wmma::mma_sync(acc_f, fa, fb, acc_f);
            }
        } else if constexpr (V == BASE_S8_WMMA) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {  // 16-byte K slices = k16 steps
                wmma::fragment<wmma::matrix_a, 16, 16, 16, signed char, wmma::row_major> fa;
                wmma::fragment<wmma::matrix_b, 16, 16, 16, signed char, wmma::col_major> fb;
                wmma::load_matrix_sync(fa, reinterpret_cast<const signed char *>(sa + ks * (BM * 32) + wy * 16 * 32), 32);
                wmma::load_matrix_sync(fb, reinterpret_cast<const signed char *>(sb + ks * (BN * 32) + wx * 16 * 32), 32);
                wmma::mma_sync(acc_i, fa, fb, acc_i);
            }
        } else if constexpr (V == BASE_S4_WMMA) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {  // 16-byte K slices = k32 steps of nibbles
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    wmma::fragment<wmma::matrix_a, 8, 8, 32, wmma::experimental::precision::s4, wmma::row_major> fa;
                    wmma::load_matrix_sync(fa, sa + ks * (BM * 32) + (wy * 16 + i * 8) * 32, 64);
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        wmma::fragment<wmma::matrix_b, 8, 8, 32, wmma::experimental::precision::s4, wmma::col_major> fb;
                        wmma::load_matrix_sync(fb, sb + ks * (BN * 32) + (wx * 16 + j * 8) * 32, 64);
                        wmma::mma_sync(acc_4[i][j], fa, fb, acc_4[i][j]);
                    }
                }
            }
        } else if constexpr (V == BASE_F16_MMA) {
#pragma unroll
            for (int k = 0; k < S::K; k += 16) {
                // A fragment: rows g and g+8, K pairs at 2 tq and 8 + 2 tq.
                const uint32_t a0 = ld32(sa + g * PITCH + (k + 2 * tq) * 2);
                const uint32_t a1 = ld32(sa + (g + 8) * PITCH + (k + 2 * tq) * 2);
                const uint32_t a2 = ld32(sa + g * PITCH + (k + 8 + 2 * tq) * 2);
                const uint32_t a3 = ld32(sa + (g + 8) * PITCH + (k + 8 + 2 * tq) * 2);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    // B fragment of the row-major B tile: column n, K pairs packed by hand.
                    const int n = wx * 16 + j * 8 + g;
                    const uint16_t *b = reinterpret_cast<const uint16_t *>(sb);
                    const int bp = S::B_PITCH / 2;
                    const uint32_t b0 = uint32_t(b[(k + 2 * tq) * bp + n]) | (uint32_t(b[(k + 2 * tq + 1) * bp + n]) << 16);
                    const uint32_t b1 =
                        uint32_t(b[(k + 8 + 2 * tq) * bp + n]) | (uint32_t(b[(k + 9 + 2 * tq) * bp + n]) << 16);
                    asm volatile(
                        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                        "{%0,%1,%2,%3};"
                        : "+f"(cf[j][0]), "+f"(cf[j][1]), "+f"(cf[j][2]), "+f"(cf[j][3])
                        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
                }
            }
        } else if constexpr (V == BASE_S8_MMA) {
#pragma unroll
            for (int k = 0; k < S::K; k += 32) {  // bytes = values
                const uint32_t a0 = ld32(sa + g * PITCH + k + 4 * tq);
                const uint32_t a1 = ld32(sa + (g + 8) * PITCH + k + 4 * tq);
                const uint32_t a2 = ld32(sa + g * PITCH + k + 16 + 4 * tq);
                const uint32_t a3 = ld32(sa + (g + 8) * PITCH + k + 16 + 4 * tq);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const uint8_t *bn = sb + (wx * 16 + j * 8 + g) * PITCH;
                    const uint32_t b0 = ld32(bn + k + 4 * tq), b1 = ld32(bn + k + 16 + 4 * tq);
                    asm volatile(
                        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                        "{%0,%1,%2,%3};"
                        : "+r"(ci[j][0]), "+r"(ci[j][1]), "+r"(ci[j][2]), "+r"(ci[j][3])
                        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
                }
            }
        } else if constexpr (V == BASE_F16_LDM) {
#pragma unroll
            for (int k = 0; k < S::K; k += 16) {
                uint32_t a[4];
                ldm_a(sa, k * 2, lane, a);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    // B rows k .. k + 15 (K) of the row-major tile, the 8 columns
                    // of tile j, transposed into the k-pair fragment b0, b1.
                    uint32_t b0, b1;
                    const int kr = k + (lane & 7) + 8 * ((lane >> 3) & 1);
                    ldm_x2_trans(sb + kr * S::B_PITCH + (wx * 16 + j * 8) * 2, b0, b1);
                    asm volatile(
                        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                        "{%0,%1,%2,%3};"
                        : "+f"(cf[j][0]), "+f"(cf[j][1]), "+f"(cf[j][2]), "+f"(cf[j][3])
                        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
                }
            }
        } else if constexpr (V == BASE_S8_LDM || V == BASE_S4_LDM) {
#pragma unroll
            for (int k = 0; k < ROWB; k += 32) {  // 32 bytes per step: k32 of s8, k64 of s4
                uint32_t a[4];
                ldm_a(sa, k, lane, a);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    // Column-major B: the 8 N-rows of tile j, bytes k .. k + 15 and
                    // k + 16 .. k + 31 (lanes 0-7 and 8-15 give the row addresses).
                    uint32_t b0, b1;
                    ldm_x2(sb + (wx * 16 + j * 8 + (lane & 7)) * PITCH + k + 16 * ((lane >> 3) & 1), b0, b1);
                    if constexpr (V == BASE_S8_LDM)
                        asm volatile(
                            "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                            "{%0,%1,%2,%3};"
                            : "+r"(ci[j][0]), "+r"(ci[j][1]), "+r"(ci[j][2]), "+r"(ci[j][3])
                            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
                    else
                        asm volatile(
                            "mma.sync.aligned.m16n8k64.row.col.s32.s4.s4.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                            "{%0,%1,%2,%3};"
                            : "+r"(ci[j][0]), "+r"(ci[j][1]), "+r"(ci[j][2]), "+r"(ci[j][3])
                            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
                }
            }
        } else {  // BASE_S4_MMA
#pragma unroll
            for (int k = 0; k < S::K / 2; k += 32) {  // k in bytes; 64 nibbles per step
                const uint32_t a0 = ld32(sa + g * PITCH + k + 4 * tq);
                const uint32_t a1 = ld32(sa + (g + 8) * PITCH + k + 4 * tq);
                const uint32_t a2 = ld32(sa + g * PITCH + k + 16 + 4 * tq);
                const uint32_t a3 = ld32(sa + (g + 8) * PITCH + k + 16 + 4 * tq);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const uint8_t *bn = sb + (wx * 16 + j * 8 + g) * PITCH;
                    const uint32_t b0 = ld32(bn + k + 4 * tq), b1 = ld32(bn + k + 16 + 4 * tq);
                    asm volatile(
                        "mma.sync.aligned.m16n8k64.row.col.s32.s4.s4.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                        "{%0,%1,%2,%3};"
                        : "+r"(ci[j][0]), "+r"(ci[j][1]), "+r"(ci[j][2]), "+r"(ci[j][3])
                        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
                }
            }
        }
        cp_async_wait_all();
        __syncthreads();
    }

    // Epilogue: the warp's 16 x 16 tile of C.
    const int row0 = m0 + wy * 16, col0 = n0 + wx * 16;
    if constexpr (V == BASE_F16_WMMA) {
        wmma::store_matrix_sync(static_cast<float *>(C) + int64_t(row0) * ldc + col0, acc_f, unsigned(ldc),
                                wmma::mem_row_major);
    } else if constexpr (V == BASE_S8_WMMA) {
        wmma::store_matrix_sync(static_cast<int *>(C) + int64_t(row0) * ldc + col0, acc_i, unsigned(ldc),
                                wmma::mem_row_major);
    } else if constexpr (V == BASE_S4_WMMA) {
        for (int i = 0; i < 2; ++i)
            for (int j = 0; j < 2; ++j)
                wmma::store_matrix_sync(static_cast<int *>(C) + int64_t(row0 + 8 * i) * ldc + col0 + 8 * j,
                                        acc_4[i][j], unsigned(ldc), wmma::mem_row_major);
    } else {
        // mma.sync accumulators: c0, c1 at row g, columns 2 tq, 2 tq + 1; c2, c3 at row g + 8.
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int c = col0 + j * 8 + 2 * tq;
            if constexpr (INT_C) {
                int *Ci = static_cast<int *>(C);
                *reinterpret_cast<int2 *>(Ci + int64_t(row0 + g) * ldc + c) = make_int2(ci[j][0], ci[j][1]);
                *reinterpret_cast<int2 *>(Ci + int64_t(row0 + g + 8) * ldc + c) = make_int2(ci[j][2], ci[j][3]);
            } else {
                float *Cf = static_cast<float *>(C);
                *reinterpret_cast<float2 *>(Cf + int64_t(row0 + g) * ldc + c) = make_float2(cf[j][0], cf[j][1]);
                *reinterpret_cast<float2 *>(Cf + int64_t(row0 + g + 8) * ldc + c) = make_float2(cf[j][2], cf[j][3]);
            }
        }
    }
}

template <Variant V>
cudaError_t launch_v(const void *A, int64_t lda_b, const void *B, int64_t ldb_b, void *C, int64_t ldc, int M,
                     int N, int K, cudaStream_t s) {
    const dim3 grid(N / BN, M / BM);
    baseline_kernel<V><<<grid, THREADS, 0, s>>>(static_cast<const uint8_t *>(A), lda_b,
                                                static_cast<const uint8_t *>(B), ldb_b, C, ldc, K);
    return cudaGetLastError();
}

}  // namespace

int baseline_k_multiple(Variant v) {
    switch (v) {
        case BASE_F16_WMMA:
        case BASE_F16_MMA:
        case BASE_F16_LDM: return 32;
        case BASE_S8_WMMA:
        case BASE_S8_MMA:
        case BASE_S8_LDM: return 64;
        default: return 128;
    }
}

cudaError_t launch_baseline(Variant v, const void *A, int64_t lda_b, const void *B, int64_t ldb_b, void *C,
                            int64_t ldc, int M, int N, int K, cudaStream_t s) {
    switch (v) {
        case BASE_F16_WMMA: return launch_v<BASE_F16_WMMA>(A, lda_b, B, ldb_b, C, ldc, M, N, K, s);
        case BASE_F16_MMA: return launch_v<BASE_F16_MMA>(A, lda_b, B, ldb_b, C, ldc, M, N, K, s);
        case BASE_S8_WMMA: return launch_v<BASE_S8_WMMA>(A, lda_b, B, ldb_b, C, ldc, M, N, K, s);
        case BASE_S8_MMA: return launch_v<BASE_S8_MMA>(A, lda_b, B, ldb_b, C, ldc, M, N, K, s);
        case BASE_S4_WMMA: return launch_v<BASE_S4_WMMA>(A, lda_b, B, ldb_b, C, ldc, M, N, K, s);
        case BASE_S4_MMA: return launch_v<BASE_S4_MMA>(A, lda_b, B, ldb_b, C, ldc, M, N, K, s);
        case BASE_F16_LDM: return launch_v<BASE_F16_LDM>(A, lda_b, B, ldb_b, C, ldc, M, N, K, s);
        case BASE_S8_LDM: return launch_v<BASE_S8_LDM>(A, lda_b, B, ldb_b, C, ldc, M, N, K, s);
        case BASE_S4_LDM: return launch_v<BASE_S4_LDM>(A, lda_b, B, ldb_b, C, ldc, M, N, K, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace ptc
