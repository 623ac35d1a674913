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
#include <cstring>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "convert.cuh"
#include "ptx.cuh"

namespace ptc {
namespace {

// The two conversions, as element types, 16-byte input vectors and a
// vector / scalar conversion.
struct S8ToF16 {
    using In = int8_t;
    using Out = uint16_t;
    static constexpr int VEC = 16;  // elements per 16-byte input vector (32 output bytes)
    __device__ static const uint8_t *row_at(const uint8_t *row, int c0) { return row + c0; }
    __device__ static void vector(const uint4 &x, uint4 &o0, uint4 &o1) { cvt_s8_f16_x16(x, o0, o1); }
    __device__ static void scalar(const uint8_t *s, Out *d, int n) {
        for (int j = 0; j < n; ++j) d[j] = s8_to_f16_bits(static_cast<int8_t>(s[j]));
    }
};

struct S4ToE4M3 {
    using Out = uint8_t;
    static constexpr int VEC = 32;  // packed: 32 elements per 16-byte input vector (32 output bytes)
    __device__ static const uint8_t *row_at(const uint8_t *row, int c0) { return row + c0 / 2; }
    __device__ static void vector(const uint4 &x, uint4 &o0, uint4 &o1) { cvt_s4_e4m3_x32(x, o0, o1); }
    __device__ static void scalar(const uint8_t *s, Out *d, int n) {
        for (int j = 0; j < n; ++j) {
            const uint32_t b = s[j >> 1];
            d[j] = s4_to_e4m3_byte((j & 1) ? (b >> 4) : b);
        }
    }
};

// Converts rows [0, rows_a) of A and then rows [0, rows_b) of B, cols
// elements each (source pitches in bytes, destination pitch in elements).
// A group of 2^tpr_log2 threads covers one row; a 256-thread block covers
// 256 >> tpr_log2 rows per pass and strides over rows by the grid, so the
// row and vector of a thread come from a shift and a mask, not a division.
// Each thread issues UNROLL loads (vectors lane, lane + group, ...) before
// converting them; the ragged end of a row is converted element by element,
// so no byte past a row's last element is read.  W32: 32-byte vectors (one
// 32-byte load, two 32-byte stores; source bases and pitches 32-byte
// aligned), measured 1.5-3.5% faster per integer GEMM call than 16-byte ones.
constexpr int UNROLL = 4;

__device__ __forceinline__ void ld_global_cs_v8(const uint8_t *p, uint4 &lo, uint4 &hi) {
    asm volatile("ld.global.cs.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y), "=r"(hi.z), "=r"(hi.w)
                 : "l"(p));
}

__device__ __forceinline__ void st_global_v8_2x(void *p, const uint4 &lo, const uint4 &hi) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(lo.x), "r"(lo.y), "r"(lo.z),
                 "r"(lo.w), "r"(hi.x), "r"(hi.y), "r"(hi.z), "r"(hi.w)
                 : "memory");
}

template <class Op, bool W32>
__global__ void __launch_bounds__(256) convert_kernel(const uint8_t *__restrict__ src_a, int64_t lds_a, int rows_a,
                                                      const uint8_t *__restrict__ src_b, int64_t lds_b, int rows_b,
                                                      int cols, typename Op::Out *__restrict__ dst_a,
                                                      typename Op::Out *__restrict__ dst_b, int64_t ldd, int tpr_log2) {
    using Out = typename Op::Out;
    constexpr int V = W32 ? 2 * Op::VEC : Op::VEC;  // elements per input vector
    // Launched after a kernel that may still run (programmatic serialization):
    // its writes (and its reads of this workspace) are complete past here.  The
    // GEMM that follows may launch at once and set up while this pass runs.
    griddep_wait();
    griddep_launch_dependents();
    const int tpr = 1 << tpr_log2;
    const int lane = threadIdx.x & (tpr - 1);
    const int rpb = blockDim.x >> tpr_log2;
    const int vpr = (cols + V - 1) / V;
    const int64_t rows = int64_t(rows_a) + rows_b;
    for (int64_t r = int64_t(blockIdx.x) * rpb + (threadIdx.x >> tpr_log2); r < rows; r += int64_t(gridDim.x) * rpb) {
        const uint8_t *srow;
        Out *drow;
        if (r < rows_a) {
            srow = src_a + r * lds_a;
            drow = dst_a + r * ldd;
        } else {
            srow = src_b + (r - rows_a) * lds_b;
            drow = dst_b + (r - rows_a) * ldd;
        }
        for (int v0 = lane; v0 < vpr; v0 += tpr * UNROLL) {
            uint4 x[UNROLL][W32 ? 2 : 1];
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const int c0 = (v0 + u * tpr) * V;
                if (c0 + V <= cols) {
                    if constexpr (W32)
                        ld_global_cs_v8(Op::row_at(srow, c0), x[u][0], x[u][W32 ? 1 : 0]);
                    else
                        x[u][0] = __ldcs(reinterpret_cast<const uint4 *>(Op::row_at(srow, c0)));
                }
            }
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const int c0 = (v0 + u * tpr) * V;
                if (c0 + V <= cols) {
                    uint4 o0, o1;
                    Op::vector(x[u][0], o0, o1);
                    if constexpr (W32) {
                        uint4 o2, o3;
                        Op::vector(x[u][W32 ? 1 : 0], o2, o3);
                        st_global_v8_2x(drow + c0, o0, o1);
                        st_global_v8_2x(drow + c0 + Op::VEC, o2, o3);
                    } else {
                        uint4 *d = reinterpret_cast<uint4 *>(drow + c0);
                        d[0] = o0;
                        d[1] = o1;
                    }
                } else if (c0 < cols) {
                    Op::scalar(Op::row_at(srow, c0), drow + c0, cols - c0);
                }
            }
        }
    }
}

// log2 of the threads per row: enough for one pass of UNROLL vectors per
// thread over a row, at most the whole block.
int threads_per_row_log2(int cols, int vec) {
    const int vpr = (cols + vec - 1) / vec;
    int l = 0;
    while (l < 8 && (1 << l) * UNROLL < vpr) ++l;
    return l;
}

}  // namespace

cudaError_t launch_s8_to_f16(const int8_t *src, int64_t lds, int rows, int cols, uint16_t *dst,
                             int64_t ldd, int grid, cudaStream_t stream, bool pdl) {
    return launch_s8_to_f16_pair(src, lds, rows, src, lds, 0, cols, dst, dst, ldd, grid, stream, pdl);
}

// 32-byte vectors when both sources start on 32-byte boundaries and their
// pitches keep every row there (the workspace rows always are).
static bool aligned32(const void *a, int64_t lda, const void *b, int64_t ldb) {
    return (reinterpret_cast<uintptr_t>(a) % 32) == 0 && (reinterpret_cast<uintptr_t>(b) % 32) == 0 && lda % 32 == 0 &&
           ldb % 32 == 0;
}

template <class Op>
cudaError_t launch_convert(const uint8_t *a, int64_t lda, int rows_a, const uint8_t *b, int64_t ldb, int rows_b,
                           int cols, typename Op::Out *dst_a, typename Op::Out *dst_b, int64_t ldd, int grid,
                           cudaStream_t stream, bool pdl) {
    const bool w32 = aligned32(a, lda, b, ldb);
    auto *fn = w32 ? convert_kernel<Op, true> : convert_kernel<Op, false>;
    const int tpr_log2 = threads_per_row_log2(cols, w32 ? 2 * Op::VEC : Op::VEC);
    // No more CTAs than there are row groups to convert (small operands).
    const int64_t rows_per_block = 256 >> tpr_log2;
    const int64_t needed = (int64_t(rows_a) + rows_b + rows_per_block - 1) / rows_per_block;
    if (needed < grid) grid = int(needed > 0 ? needed : 1);
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cudaLaunchAttribute attr[1];
    std::memset(attr, 0, sizeof(attr));
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    cudaError_t e = cudaLaunchKernelEx(&cfg, fn, a, lda, rows_a, b, ldb, rows_b, cols, dst_a, dst_b, ldd, tpr_log2);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_s8_to_f16_pair(const int8_t *a, int64_t lda, int rows_a, const int8_t *b,
                                  int64_t ldb, int rows_b, int cols, uint16_t *dst_a, uint16_t *dst_b,
                                  int64_t ldd, int grid, cudaStream_t stream, bool pdl) {
    return launch_convert<S8ToF16>(reinterpret_cast<const uint8_t *>(a), lda, rows_a,
                                   reinterpret_cast<const uint8_t *>(b), ldb, rows_b, cols, dst_a, dst_b, ldd, grid,
                                   stream, pdl);
}

cudaError_t launch_s4_to_e4m3_pair(const uint8_t *a, int64_t lda, int rows_a, const uint8_t *b,
                                   int64_t ldb, int rows_b, int cols, uint8_t *dst_a, uint8_t *dst_b,
                                   int64_t ldd, int grid, cudaStream_t stream, bool pdl) {
    return launch_convert<S4ToE4M3>(a, lda, rows_a, b, ldb, rows_b, cols, dst_a, dst_b, ldd, grid, stream, pdl);
}

}  // namespace ptc
