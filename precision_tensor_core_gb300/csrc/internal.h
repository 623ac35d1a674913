// internal.h -- declarations shared by the host side of libptc (not part of
// the public C ABI; see include/ptc.h for that).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace ptc {

// Output tile of one CTA and one tensor-memory accumulator buffer.
constexpr int kBM = 128;
constexpr int kBN = 256;
// Bytes of K held per operand row per pipeline stage: one 128-byte swizzle row
// (64 FP16 or 128 E4M3 elements).
constexpr int kRowBytes = 128;

enum class Kind : int { F16 = 0, E4M3 = 1 };

// Arguments of one GEMM kernel launch (the tensor maps travel separately).
struct GemmArgs {
    void *C;               // float (FP16 path) or int32 (integer paths), row-major
    int64_t ldc;           // elements
    int M, N, K;           // K in operand elements
    int tiles_m, tiles_n;  // output tiles of (kBM * ctas) x bn
    int bn;                // one-CTA launches: tile width 256 (0 means 256), 128 or 64
    int num_tiles;
    int num_kb;            // K blocks of kRowBytes bytes
    int kb_per_chunk;      // K blocks summed in one accumulator buffer before the
                           // epilogue folds the partial sum into int32 registers
    int group_m;           // tiles of M per raster group (L2 reuse)
    int stall_tile;        // test hook: withhold this tile's operands (-1: none)
    int l2_hint;           // L2 policy of operand loads: 0 none, 1 A evict-last and
                           // B evict-first, 2 A evict-last, 3 both evict-normal
    uint64_t wait_limit_ns;
    // Work list of the launch (set by launch_gemm): the last tail_split tiles
    // run as two units each over the two halves of K, num_vunits units in all;
    // the halves exchange partial sums through split_part, ordered by the
    // arrival counters split_count (zero at launch).
    int stage_kb;          // CTA pairs: K blocks per ring stage, 1 or 2 (0: 2)
    int c_wide;            // 1: C's base and pitch allow 32-byte stores (set by launch_gemm)
    int c_tma;             // 1: a TMA map of 4-byte C is passed; each cluster's last unit stores
                           // through it (set by launch_gemm)
    int ksplit;            // single-wave one-CTA launches: CTAs per tile sharing its K range
                           // in a cluster (0: chosen by size, 1: none, 2 / 4 / 8: that many
                           // when the launch allows it; tuning knob "ksplit")
    int pdl;               // 1: launched with programmatic stream serialization (knob "pdl")
    int in_ring;           // 1: one-CTA integer launch whose tensor maps view the raw s8 / packed
                           // s4 operands (boxes of 64 bytes x 128 rows of A, x bn rows of B, no
                           // swizzle); the epilogue warps convert each K block in shared memory
    int split_ok;          // 1: the tail may be split (tuning knob "tail_split")
    int split_min_kb;      // ... when K spans at least this many K blocks
    int tail_split;
    int num_vunits;
    int split_reduce;      // 1: both halves of a split tile add their partial sums into C by TMA
                           // reductions (FP32 C, int32 C); the first half's cluster zeroes the
                           // tile's C at its start and sets split_count[slice] (one flag per
                           // epilogue warp slice); no partial-sum workspace
    uint32_t *split_count;
    float *split_part;
    // Clock record (knob "clock_probe"): when set, thread 0 of every CTA adds
    // its SM clock cycles, its global-timer nanoseconds and 1 to clock_probe[0..2]
    // (set by launch_gemm from `probe`).
    int probe;
    unsigned long long *clock_probe;
    // CTA pairs per thread-block cluster (knob "multicast"): 1, or 2 pairs that
    // compute two adjacent tile columns and share A by TMA multicast (the A
    // tensor map then has boxes of 64 rows).
    int pairs;
    // Integer routes with the conversion inside the GEMM (conv = 1): converter
    // warps rewrite the raw operands (s8, or packed s4) into the workspace rows
    // that the tensor maps read (binary16 / E4M3, conv_ldw elements per row),
    // in items of a few rows x kConvSlice K elements, in the order the tiles
    // need them: the K slices of the panels (128 rows) of A and B that the
    // first wave uses (conv_front_a / conv_front_b panels) slice by slice,
    // then the other B panels, then the other A panels.  Each item adds 1 to
    // the counter of its (panel, slice) (A panels first, then B) and to the
    // last counter; the producer loads a slice of a panel once its counter
    // holds all its items.  The counters are zero at launch.
    int conv;
    const uint8_t *conv_a, *conv_b;  // raw A (M rows) and B (N rows of K)
    int64_t conv_lda, conv_ldb;      // their row pitches in bytes
    void *conv_wa, *conv_wb;         // workspace rows
    int64_t conv_ldw;                // workspace row pitch in elements
    uint32_t *conv_count;            // (panels of A + panels of B) x slices counters, then one more
    int conv_front_a, conv_front_b;
    // Integer routes only: output of the epilogue.
    int out_mode;          // OUT_S32, or OUT_F32 / OUT_BF16 / OUT_F16 (scaled)
    const float *scale_a;  // M row scales (scaled modes; NULL: 1)
    const float *scale_b;  // N column scales (scaled modes; NULL: 1)
};

// Epilogue outputs of the integer routes.  The scaled modes write
// rn(rn(rn(float(acc)) * scale_a[i]) * scale_b[j]) rounded to the output type.
enum OutMode : int { OUT_S32 = 0, OUT_F32 = 1, OUT_BF16 = 2, OUT_F16 = 3 };

// Dynamic shared memory the GEMM kernel needs (ctas = 1: one CTA per
// 128 x 256 tile; ctas = 2: a CTA pair per 256 x 256 tile).
size_t gemm_smem_bytes(int ctas);
// Counters an integer launch with conversion in the GEMM kernel uses (one per
// panel of 128 rows of A or B and K slice, plus one), zeroed by that launch.
int64_t conv_counter_words(int64_t M, int64_t N, int64_t K);

// Epilogues of the tensor-core GEMM kernel.
enum Epi : int {
    EPI_F32 = 0,     // FP32 accumulators -> FP32 C
    EPI_INT = 1,     // FP32 chunk sums folded into int32 -> int32 or scaled output
    EPI_F16ACC = 2,  // FP16 accumulators -> FP16 C
};

// Launch the persistent tensor-core GEMM on at most `sms` SMs.
//   F16  + B MN-major + EPI_F32:     gemm_f16
//   F16  + B MN-major + EPI_F16ACC:  gemm_f16_f16acc
//   F16  + B K-major  + EPI_INT:     gemm_s8 (operands converted s8 -> f16)
//   E4M3 + B K-major  + EPI_INT:     gemm_s4 (operands converted s4 -> e4m3)
// args.tiles_m counts tiles of kBM * ctas rows, args.tiles_n tiles of args.bn
// columns (kBN for CTA pairs).  The tensor map of A has boxes of kBM rows;
// that of B boxes of bn / ctas rows (K-major) or 64 x 64 (MN-major).
// With a non-null pool (and args.split_ok) a short last wave of 256-wide tiles
// is split in K, using a workspace of at most ~20 MB taken from the pool on
// `stream` and returned after the kernel; a null pool runs every tile whole.
// One-CTA 256-wide launches run as K-split clusters when pick_ksplit(...,
// args.ksplit, ...) returns more than 1 (no workspace).  args.pdl launches
// with programmatic stream serialization.  args.in_ring (integer kinds, one
// CTA, K-major B) converts the raw operands inside the kernel; such launches
// never split the tail.
cudaError_t launch_gemm(Kind kind, bool b_mn_major, int epi, int ctas, const CUtensorMap &ta,
                        const CUtensorMap &tb, const GemmArgs &args, int sms, cudaMemPool_t pool,
                        cudaStream_t stream);

// Clusters of 2, 4 and 8 one-CTA tiles that fit one wave on a device (0 when
// that cluster shape cannot run).
struct ClusterCaps {
    int c2 = 0, c4 = 0, c8 = 0;
    int of(int ks) const { return ks == 2 ? c2 : ks == 4 ? c4 : ks == 8 ? c8 : 0; }
};

// The current device's capacities (queried once per device and thread).
ClusterCaps cluster_caps(int sms);

// CTAs per K-split cluster for a one-CTA launch of `tiles` 256-wide output
// tiles of num_kb K blocks each: 1 (no split), 2, 4 or 8.  knob: 0 chooses by
// size (the largest KS whose clusters fit one wave and that sheds each CTA at
// least 8 K blocks), 1 never, 2 / 4 / 8 that KS when it fits.  Host-only and
// pure given the capacities.
int pick_ksplit_pure(int tiles, int num_kb, int knob, int sms, const ClusterCaps &caps);
int pick_ksplit(int tiles, int num_kb, int knob, int sms);

// Launch shape of the calling thread's last GEMM kernel launch (grid CTAs,
// CTAs per cluster, CTAs sharing a tile's K range, tile width); zeros before
// the first.
void last_launch(int *grid, int *cluster, int *ksplit, int *tile_n);

// C[M x N] = 0 for elements of esize (2 or 4) bytes, ldc in elements.
cudaError_t launch_zero_fill(void *C, int64_t ldc, int M, int N, int esize, int grid, cudaStream_t stream);

// Reads and clears the device error word of the current device.
cudaError_t read_and_clear_error_word(uint32_t *out);

// Clock record of the GEMM kernels on the current device, per kernel family
// (0: FP16 kind with FP32 / FP16 output, 1: FP16 kind with integer folds
// (INT8), 2: E4M3 kind (INT4)): SM clock cycles, global-timer nanoseconds and
// CTAs, summed over the CTAs of every launch made with args.probe set.  Reads
// and clears the record (synchronous).
cudaError_t read_and_clear_clock_probe(unsigned long long out[9]);

// Operand preparation for the integer routes: exact element conversion into
// dense, 128-byte-pitched workspace matrices of `cols` columns.
//   s8 -> binary16: source pitches in bytes, destination pitch ldd elements
cudaError_t launch_s8_to_f16(const int8_t *src, int64_t lds, int rows, int cols, uint16_t *dst,
                             int64_t ldd, int grid, cudaStream_t stream, bool pdl = false);
//   both operands in one launch: rows_a rows of A, then rows_b rows of B
cudaError_t launch_s8_to_f16_pair(const int8_t *a, int64_t lda, int rows_a, const int8_t *b,
                                  int64_t ldb, int rows_b, int cols, uint16_t *dst_a, uint16_t *dst_b,
                                  int64_t ldd, int grid, cudaStream_t stream, bool pdl = false);
//   packed s4 -> E4M3, both operands: source pitches in BYTES, ldd in elements
cudaError_t launch_s4_to_e4m3_pair(const uint8_t *a, int64_t lda, int rows_a, const uint8_t *b,
                                   int64_t ldb, int rows_b, int cols, uint8_t *dst_a, uint8_t *dst_b,
                                   int64_t ldd, int grid, cudaStream_t stream, bool pdl = false);
// pdl: launched with programmatic stream serialization (it may start before the
// previous kernel in the stream ends; it waits for it before touching memory).

// The paper's kernel families on GB300 (baseline.cu): WMMA and mma.sync.
enum Variant : int {
    BASE_F16_WMMA = 0,
    BASE_F16_MMA = 1,
    BASE_S8_WMMA = 2,
    BASE_S8_MMA = 3,
    BASE_S4_WMMA = 4,
    BASE_S4_MMA = 5,
    // The same mma.sync kernels with fragments loaded by ldmatrix (A: .x4,
    // B: .x2, FP16 B transposed on the load).
    BASE_F16_LDM = 6,
    BASE_S8_LDM = 7,
    BASE_S4_LDM = 8,
};
// K must be a multiple of this many values for variant v (M of 32, N of 64).
int baseline_k_multiple(Variant v);
// A row-major, B column-major (integer) or row-major (FP16); pitches in bytes;
// C row-major FP32 (FP16 variants) or int32, ldc in elements.
cudaError_t launch_baseline(Variant v, const void *A, int64_t lda_b, const void *B, int64_t ldb_b, void *C,
                            int64_t ldc, int M, int N, int K, cudaStream_t s);

// Adds to the library's kernel-launch counter (ptc_kernel_launch_count).
void note_launches(uint64_t n);
// Sets the calling thread's detail text shown by gemm_status_string.
void set_message(const char *text);
// TMA tensor map of a row-major matrix (2-byte elements, or 1-byte when
// one_byte), 128-byte swizzle, zero fill outside; returns a PTC_* status.
// C as 4-byte elements: N x M (ldc elements between rows), boxes of 32 x 32
// with the 128-byte swizzle, for the epilogue's TMA stores.
int encode_tmap_c32(CUtensorMap *map, const void *C, uint64_t n, uint64_t m, uint64_t ldc, bool fp32);
int encode_tmap_2d(CUtensorMap *map, bool one_byte, const void *base, uint64_t inner, uint64_t outer,
                   uint64_t pitch, uint32_t box_inner, uint32_t box_outer);

}  // namespace ptc
