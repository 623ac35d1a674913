// gemm_tc.cu -- persistent, warp-specialised tensor-core GEMM for sm_103a.
//
// The method is the tiled tensor-core GEMM of "Hand-Written PTX Tensor-Core
// GEMM Kernels: A Multi-Precision Study on NVIDIA L4" (section III-A: output
// tiles per block, a K loop that stages A/B tiles in shared memory while the
// tensor cores consume the previous ones, Listing 1), rebuilt for GB300:
//
//   warp 0      TMA producer: one thread streams 128-byte-wide K blocks of A
//               and B into a STAGES-deep shared-memory ring (128-byte swizzle),
//               completing on per-stage "full" mbarriers (replaces cp.async +
//               commit_group / wait_group + __syncthreads buffer rotation).
//   warp 1      allocates 2 x BN tensor-memory columns, then one thread
//               issues tcgen05.mma (N = BN, K = 32 bytes per instruction)
//               into a double-buffered tensor-memory accumulator and frees
//               ring stages with tcgen05.commit -> "empty" barriers (replaces
//               ldmatrix + mma.sync and register accumulators).
//   warps 2-9   epilogue: tcgen05.ld tensor memory -> registers -> global C,
//               overlapped with the next tile's MMAs through the second
//               accumulator buffer; 32-byte stores per lane, or 32 x 32
//               blocks staged in the then idle ring and written by TMA stores
//               where nothing hides the epilogue (4-byte C of a single-wave
//               launch, and the last tile of each cluster in FP32 C).
//   (CTA pairs that convert integer operands in the kernel run 16 warps:
//   producer, MMA issuer, converter warps 2-3, epilogue warps 4-11 and
//   converter warps 12-15; see Cfg::PFU.)
//
// Shapes of the same kernel:
//   CTAS = 1    one CTA per 128 x BN output tile (M = 128 MMAs): BN = 256 with
//               4 ring stages of one K block, or, for products too small to
//               occupy the SMs with 256-wide tiles, BN = 128 / 64 (6 / 8
//               stages), which spreads C over more SMs (each SM writes to L2
//               at ~32 bytes per clock, so a 128 x 256 FP32 tile takes ~2 us
//               to leave its SM).
//   CTAS = 2    a cluster of two CTAs per 256 x 256 output tile
//               (tcgen05 cta_group::2, M = 256 MMAs issued by the even CTA):
//               each CTA stages its own 128 rows of A and half of B, so a CTA
//               moves 32 KiB per K block instead of 48 KiB; the ring holds 3
//               stages of two K blocks (or, as a tuning choice, 7 of one).
//   KS = 2/4/8  one-CTA tiles in clusters of KS CTAs that share a tile's K
//               range (split-K inside a cluster), for single-wave launches
//               whose tiles would leave most SMs idle (8 only for 256-wide
//               tiles): each CTA multiplies about 1/KS of the K blocks,
//               writes its 128 x BN partial sums into its idle ring, and
//               after a cluster barrier completes 128/KS rows of the tile by
//               adding the KS partials in rank order, read from the peers'
//               shared memory (distributed shared memory).  No workspace, no
//               atomics, the same sums every run.
//
// The work list: output tiles in grouped raster order, strided over the
// clusters; when the last wave would leave at least half of the clusters idle,
// its tiles run as two K halves (see work_unit), added into C by TMA
// reductions (FP32 / int32 C of CTA pairs) or through a partial-sum exchange.
//
// Integer routes: sm_103a has no integer tcgen05 MMA, so INT8 runs on the
// FP16 kind (every s8 value is an exact binary16) and INT4 on the E4M3 kind
// (every s4 value is an exact E4M3).  Products are exact and the FP32 sums are
// exact integers while |partial sum| <= 2^24, so the K loop is cut into chunks
// of kb_per_chunk K blocks, each summed in its own accumulator buffer; the
// epilogue converts each chunk's (integral) FP32 sums to int32 and adds them
// in registers.  The int32 result is therefore the exact sum modulo 2^32.
// The operands arrive converted (binary16 / E4M3 rows written by a separate
// pass), or, with FU (one-CTA launches of small products), raw: the producer
// loads 64-byte K blocks of the s8 / packed s4 rows into a second ring and the
// epilogue warps, idle during the K loop, convert each into the MMA stage in
// the 128-byte-swizzled layout (fence.proxy.async, then eight arrivals
// complete the stage's full barrier).  They fold chunk c only after
// converting it and convert chunk c + 2 only after folding chunk c, whose
// accumulator buffer chunk c + 2 reuses, so the rings always drain.
//
// Tiles are spread over a persistent grid of at most one CTA per SM with no
// dependency between clusters (no grid-wide spin barrier).  The kernel may be
// launched while the previous kernel of the stream still runs (programmatic
// serialization): it sets up barriers and tensor memory, then waits for that
// kernel before its first global-memory access.  Every wait is
// bounded by a %globaltimer limit: on expiry the CTA raises an abort flag,
// records PTC_ERR_TIMEOUT in a device error word, lets its in-flight copies
// and MMAs land, frees tensor memory and exits.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstring>
#include <type_traits>

#include "convert.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace ptc {

__device__ uint32_t g_error_word;
// Clock record: per kernel family, SM cycles, nanoseconds and CTAs (see
// read_and_clear_clock_probe).
__device__ unsigned long long g_clock_probe[3][3];

namespace {

constexpr int EPI_WARPS = 8;
constexpr int THREADS = 64 + 32 * EPI_WARPS;  // warps 0, 1 and the epilogue warps 2 .. 9
// CTA pairs with in-ring conversion: 16 warps.  Warpgroup 0 holds the producer
// (warp 0), the MMA issuer (warp 1) and converter warps 2 and 3, warpgroups 1
// and 2 the epilogue warps (4 .. 11), warpgroup 3 converter warps 12 .. 15.  The
// launch grants 128 registers per thread (65,536 / 512); warpgroups 0 and 3
// give back all but kRegsLow (the producer, MMA and converter code fits in
// 80 without spills), the epilogue warpgroups take kRegsHigh (their 128 int32
// partial sums and the tensor-memory loads in flight):
// 8 warps x 80 + 8 warps x 176 = 16 warps x 128 registers per lane.
constexpr int PAIR_FU_THREADS = 512;
constexpr int CONV_WARPS = 4;  // converter warps of warpgroup 3 (warpgroup 0 adds two more)
constexpr uint32_t kRegsLow = 80, kRegsHigh = 176;
static_assert(8 * kRegsLow + 8 * kRegsHigh == (PAIR_FU_THREADS / 32) * (65536 / PAIR_FU_THREADS),
              "warpgroup register budgets sum to the launch's registers");
constexpr int KSTEP_BYTES = 32;                 // K bytes per tcgen05.mma (16 f16 / 32 e4m3)
constexpr int KSTEPS = kRowBytes / KSTEP_BYTES; // MMAs per stage

// Per-CTA shapes of the variants.  A CTA stages 128 rows of A; alone it
// stages all BN rows of B (a 192 KiB ring of one-K-block stages: 4 of 48 KiB
// for 256-wide tiles, 6 of 32 KiB for 128-wide, 8 of 24 KiB for 64-wide), in
// a pair it stages half of B (the pair's MMAs read B from both CTAs), in 3
// stages of two K blocks (64 KiB each) by default or 7 stages of one K block
// (32 KiB each): two-block stages take half as many barrier round trips per
// byte and measured 3-6% faster.
//
// In-ring conversion (FU, integer launches): the producer loads K blocks of
// the raw operands (64 bytes per row: 64 s8 or 128 packed s4) into a second
// ring, and converting warps write each into an MMA ring stage.  One CTA per
// tile: the epilogue warps, idle during the K loop, convert; both rings have
// the same depth and fit 216 KiB (6 stages for 64-wide tiles, 4 for 128-wide,
// 3 for 256-wide).  CTA pairs: six dedicated converter warps per CTA (the
// epilogue warps of a multi-wave product fold and store while the next tile is
// multiplied); 8 raw stages of 16 KiB (half the bytes of a converted K block,
// so twice the K blocks in flight per byte) and 3 MMA stages of 32 KiB.  That
// route is slower than the separate conversion pass for CTA pairs (the
// conversion and its proxy fence take longer than a K block's MMAs) and runs
// only when the pair_in_ring knob asks for it.
constexpr int kRing1 = 4 * (kBM + kBN) * kRowBytes;  // one-CTA ring bytes
constexpr int kRingFu = 216 * 1024;                  // both rings, in-ring conversion
constexpr int kRawRow = 64;                          // raw operand bytes per row and K block
constexpr int kPairFuStages = 3, kPairFuRawStages = 8;
template <int CTAS, int SUBK, int BN, bool FU = false, bool GC = false>
struct Cfg {
    static_assert(CTAS == 2 || SUBK == 1, "one CTA stages one K block at a time");
    static_assert(BN == kBN || (CTAS == 1 && (BN == 64 || BN == 128)), "narrow tiles are one-CTA tiles");
    static_assert(!FU || CTAS == 1 || SUBK == 1, "in-ring conversion stages one K block at a time");
    static_assert(!(FU && GC), "operands converted in the ring or in global memory, not both");
    static constexpr bool PFU = FU && CTAS == 2;  // pair with dedicated converter warps
    // 16 warps with per-warpgroup register budgets: pairs converting in the
    // ring, and launches converting the operands in global memory (GC).
    static constexpr bool WIDE = PFU || GC;
    static constexpr int THREADS_ = WIDE ? PAIR_FU_THREADS : THREADS;
    static constexpr int EPI_WARP0 = WIDE ? 4 : 2;  // first epilogue warp
    static constexpr int CONV_WARP0 = 12;           // first converter warp of warpgroup 3 (WIDE)
    static constexpr int SUB = SUBK;  // K blocks per stage
    static constexpr int B_ROWS = BN / CTAS;
    static constexpr int A_BLOCK = kBM * kRowBytes;     // one K block of A
    static constexpr int B_BLOCK = B_ROWS * kRowBytes;  // one K block of B
    static constexpr int A_STAGE = SUB * A_BLOCK;
    static constexpr int B_STAGE = SUB * B_BLOCK;
    static constexpr int STAGE = A_STAGE + B_STAGE;
    static constexpr int RAW_A = FU ? kBM * kRawRow : 0;              // raw A rows of a stage
    static constexpr int RAW_STAGE = FU ? (kBM + B_ROWS) * kRawRow : 0;  // raw A, then raw B
    static constexpr int STAGES = PFU ? kPairFuStages
                                  : FU ? kRingFu / (STAGE + RAW_STAGE)
                                       : CTAS == 1 ? kRing1 / STAGE : (SUBK == 1 ? 7 : 3);
    static constexpr int RSTAGES = PFU ? kPairFuRawStages : FU ? STAGES : 1;  // raw ring depth
    static constexpr int RING = STAGES * STAGE + (FU ? RSTAGES * RAW_STAGE : 0);  // bytes of both rings
    static_assert(RAW_A % 1024 == 0 && RAW_STAGE % 1024 == 0, "raw boxes start on 1024-byte boundaries");
    static constexpr int TMEM_COLS = 2 * BN;  // two accumulators of BN columns
};

template <int STAGES, int SUB, int RSTAGES = STAGES>
struct SharedTail {
    uint64_t full[STAGES * SUB];  // per K block of a stage: its operands have landed (or been converted)
    uint64_t empty[STAGES];       // per stage: its MMAs have read it
    uint64_t rfull[RSTAGES];      // in-ring conversion: the raw stage has landed
    uint64_t rempty[RSTAGES];     // ... and has been read by the converting warps
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint64_t probe_c0, probe_t0;  // clock record: SM cycles and ns at the start of work
    uint32_t tmem_base;
    AbortState abort;
};

// A single-wave launch stages C for TMA stores in the ring, which is idle once
// a CTA's only tile has been multiplied: 32 x 128 four-byte values per
// epilogue warp (four 32 x 32 blocks of 4 KiB).
constexpr int kStageC = 32 * 32 * 4;
constexpr int kStageWarp = 4 * kStageC;

template <int CTAS, int SUBK, int BN = kBN, bool FU = false>
constexpr size_t smem_bytes() {
    using C_ = Cfg<CTAS, SUBK, BN, FU>;
    return 1024 + size_t(C_::RING) + sizeof(SharedTail<C_::STAGES, SUBK, C_::RSTAGES>);
}
static_assert(smem_bytes<1, 1>() <= 232448 && smem_bytes<2, 1>() <= 232448 && smem_bytes<2, 2>() <= 232448 &&
                  smem_bytes<1, 1, 128>() <= 232448 && smem_bytes<1, 1, 64>() <= 232448 &&
                  smem_bytes<1, 1, kBN, true>() <= 232448 && smem_bytes<1, 1, 128, true>() <= 232448 &&
                  smem_bytes<1, 1, 64, true>() <= 232448 && smem_bytes<2, 1, kBN, true>() <= 232448,
              "shared memory budget");
static_assert(Cfg<1, 1, 64, true>::STAGES == 6 && Cfg<1, 1, 128, true>::STAGES == 4 &&
                  Cfg<1, 1, kBN, true>::STAGES == 3,
              "in-ring conversion depths");
// The ring staging of C and of K-split partial sums spans the first 128 KiB.
static_assert(Cfg<1, 1, 64, true>::RING >= EPI_WARPS * kStageWarp && Cfg<1, 1, kBN, true>::RING >= kBM * kBN * 4 &&
                  Cfg<1, 1, 128, true>::RING >= EPI_WARPS * kStageWarp,
              "the rings hold the C staging and the partial sums");
// A K-split cluster's partial sums: 128 rows of BN four-byte values, row r at
// r * 4 BN bytes, its 16-byte piece j at piece j ^ (r & 7) (the writers, one
// row per lane, and the readers, one piece per lane, do not conflict).
static_assert(Cfg<1, 1, kBN>::STAGES * Cfg<1, 1, kBN>::STAGE >= kBM * kBN * 4,
              "the ring holds a tile's partial sums");
static_assert(Cfg<1, 1, kBN>::STAGES * Cfg<1, 1, kBN>::STAGE >= EPI_WARPS * kStageWarp &&
                  Cfg<1, 1, 128>::STAGES * Cfg<1, 1, 128>::STAGE >= EPI_WARPS * kStageWarp &&
                  Cfg<1, 1, 64>::STAGES * Cfg<1, 1, 64>::STAGE >= EPI_WARPS * kStageWarp &&
                  Cfg<2, 1, kBN>::STAGES * Cfg<2, 1, kBN>::STAGE >= EPI_WARPS * kStageWarp &&
                  Cfg<2, 2, kBN>::STAGES * Cfg<2, 2, kBN>::STAGE >= EPI_WARPS * kStageWarp,
              "the ring holds the C staging of a single-wave launch");

__device__ __forceinline__ void tile_coords(int t, const GemmArgs &a, int &mb, int &nb) {
    const int per_group = a.group_m * a.tiles_n;
    const int g = t / per_group;
    const int first_m = g * a.group_m;
    const int gsz = min(a.tiles_m - first_m, a.group_m);
    const int r = t - g * per_group;
    mb = first_m + r % gsz;
    nb = r / gsz;
}

// Entry v of the launch's work list: whole tiles in raster order, then, when
// the last wave would leave at least half of the clusters idle, each of its
// tiles as two units over the two halves of the K range.  Both halves feed the
// tensor cores at the rate of a whole tile; the epilogue warp that finishes
// second adds the other half's partial sums (no waiting on either side).
struct WorkRef {
    int mb, nb;    // tile coordinates in units of (kBM * CTAS) x BN
    int kb0, kb1;  // K blocks of this unit
    int part;      // 0: whole tile; 1, 2: first / second K half of split tile `slot`
    int slot;
};

// The split point is a multiple of `sub` K blocks (the K blocks of one stage),
// at least one stage; a split tile has more than `sub` K blocks, so that
// neither half is empty.
__device__ __forceinline__ WorkRef work_unit(int v, const GemmArgs &a, int sub) {
    const int full = a.num_tiles - a.tail_split;
    WorkRef r;
    if (v < full) {
        tile_coords(v, a, r.mb, r.nb);
        r.kb0 = 0;
        r.kb1 = a.num_kb;
        r.part = 0;
        r.slot = 0;
    } else {
        const int u = v - full;
        r.slot = u >> 1;
        tile_coords(full + r.slot, a, r.mb, r.nb);
        const int mid = max(sub, (a.num_kb >> 1) / sub * sub);
        r.part = 1 + (u & 1);
        r.kb0 = (u & 1) ? mid : 0;
        r.kb1 = (u & 1) ? a.num_kb : mid;
    }
    return r;
}

// Partial sums of one epilogue warp's 32 x 128 slice of a split tile, stored
// as float4 [column / 4][lane] so that each warp-wide 16-byte access covers
// 512 contiguous bytes.  Integer partials are stored by bit pattern.
constexpr int kSliceWords = 32 * (kBN / 2);

__device__ __forceinline__ float4 *split_partial(const GemmArgs &a, int slice, int half) {
    return reinterpret_cast<float4 *>(a.split_part + size_t(slice * 2 + half) * kSliceWords);
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t *p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// True when the other half of this slice has already published its partial
// sums (then this warp completes the tile without publishing its own).
__device__ __forceinline__ bool split_other_done(const uint32_t *cnt, int lane) {
    uint32_t v = 0;
    if (lane == 0) v = ld_acquire_gpu(cnt);
    v = __shfl_sync(0xffffffffu, v, 0);
    __threadfence();
    return v != 0;
}

// Publish this warp's partial sums (already stored by every lane); true when
// the other half had published first, so that this warp completes the tile.
__device__ __forceinline__ bool split_publish(uint32_t *cnt, int lane) {
    __threadfence();
    __syncwarp();
    uint32_t old = 0;
    if (lane == 0) old = atom_add_acq_rel_gpu(cnt, 1u);
    old = __shfl_sync(0xffffffffu, old, 0);
    __threadfence();
    return old != 0;
}

__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ---------------------------------------------------------------- conversion
// Integer launches that convert their operands themselves (GC): converter
// warps rewrite the raw s8 / packed s4 rows of A and B into the workspace rows
// that the tensor maps read, one element at a time exactly as the separate
// pass does, in items of 2 KiB of raw operand (a few rows x kConvSlice K
// elements).  Each (panel of kConvPanel rows, K slice) has a counter that its
// items raise; a producer loads a slice of a panel once the counter holds all
// the items.  Items go in the order the tiles need them (GemmArgs::conv), so
// the first wave's MMAs start after the first slice of their panels.
constexpr int kConvSlice = 256;  // K elements per slice
constexpr int kConvPanel = 128;  // rows per panel
constexpr int kConvWarps = 6;    // converter warps per CTA (2, 3 and 12 .. 15)

template <Kind KIND>
struct ConvItem {
    static constexpr int ROWS = KIND == Kind::F16 ? 8 : 16;       // rows of 256 s8 or 128 packed-s4 bytes
    static constexpr int ITEMS = kConvPanel / ROWS;               // items per (panel, slice)
    static constexpr int VPR = 128 / ROWS;                        // 16-byte raw vectors per row
    static constexpr int EPV = KIND == Kind::F16 ? 16 : 32;       // elements per raw vector
    static constexpr int OUT = KIND == Kind::F16 ? 2 : 1;         // workspace bytes per element
    static_assert(VPR * EPV == kConvSlice && ROWS * VPR == 128, "an item is 128 vectors of 16 bytes");
};

struct ConvGeom {
    int S, PA, PB;  // K slices, panels of A, panels of B
    __device__ __forceinline__ explicit ConvGeom(const GemmArgs &a)
        : S((a.K + kConvSlice - 1) / kConvSlice), PA((a.M + kConvPanel - 1) / kConvPanel),
          PB((a.N + kConvPanel - 1) / kConvPanel) {}
    __device__ __forceinline__ int units() const { return (PA + PB) * S; }
    // Counter of (operand, panel, slice): A panels first, then B panels.
    __device__ __forceinline__ int counter(bool b, int p, int s) const { return ((b ? PA : 0) + p) * S + s; }
};

__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Unit u of the conversion order: the first wave's panels (fa of A, fb of B)
// slice by slice, then the other B panels, then the other A panels, each
// panel slice by slice.
__device__ __forceinline__ void conv_unit(const ConvGeom &g, int fa, int fb, int u, bool &is_b, int &p, int &s) {
    const int front = (fa + fb) * g.S;
    if (u < front) {
        s = u / (fa + fb);
        const int i = u - s * (fa + fb);
        is_b = i >= fa;
        p = is_b ? i - fa : i;
        return;
    }
    u -= front;
    const int rest_b = (g.PB - fb) * g.S;
    is_b = u < rest_b;
    if (!is_b) u -= rest_b;
    p = (is_b ? fb : fa) + u / g.S;
    s = u % g.S;
}

// Vector v (0 .. 127) of an item of unit (is_b, p, sl), item q of the unit:
// its raw source, its workspace destination and the elements below K that it
// holds (0: none, EPV: the whole vector).
template <Kind KIND>
__device__ __forceinline__ int conv_vec(const GemmArgs &a, bool is_b, int p, int sl, int q, int v, const uint8_t *&src,
                                        uint8_t *&dst) {
    using CI = ConvItem<KIND>;
    const int row = p * kConvPanel + q * CI::ROWS + v / CI::VPR;
    const int c = sl * kConvSlice + (v % CI::VPR) * CI::EPV;
    src = (is_b ? a.conv_b : a.conv_a) + int64_t(row) * (is_b ? a.conv_ldb : a.conv_lda) +
          (KIND == Kind::F16 ? c : c / 2);
    dst = static_cast<uint8_t *>(is_b ? a.conv_wb : a.conv_wa) + (int64_t(row) * a.conv_ldw + c) * CI::OUT;
    return row < (is_b ? a.N : a.M) ? max(0, min(CI::EPV, a.K - c)) : 0;
}

// Converter warp g of G: items g, g + G, ..., in batches of four: two items'
// loads in flight together, converted and stored, then the next two (whose
// loads overlap the first stores' drain); one device-scope fence per batch,
// then relaxed additions to the counts (fence-based release; the producers
// read the counts relaxed and fence before their loads).  Only the loaded
// vectors and the items' indices stay live across the loads (the converter
// warpgroups run in 80 registers).
template <Kind KIND>
__device__ void convert_global(const GemmArgs &a, int g, int G, int lane, AbortState *ab) {
    using CI = ConvItem<KIND>;
    const ConvGeom geom(a);
    const int total = geom.units() * CI::ITEMS;
    auto item = [&](int i) { return (i >= total || (a.stall_tile == -2 && i == 0)) ? -1 : i; };  // test hook: item 0
    for (int i0 = g; i0 < total; i0 += 4 * G) {
        if (ab->flag) return;
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
            uint4 x[2][4];
#pragma unroll
            for (int w = 0; w < 2; ++w) {
                const int it = item(i0 + (2 * half + w) * G);
                if (it < 0) continue;
                bool is_b;
                int p, sl;
                conv_unit(geom, a.conv_front_a, a.conv_front_b, it / CI::ITEMS, is_b, p, sl);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint8_t *src;
                    uint8_t *dst;
                    if (conv_vec<KIND>(a, is_b, p, sl, it % CI::ITEMS, lane + 32 * j, src, dst) == CI::EPV)
                        x[w][j] = __ldcs(reinterpret_cast<const uint4 *>(src));
                }
            }
#pragma unroll
            for (int w = 0; w < 2; ++w) {
                const int it = item(i0 + (2 * half + w) * G);
                if (it < 0) continue;
                bool is_b;
                int p, sl;
                conv_unit(geom, a.conv_front_a, a.conv_front_b, it / CI::ITEMS, is_b, p, sl);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint8_t *src;
                    uint8_t *dst;
                    const int n = conv_vec<KIND>(a, is_b, p, sl, it % CI::ITEMS, lane + 32 * j, src, dst);
                    if (n == CI::EPV) {
                        uint4 o0, o1;
                        if constexpr (KIND == Kind::F16)
                            cvt_s8_f16_x16(x[w][j], o0, o1);
                        else
                            cvt_s4_e4m3_x32(x[w][j], o0, o1);
                        reinterpret_cast<uint4 *>(dst)[0] = o0;
                        reinterpret_cast<uint4 *>(dst)[1] = o1;
                    } else {
                        for (int e = 0; e < n; ++e) {  // the ragged end of a row: no byte past K is read
                            if constexpr (KIND == Kind::F16) {
                                reinterpret_cast<uint16_t *>(dst)[e] = s8_to_f16_bits(static_cast<int8_t>(src[e]));
                            } else {
                                const uint32_t b = src[e >> 1];
                                dst[e] = s4_to_e4m3_byte((e & 1) ? (b >> 4) : b);
                            }
                        }
                    }
                }
            }
        }
        __threadfence();
        __syncwarp();
        if (lane == 0) {
            int n = 0;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const int it = item(i0 + w * G);
                if (it < 0) continue;
                bool is_b;
                int p, sl;
                conv_unit(geom, a.conv_front_a, a.conv_front_b, it / CI::ITEMS, is_b, p, sl);
                atomicAdd(a.conv_count + geom.counter(is_b, p, sl), 1u);
                ++n;
            }
            if (n) atomicAdd(a.conv_count + geom.units(), uint32_t(n));
        }
        __syncwarp();
    }
}

__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// Bounded wait of a producer until the counters i0 .. i2 (-1: none) hold
// `need` items each (`seen`: their values read earlier, relaxed); then acquire
// (fence) and order its coming TMA loads after the converters' stores (proxy
// fence).  False on timeout or abort.
__device__ __forceinline__ bool conv_wait(const uint32_t *cnt, int i0, int i1, int i2, uint32_t need, uint32_t seen,
                                          AbortState *ab, uint64_t limit) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t m = seen;;) {
        if (m >= need) break;
        const uint32_t a = i0 >= 0 ? ld_relaxed_gpu(cnt + i0) : need;
        const uint32_t b = i1 >= 0 ? ld_relaxed_gpu(cnt + i1) : need;
        const uint32_t c = i2 >= 0 ? ld_relaxed_gpu(cnt + i2) : need;
        m = min(a, min(b, c));
        if (m >= need) break;
        if (ab->flag) return false;
        if (globaltimer_ns() - t0 > limit) {
            ab->flag = 1;
            atomicCAS(&g_error_word, 0u, kErrTimeout);
            return false;
        }
    }
    fence_acq_rel_gpu();
    fence_proxy_async_global();
    return true;
}

// Split tiles added into C by TMA reductions: the first half's cluster zeroes
// the tile's C at its start and sets one flag per epilogue warp slice.  Before
// its reductions a warp waits (bounded; the zeroing happened long before in
// practice) until its slice's flag is set, then fences so that its TMA
// reductions come after the zeros.  False on timeout or abort.
__device__ __forceinline__ bool split_zeroed_wait(const uint32_t *flag, AbortState *ab, uint64_t limit, int lane) {
    uint32_t ok = 1;
    if (lane == 0) {
        const uint64_t t0 = globaltimer_ns();
        while (ld_acquire_gpu(flag) == 0) {
            if (ab->flag) {
                ok = 0;
                break;
            }
            if (globaltimer_ns() - t0 > limit) {
                ab->flag = 1;
                atomicCAS(&g_error_word, 0u, kErrTimeout);
                ok = 0;
                break;
            }
        }
        if (ok) fence_proxy_async_global();
    }
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Warp-uniform bounded wait: lane 0 polls, the outcome is broadcast.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, AbortState *ab,
                                          uint64_t limit, int lane) {
    uint32_t ok = 0;
    if (lane == 0) ok = mbar_wait(bar, parity, ab, &g_error_word, limit) ? 1u : 0u;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Bounded pause (abort path of a CTA pair, whose copies complete on the even
// CTA's barrier and cannot be awaited locally).
__device__ __forceinline__ void pause_ns(uint64_t ns) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < ns) {
    }
}

// One 32-byte store (a whole L2 sector) of eight 32-bit words; dst 32-byte aligned.
__device__ __forceinline__ void st_global_v8(uint32_t *dst, const uint32_t *w) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                 "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

template <typename T>
__device__ __forceinline__ void store_32(T *dst, const uint32_t (&v)[32], int valid, bool wide) {
    if (valid >= 32) {
        if (wide) {
#pragma unroll
            for (int i = 0; i < 4; ++i) st_global_v8(reinterpret_cast<uint32_t *>(dst) + 8 * i, &v[8 * i]);
        } else {
            uint4 *d = reinterpret_cast<uint4 *>(dst);
#pragma unroll
            for (int i = 0; i < 8; ++i) d[i] = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        }
    } else {
        uint32_t *d = reinterpret_cast<uint32_t *>(dst);
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (j < valid) d[j] = v[j];
    }
}

// A 32 x 32 block of 4-byte C through a staging buffer `stg` (1024-byte
// aligned; row `lane` holds the lane's 32 values in 128 bytes with the
// 128-byte swizzle, so that the warp's writes do not conflict), then to C at
// (col, row0) by one TMA store that clips at M and N:
//   stage_begin, stage_put for each 16-byte piece j = 0..7, stage_end.
// A store reads its buffer asynchronously; stage_begin with `wait` first
// waits until every earlier store of this warp has read its buffer.
__device__ __forceinline__ void stage_begin(int lane, bool wait) {
    if (wait) {
        if (lane == 0) bulk_wait_group_read0();
        __syncwarp();
    }
}

__device__ __forceinline__ void stage_put(uint32_t stg, int lane, int j, uint32_t a, uint32_t b, uint32_t c,
                                          uint32_t d) {
    st_shared_v4(stg + uint32_t(lane) * 128u + (uint32_t(j ^ (lane & 7)) << 4), a, b, c, d);
}

__device__ __forceinline__ void stage_end(const CUtensorMap *tmC, uint32_t stg, int lane, int col, int row0) {
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        tma_store_2d(tmC, stg, col, row0);
        bulk_commit_group();
    }
}

// `add`: the block is added into C (FP32 or int32, by the tensor map's type)
// by a TMA reduction instead of stored.
__device__ __forceinline__ void tma_store_block(const CUtensorMap *tmC, uint32_t stg, const uint32_t (&v)[32],
                                                int lane, int col, int row0, bool wait, bool add = false) {
    stage_begin(lane, wait);
#pragma unroll
    for (int j = 0; j < 8; ++j) stage_put(stg, lane, j, v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        if (add)
            tma_reduce_add_2d(tmC, stg, col, row0);
        else
            tma_store_2d(tmC, stg, col, row0);
        bulk_commit_group();
    }
}

// Scaled integer epilogue (dequantisation): for the HALF columns col0 .. of
// `row`, value = rn(rn(rn(float(acc)) * sa) * sb) in FP32, in that order and
// without contraction, then rounded to nearest-even in the output type.
// Columns at or beyond N are not written.
template <int HALF>
__device__ __forceinline__ void store_scaled_row(const GemmArgs &args, int row, int col0,
                                                 const int32_t (&acc)[HALF], const CUtensorMap *tmC,
                                                 bool use_tma, uint32_t stg, int lane, int row0, bool pending) {
    const float sa = (args.scale_a && row < args.M) ? __ldg(args.scale_a + row) : 1.0f;
#pragma unroll
    for (int c = 0; c < HALF / 32; ++c) {
        const int cc = col0 + 32 * c;
        if (cc >= args.N) break;
        const int valid = min(32, args.N - cc);
        if (use_tma) {
            // FP32 output through the staging buffer (the whole warp takes part).
            const uint32_t blk = stg + uint32_t(c * kStageC);
            stage_begin(lane, pending && c == 0);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float f4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int jj = 4 * j + e;
                    const float sb = (args.scale_b && jj < valid) ? __ldg(args.scale_b + cc + jj) : 1.0f;
                    f4[e] = __fmul_rn(__fmul_rn(__int2float_rn(acc[32 * c + jj]), sa), sb);
                }
                stage_put(blk, lane, j, __float_as_uint(f4[0]), __float_as_uint(f4[1]), __float_as_uint(f4[2]),
                          __float_as_uint(f4[3]));
            }
            stage_end(tmC, blk, lane, cc, row0);
            continue;
        }
        if (row >= args.M) continue;
        float f[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const float sb = (args.scale_b && j < valid) ? __ldg(args.scale_b + cc + j) : 1.0f;
            f[j] = __fmul_rn(__fmul_rn(__int2float_rn(acc[32 * c + j]), sa), sb);
        }
        if (args.out_mode == OUT_F32) {
            uint32_t v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(f[j]);
            store_32(reinterpret_cast<float *>(args.C) + int64_t(row) * args.ldc + cc, v, valid, args.c_wide);
        } else {
            // 16-bit outputs: pairs packed into 32-bit words, 64 bytes per 32 columns.
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                uint32_t lo, hi;
                if (args.out_mode == OUT_BF16) {
                    lo = __bfloat16_as_ushort(__float2bfloat16_rn(f[2 * j]));
                    hi = __bfloat16_as_ushort(__float2bfloat16_rn(f[2 * j + 1]));
                } else {
                    lo = __half_as_ushort(__float2half_rn(f[2 * j]));
                    hi = __half_as_ushort(__float2half_rn(f[2 * j + 1]));
                }
                w[j] = lo | (hi << 16);
            }
            uint16_t *dst = reinterpret_cast<uint16_t *>(args.C) + int64_t(row) * args.ldc + cc;
            if (valid == 32 && args.c_wide) {
                st_global_v8(reinterpret_cast<uint32_t *>(dst), &w[0]);
                st_global_v8(reinterpret_cast<uint32_t *>(dst) + 8, &w[8]);
            } else if (valid == 32) {
                uint4 *d = reinterpret_cast<uint4 *>(dst);
#pragma unroll
                for (int i = 0; i < 4; ++i) d[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (j < valid) dst[j] = static_cast<uint16_t>(w[j >> 1] >> ((j & 1) * 16));
            }
        }
    }
}

// 32 FP16 accumulators (the low half of each 32-bit tensor-memory column) to
// dst[0 .. valid), valid capped at 32; `wide`: two 32-byte stores.
__device__ __forceinline__ void store_f16acc_32(uint16_t *dst, const uint32_t (&r)[32], int valid, bool wide) {
    if (valid >= 32) {
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) w[j] = (r[2 * j] & 0xFFFFu) | (r[2 * j + 1] << 16);
        if (wide) {
            st_global_v8(reinterpret_cast<uint32_t *>(dst), &w[0]);
            st_global_v8(reinterpret_cast<uint32_t *>(dst) + 8, &w[8]);
        } else {
            uint4 *d = reinterpret_cast<uint4 *>(dst);
#pragma unroll
            for (int i = 0; i < 4; ++i) d[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (j < valid) dst[j] = static_cast<uint16_t>(r[j]);
    }
}

// Epilogue of one K half of a split tile (FP32 or FP16 accumulators), for
// this warp's 32 x 128 slice at tensor-memory address t_acc: publish the
// partial sums (to `mine`), or, when the other half has published first, add
// its partial sums (`other`; in FP32, the same bits whichever half adds) and
// store C.  crow points at C[row][col0] (null when row >= M); `valid` is the
// number of columns of the slice below N; `wide`: 32-byte C stores.  Inlined:
// as an out-of-line call from the CTA-pair kernel its 32-byte stores after the
// first 32 columns were lost (caught by the split-tile parity tests).
template <int EPI>
__device__ __forceinline__ void split_epilogue(uint32_t t_acc, uint32_t *cnt, float4 *mine, const float4 *other,
                                               void *crow, int valid, bool wide, int lane) {
    bool finish = split_other_done(cnt, lane);
    if (!finish) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            uint32_t r[32];
            tmem_ld_32cols(t_acc + uint32_t(32 * c), r);
            tmem_ld_wait();
            float f[32];
#pragma unroll
            for (int j = 0; j < 32; ++j)
                f[j] = (EPI == EPI_F16ACC) ? __half2float(__ushort_as_half(static_cast<uint16_t>(r[j]))) : __uint_as_float(r[j]);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                mine[(8 * c + i) * 32 + lane] = make_float4(f[4 * i], f[4 * i + 1], f[4 * i + 2], f[4 * i + 3]);
        }
        finish = split_publish(cnt, lane);
    }
    if (!finish) return;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld_32cols(t_acc + uint32_t(32 * c), r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 o = __ldcg(other + (8 * c + i) * 32 + lane);
            const float ov[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = 4 * i + e;
                if constexpr (EPI == EPI_F16ACC)
                    r[j] = __half_as_ushort(
                        __float2half_rn(__fadd_rn(__half2float(__ushort_as_half(static_cast<uint16_t>(r[j]))), ov[e])));
                else
                    r[j] = __float_as_uint(__fadd_rn(__uint_as_float(r[j]), ov[e]));
            }
        }
        const int v = valid - 32 * c;
        if (crow != nullptr && v > 0) {
            if constexpr (EPI == EPI_F16ACC)
                store_f16acc_32(static_cast<uint16_t *>(crow) + 32 * c, r, v, wide);
            else
                store_32(static_cast<float *>(crow) + 32 * c, r, v, wide);
        }
    }
}

// K-split clusters: CTA `krank` of `ks` multiplies K blocks [kb0, kb1) of the
// unit, an even share (the first num_kb % ks CTAs take one block more).
__device__ __forceinline__ void ksplit_range(WorkRef &w, int krank, int ks) {
    const int n = w.kb1 - w.kb0, q = n / ks, r = n % ks;
    const int b = w.kb0 + krank * q + min(krank, r);
    w.kb0 = b;
    w.kb1 = b + q + (krank < r ? 1 : 0);
}

// 32 four-byte partial sums of local row `row`, columns 4 * piece0 .., into
// the partial-sum layout (rows of PROW bytes) at shared address `base`.
template <int PROW>
__device__ __forceinline__ void put_partial(uint32_t base, int row, int piece0, const uint32_t (&v)[32]) {
    const uint32_t rb = base + uint32_t(row) * PROW;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        st_shared_v4(rb + (uint32_t((piece0 + i) ^ (row & 7)) << 4), v[4 * i], v[4 * i + 1], v[4 * i + 2],
                     v[4 * i + 3]);
}

// Four consecutive results of one row to C (row-major, ldc elements) at
// column `col`; `valid` of them lie below N.  16-byte (4-byte C) or 8-byte
// (2-byte C) stores, aligned because C rows start on 16-byte boundaries.
template <typename T>
__device__ __forceinline__ void store_4(T *dst, const T (&v)[4], int valid) {
    if (valid >= 4) {
        if constexpr (sizeof(T) == 4) {
            *reinterpret_cast<uint4 *>(dst) = make_uint4(reinterpret_cast<const uint32_t &>(v[0]),
                                                         reinterpret_cast<const uint32_t &>(v[1]),
                                                         reinterpret_cast<const uint32_t &>(v[2]),
                                                         reinterpret_cast<const uint32_t &>(v[3]));
        } else {
            *reinterpret_cast<uint2 *>(dst) = make_uint2(uint32_t(v[0]) | (uint32_t(v[1]) << 16),
                                                         uint32_t(v[2]) | (uint32_t(v[3]) << 16));
        }
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (e < valid) dst[e] = v[e];
    }
}

// Sum of the KS partials of four consecutive outputs (row, col ..), in rank
// order, stored to C: FP32 sums with round-to-nearest additions (FP16
// accumulators were widened exactly to FP32 and the sum is rounded to binary16
// once), int32 sums wrapping mod 2^32, then the output conversion.
template <int EPI, int KS>
__device__ __forceinline__ void ksplit_finish(const GemmArgs &args, int row, int col, const uint4 (&p)[KS]) {
    const int valid = args.N - col;
    if constexpr (EPI == EPI_INT) {
        uint32_t s[4] = {p[0].x, p[0].y, p[0].z, p[0].w};
#pragma unroll
        for (int k = 1; k < KS; ++k) {
            s[0] += p[k].x;
            s[1] += p[k].y;
            s[2] += p[k].z;
            s[3] += p[k].w;
        }
        if (args.out_mode == OUT_S32) {
            const int32_t v[4] = {int32_t(s[0]), int32_t(s[1]), int32_t(s[2]), int32_t(s[3])};
            store_4(reinterpret_cast<int32_t *>(args.C) + int64_t(row) * args.ldc + col, v, valid);
            return;
        }
        const float sa = args.scale_a ? __ldg(args.scale_a + row) : 1.0f;
        float f[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float sb = (args.scale_b && e < valid) ? __ldg(args.scale_b + col + e) : 1.0f;
            f[e] = __fmul_rn(__fmul_rn(__int2float_rn(int32_t(s[e])), sa), sb);
        }
        if (args.out_mode == OUT_F32) {
            store_4(reinterpret_cast<float *>(args.C) + int64_t(row) * args.ldc + col, f, valid);
        } else {
            uint16_t h[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                h[e] = args.out_mode == OUT_BF16 ? __bfloat16_as_ushort(__float2bfloat16_rn(f[e]))
                                                 : __half_as_ushort(__float2half_rn(f[e]));
            store_4(reinterpret_cast<uint16_t *>(args.C) + int64_t(row) * args.ldc + col, h, valid);
        }
    } else {
        float f[4] = {__uint_as_float(p[0].x), __uint_as_float(p[0].y), __uint_as_float(p[0].z),
                      __uint_as_float(p[0].w)};
#pragma unroll
        for (int k = 1; k < KS; ++k) {
            f[0] = __fadd_rn(f[0], __uint_as_float(p[k].x));
            f[1] = __fadd_rn(f[1], __uint_as_float(p[k].y));
            f[2] = __fadd_rn(f[2], __uint_as_float(p[k].z));
            f[3] = __fadd_rn(f[3], __uint_as_float(p[k].w));
        }
        if constexpr (EPI == EPI_F16ACC) {
            uint16_t h[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) h[e] = __half_as_ushort(__float2half_rn(f[e]));
            store_4(reinterpret_cast<uint16_t *>(args.C) + int64_t(row) * args.ldc + col, h, valid);
        } else {
            store_4(reinterpret_cast<float *>(args.C) + int64_t(row) * args.ldc + col, f, valid);
        }
    }
}

// Completion of a K-split tile of BN columns: this CTA (`krank` of KS) owns
// local rows krank * 128/KS .. of the tile (mb, nb), BN / 4 16-byte pieces per
// row.  The 256 epilogue threads take consecutive pieces (a warp covers 512
// contiguous bytes of C per store), two at a time with all 2 x KS loads in
// flight before the sums (distributed shared memory is latency-bound; this
// CTA's own partial sums are read locally).  Every thread makes the same
// number of passes; once the last pass's loads are done the thread arrives on
// the cluster barrier (it reads no peer's memory after that), so that the
// barrier's latency overlaps the last sums and stores.
template <int EPI, int KS, int BN>
__device__ __forceinline__ void ksplit_complete(const GemmArgs &args, int mb, int nb, int krank, uint32_t base,
                                                int ew, int lane) {
    constexpr int R = kBM / KS;
    constexpr int PPR = BN / 4;     // pieces per row
    constexpr int PROW = BN * 4;    // partial-sum row bytes
    constexpr int NT = EPI_WARPS * 32;
    static_assert((R * PPR) % (2 * NT) == 0, "whole passes of two pieces per thread");
#pragma unroll 1
    for (int i0 = ew * 32 + lane; i0 < R * PPR; i0 += 2 * NT) {
        uint4 p[2][KS];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int idx = i0 + u * NT;
            const int lr = krank * R + idx / PPR;
            const int piece = idx % PPR;
            const uint32_t addr = base + uint32_t(lr) * PROW + (uint32_t(piece ^ (lr & 7)) << 4);
#pragma unroll
            for (int k = 0; k < KS; ++k)
                p[u][k] = k == krank ? ld_shared_v4(addr) : ld_shared_cluster_v4(mapa_shared(addr, uint32_t(k)));
        }
        if (i0 + 2 * NT >= R * PPR) cluster_arrive();
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int idx = i0 + u * NT;
            const int row = mb * kBM + krank * R + idx / PPR;
            const int col = nb * BN + 4 * (idx % PPR);
            if (row < args.M && col < args.N) ksplit_finish<EPI, KS>(args, row, col, p[u]);
        }
    }
}

// CTA r of a pair owns rows 128 r .. 128 r + 127 of the 256 x 256 tile and
// stages B rows 128 r .. 128 r + 127.  The even CTA issues the MMAs for both;
// its full barriers collect both CTAs' copies, its commits arrive on both
// CTAs' empty / accumulator-full barriers, and both CTAs' epilogues release
// accumulator buffers on its acc_empty barriers.
template <Kind KIND, bool B_MN, int EPI, int CTAS, int SUBK, int KS, int BN, bool FU = false, int PAIRS = 1,
          bool GC = false>
__global__ void __launch_bounds__(Cfg<CTAS, SUBK, BN, FU, GC>::THREADS_, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmC, const GemmArgs args) {
    static_assert(!(B_MN && KIND == Kind::E4M3), "MN-major B is used by the FP16 path only");
    static_assert(KS == 1 || CTAS == 1, "K-split clusters of one-CTA tiles");
    static_assert(!FU || (EPI == EPI_INT && !B_MN), "in-ring conversion: integer launches with K-major B");
    static_assert(PAIRS == 1 || (CTAS == 2 && SUBK == 2 && KS == 1 && BN == kBN && !FU && !GC),
                  "two pairs per cluster: two-block pair stages, operands converted by the pass");
    static_assert(!GC || (EPI == EPI_INT && !B_MN && KS == 1 && BN == kBN && PAIRS == 1),
                  "conversion in global memory: integer launches of 256-wide tiles with K-major B");
    constexpr bool INT_OUT = EPI == EPI_INT;
    constexpr int HALF = BN / 2;      // columns of an epilogue warp's slice
    constexpr int NCH = HALF / 32;    // 32-column chunks of a slice
    using C_ = Cfg<CTAS, SUBK, BN, FU, GC>;
    constexpr int TMEM_COLS = C_::TMEM_COLS;
    constexpr int STAGES = C_::STAGES;
    extern __shared__ uint8_t smem_raw[];
    // 128-byte swizzle atoms must sit on 1024-byte boundaries.
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    uint8_t *a_ring = smem;
    uint8_t *b_ring = smem + STAGES * C_::A_STAGE;
    uint8_t *raw_ring = smem + STAGES * C_::STAGE;  // in-ring conversion only
    using Tail = SharedTail<STAGES, C_::SUB, C_::RSTAGES>;
    constexpr bool PFU = C_::PFU;
    constexpr bool WIDE = C_::WIDE;
    constexpr int EPI_WARP0 = C_::EPI_WARP0;
    constexpr int PSTAGES = FU ? C_::RSTAGES : STAGES;  // the producer's ring
    Tail *st = reinterpret_cast<Tail *>(smem + C_::RING);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const uint64_t limit = args.wait_limit_ns;
    constexpr int CL = CTAS * KS * PAIRS;  // CTAs per cluster
    const uint32_t crank = (CL == 1) ? 0u : cluster_ctarank();
    const uint32_t rank = (CTAS == 1) ? 0u : (PAIRS == 1 ? crank : (crank & 1u));  // CTA of a pair
    const int krank = (KS == 1) ? 0 : int(crank);    // K share of a K-split cluster
    // Two pairs per cluster (PAIRS = 2): pair pp computes tile column 2 nb + pp of
    // unit (mb, nb); both pairs use the same rows of A, and each CTA loads half of
    // its rows and multicasts them to itself and its counterpart in the other pair.
    const uint32_t pp = (PAIRS == 2) ? (crank >> 1) : 0u;
    const uint32_t leader = (PAIRS == 2) ? (crank & ~1u) : 0u;  // even CTA of this CTA's pair
    constexpr uint16_t kAllMask = uint16_t((1u << CL) - 1u);
    const uint16_t pair_mask = uint16_t(0x3u << (2u * pp));
    const int cluster = blockIdx.x / CL;
    const int nclusters = gridDim.x / CL;

    if (threadIdx.x == 0) {
        // In-ring conversion: a stage is full once every converting warp has
        // converted its share of the raw stage into it (a pair's converter
        // warps of both CTAs arrive on the even CTA's barrier).
        constexpr uint32_t conv_arrivals = PFU ? (CONV_WARPS + 2) * CTAS : EPI_WARPS;
        for (int s = 0; s < STAGES; ++s) {
            for (int sb = 0; sb < C_::SUB; ++sb) mbar_init(&st->full[s * C_::SUB + sb], FU ? conv_arrivals : 1);
            mbar_init(&st->empty[s], PAIRS);  // one MMA commit per pair reading the stage
        }
        for (int s = 0; s < C_::RSTAGES; ++s) {
            mbar_init(&st->rfull[s], 1);
            mbar_init(&st->rempty[s], PFU ? CONV_WARPS + 2 : EPI_WARPS);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&st->acc_full[b], 1);
            mbar_init(&st->acc_empty[b], EPI_WARPS * CTAS);
        }
        mbar_init(&st->drain, 1);
        st->abort.flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (args.c_tma) tma_prefetch_desc(&tmC);
    }
    if (warp == 1) {
        tmem_alloc<CTAS>(&st->tmem_base, TMEM_COLS);
        tmem_relinquish<CTAS>();
    }
    tc_fence_before_sync();
    if constexpr (CTAS == 1)
        __syncthreads();
    else
        cluster_sync();
    tc_fence_after_sync();
    const uint32_t tmem_base = st->tmem_base;
    // Global memory from here on: after the previous kernel of the stream.
    griddep_wait();
    griddep_launch_dependents();
    if (args.clock_probe != nullptr && threadIdx.x == 0) {
        st->probe_t0 = globaltimer_ns();
        st->probe_c0 = sm_clock64();
    }

    constexpr int K_ELEMS = (KIND == Kind::F16) ? kRowBytes / 2 : kRowBytes;
    static_assert(!GC || kConvSlice % (K_ELEMS * C_::SUB) == 0, "a stage lies within one conversion slice");

    if (warp < EPI_WARP0 || (WIDE && warp >= C_::CONV_WARP0)) {
        // Producer, MMA issuer and converter warps.  With the 16-warp layout
        // their warpgroups (0 and 3) first lower their register budget together.
        if constexpr (WIDE) regs_dec<kRegsLow>();
        if (warp == 0) {
            // ------------------------------------------------------ TMA producer
            if (lane == 0) {
                // L2 policies: A panels are re-read by every N tile of a raster group,
                // B panels only by the M tiles of one group running at the same time.
                const bool hint = args.l2_hint != 0;
                uint64_t pol_a = 0, pol_b = 0;
                if (args.l2_hint == 1 || args.l2_hint == 2) pol_a = l2_policy_evict_last();
                if (args.l2_hint == 1) pol_b = l2_policy_evict_first();
                if (args.l2_hint == 2) pol_b = l2_policy_evict_normal();
                if (args.l2_hint == 3) pol_a = pol_b = l2_policy_evict_normal();
                int s = 0;
                uint32_t ph = 0;
                uint32_t outstanding = 0, out_phase = 0;  // per-stage bits of issued copies
                bool ok = true;
                // Conversion in global memory: once every item is done no slice
                // is checked again; until then each new slice of this CTA's A
                // panel and B panel(s) is awaited before its loads.
                bool conv_all = !GC;
                for (int t = cluster; t < args.num_vunits && ok; t += nclusters) {
                    WorkRef wr = work_unit(t, args, C_::SUB);
                    if constexpr (KS > 1) ksplit_range(wr, krank, KS);
                    const int m0 = wr.mb * (kBM * CTAS) + int(rank) * kBM;
                    const int n0 = (wr.nb * PAIRS + int(pp)) * BN + int(rank) * C_::B_ROWS;
                    int conv_sl = -1, conv_pre_sl = -1;
                    uint32_t conv_pre = 0;
                    if constexpr (GC) {
                        if (!conv_all) {
                            const ConvGeom geom(args);
                            conv_all = ld_relaxed_gpu(args.conv_count + geom.units()) >=
                                       uint32_t(geom.units() * ConvItem<KIND>::ITEMS);
                            if (conv_all) {
                                fence_acq_rel_gpu();
                                fence_proxy_async_global();
                            }
                        }
                    }
                    for (int kb = wr.kb0; kb < wr.kb1; kb += C_::SUB) {
                        // The stage is free once its MMAs (in-ring conversion: its
                        // converting warps) have read it.
                        if (!mbar_wait(FU ? &st->rempty[s] : &st->empty[s], ph ^ 1u, &st->abort, &g_error_word, limit)) {
                            ok = false;
                            break;
                        }
                        outstanding &= ~(1u << s);
                        if constexpr (GC) {
                            const int sl = kb * K_ELEMS / kConvSlice;  // a stage lies within one slice
                            if (!conv_all && sl != conv_sl) {
                                const ConvGeom geom(args);
                                const int pa = m0 / kConvPanel, pb = n0 / kConvPanel;
                                auto idx = [&](int s2, int &ia, int &ib0, int &ib1) {
                                    ia = pa < geom.PA ? geom.counter(false, pa, s2) : -1;
                                    ib0 = pb < geom.PB ? geom.counter(true, pb, s2) : -1;
                                    ib1 = (C_::B_ROWS > kConvPanel && pb + 1 < geom.PB) ? geom.counter(true, pb + 1, s2)
                                                                                       : -1;
                                };
                                int ia, ib0, ib1;
                                idx(sl, ia, ib0, ib1);
                                // The counts read a slice ago, when they were for this slice.
                                const uint32_t seen = conv_pre_sl == sl ? conv_pre : 0u;
                                if (!conv_wait(args.conv_count, ia, ib0, ib1, uint32_t(ConvItem<KIND>::ITEMS), seen,
                                               &st->abort, limit)) {
                                    ok = false;
                                    break;
                                }
                                conv_sl = sl;
                                // Read the next slice's counts now (relaxed: the value is
                                // used at that slice, so this load does not stall here).
                                conv_pre_sl = -1;
                                if (sl + 1 < geom.S) {
                                    idx(sl + 1, ia, ib0, ib1);
                                    const uint32_t need = ConvItem<KIND>::ITEMS;
                                    const uint32_t a0 = ia >= 0 ? ld_relaxed_gpu(args.conv_count + ia) : need;
                                    const uint32_t b0 = ib0 >= 0 ? ld_relaxed_gpu(args.conv_count + ib0) : need;
                                    const uint32_t b1 = ib1 >= 0 ? ld_relaxed_gpu(args.conv_count + ib1) : need;
                                    conv_pre = min(a0, min(b0, b1));
                                    conv_pre_sl = sl + 1;
                                }
                            }
                        }
                        const bool stall = (t == args.stall_tile && kb == wr.kb0 && rank == 0);
                        if (!stall) {
                            uint8_t *a_dst = a_ring + s * C_::A_STAGE;
                            uint8_t *b_dst = b_ring + s * C_::B_STAGE;
                            if constexpr (FU) {
                                // Raw K block: 128 rows of A, then BN rows of B, 64 bytes each.
                                uint8_t *r_dst = raw_ring + s * C_::RAW_STAGE;
                                mbar_arrive_expect_tx(&st->rfull[s], C_::RAW_STAGE);
                                if (hint) {
                                    tma_load_2d_hint(r_dst, &tmA, &st->rfull[s], kb * kRawRow, m0, pol_a);
                                    tma_load_2d_hint(r_dst + C_::RAW_A, &tmB, &st->rfull[s], kb * kRawRow, n0, pol_b);
                                } else {
                                    tma_load_2d(r_dst, &tmA, &st->rfull[s], kb * kRawRow, m0);
                                    tma_load_2d(r_dst + C_::RAW_A, &tmB, &st->rfull[s], kb * kRawRow, n0);
                                }
                                outstanding |= 1u << s;
                                out_phase = (out_phase & ~(1u << s)) | (ph << s);
                            } else if constexpr (CTAS == 1) {
                                mbar_arrive_expect_tx(&st->full[s], C_::STAGE);
                                auto load = [&](void *dst, const CUtensorMap *map, int x, int y, uint64_t pol) {
                                    if (hint)
                                        tma_load_2d_hint(dst, map, &st->full[s], x, y, pol);
                                    else
                                        tma_load_2d(dst, map, &st->full[s], x, y);
                                };
                                load(a_dst, &tmA, kb * K_ELEMS, m0, pol_a);
                                if constexpr (B_MN) {
    #pragma unroll
                                    for (int i = 0; i < C_::B_ROWS / 64; ++i)
                                        load(b_dst + i * (K_ELEMS * 128), &tmB, n0 + 64 * i, kb * K_ELEMS, pol_b);
                                } else {
                                    load(b_dst, &tmB, kb * K_ELEMS, n0, pol_b);
                                }
                                outstanding |= 1u << s;
                                out_phase = (out_phase & ~(1u << s)) | (ph << s);
                            } else {
                                // Both CTAs' copies of a K block complete on the even CTA's
                                // full barrier of that block, which alone expects the pair's
                                // bytes; each block has its own barrier, so that the MMAs
                                // start on the first block of a stage while the second lands.
                                // A block past K reads as zeros.
    #pragma unroll
                                for (int sb = 0; sb < C_::SUB; ++sb) {
                                    uint64_t *fb = &st->full[s * C_::SUB + sb];
                                    if (rank == 0) mbar_arrive_expect_tx(fb, CTAS * (C_::A_BLOCK + C_::B_BLOCK));
                                    const uint32_t bar = mapa_shared(smem_u32(fb), leader);
                                    auto load = [&](void *dst, const CUtensorMap *map, int x, int y, uint64_t pol) {
                                        if (hint)
                                            tma_load_2d_pair_hint(dst, map, bar, x, y, pol);
                                        else
                                            tma_load_2d_pair(dst, map, bar, x, y);
                                    };
                                    if constexpr (PAIRS == 2) {
                                        // Half pp of this CTA's 128 A rows (a 64-row box), to
                                        // this CTA and its counterpart in the other pair.
                                        tma_load_2d_pair_mc(a_dst + sb * C_::A_BLOCK + pp * (C_::A_BLOCK / 2), &tmA, bar,
                                                            (kb + sb) * K_ELEMS, m0 + int(pp) * (kBM / 2),
                                                            uint16_t((1u << rank) | (1u << (rank + 2))));
                                    } else {
                                        load(a_dst + sb * C_::A_BLOCK, &tmA, (kb + sb) * K_ELEMS, m0, pol_a);
                                    }
                                    if constexpr (B_MN) {
    #pragma unroll
                                        for (int i = 0; i < C_::B_ROWS / 64; ++i)
                                            load(b_dst + sb * C_::B_BLOCK + i * (K_ELEMS * 128), &tmB, n0 + 64 * i,
                                                 (kb + sb) * K_ELEMS, pol_b);
                                    } else {
                                        load(b_dst + sb * C_::B_BLOCK, &tmB, (kb + sb) * K_ELEMS, n0, pol_b);
                                    }
                                }
                            }
                        }
                        if (++s == PSTAGES) {
                            s = 0;
                            ph ^= 1u;
                        }
                    }
                }
                if (!ok) {
                    // Abort: let every copy this thread issued land before the CTA exits.
                    if constexpr (CTAS == 1 || FU) {
                        for (int q = 0; q < PSTAGES; ++q)
                            if (outstanding & (1u << q))
                                mbar_wait(FU ? &st->rfull[q] : &st->full[q], (out_phase >> q) & 1u, nullptr, nullptr, limit);
                    } else {
                        pause_ns(200000);  // copies complete on the even CTA's barrier: allow 200 us
                    }
                }
            }
            __syncwarp();
        } else if (warp == 1) {
            // ------------------------------------------------------ MMA issuer
            if (lane == 0 && rank == 0) {
                constexpr uint32_t IDESC =
                    instr_desc(EPI == EPI_F16ACC ? 0u : 1u, 0u, 0u, B_MN, kBM * CTAS,
                               BN);  // F16 x F16 or E4M3 x E4M3 -> F32 (or F16 accumulators)
                const uint32_t a_base = smem_u32(a_ring);
                const uint32_t b_base = smem_u32(b_ring);
                int s = 0;
                uint32_t ph = 0;
                int abuf = 0;
                uint32_t aph = 0;
                bool ok = true;
                for (int t = cluster; t < args.num_vunits && ok; t += nclusters) {
                    WorkRef wr = work_unit(t, args, C_::SUB);
                    if constexpr (KS > 1) ksplit_range(wr, krank, KS);
                    const int nchunks = (wr.kb1 - wr.kb0 + args.kb_per_chunk - 1) / args.kb_per_chunk;
                    for (int ch = 0; ch < nchunks && ok; ++ch) {
                        if (!mbar_wait(&st->acc_empty[abuf], aph ^ 1u, &st->abort, &g_error_word, limit)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after_sync();
                        const uint32_t d_tmem = tmem_base + uint32_t(abuf * BN);
                        const int kb0 = wr.kb0 + ch * args.kb_per_chunk;
                        const int kb1 = min(wr.kb1, kb0 + args.kb_per_chunk);
                        for (int kb = kb0; kb < kb1 && ok; kb += C_::SUB) {
                            const uint32_t a_addr = a_base + s * C_::A_STAGE;
                            const uint32_t b_addr = b_base + s * C_::B_STAGE;
    #pragma unroll
                            for (int kk = 0; kk < KSTEPS * C_::SUB; ++kk) {
                                const int k = kk % KSTEPS;
                                if (k == 0) {
                                    // The next K block of the stage has landed.
                                    if (!mbar_wait(&st->full[s * C_::SUB + kk / KSTEPS], ph, &st->abort, &g_error_word,
                                                   limit)) {
                                        ok = false;
                                        break;
                                    }
                                    tc_fence_after_sync();
                                }
                                const uint32_t a_blk = a_addr + (kk / KSTEPS) * C_::A_BLOCK;
                                const uint32_t b_blk = b_addr + (kk / KSTEPS) * C_::B_BLOCK;
                                const uint64_t adesc = smem_desc_sw128(a_blk + k * KSTEP_BYTES, 16, 1024);
                                uint64_t bdesc;
                                if constexpr (B_MN)
                                    bdesc = smem_desc_sw128(b_blk + k * (16 * 128), K_ELEMS * 128, 1024);
                                else
                                    bdesc = smem_desc_sw128(b_blk + k * KSTEP_BYTES, 16, 1024);
                                const uint32_t acc = (kb > kb0 || kk > 0) ? 1u : 0u;
                                mma<CTAS, KIND == Kind::E4M3>(d_tmem, adesc, bdesc, IDESC, acc);
                            }
                            if (!ok) break;
                            if constexpr (CTAS == 1)
                                mma_commit<1>(&st->empty[s]);
                            else
                                mma_commit_pair(&st->empty[s], kAllMask);  // every CTA that writes the stage
                            if (++s == STAGES) {
                                s = 0;
                                ph ^= 1u;
                            }
                        }
                        if (!ok) break;
                        if constexpr (CTAS == 1)
                            mma_commit<1>(&st->acc_full[abuf]);
                        else
                            mma_commit_pair(&st->acc_full[abuf], pair_mask);
                        if (++abuf == 2) {
                            abuf = 0;
                            aph ^= 1u;
                        }
                    }
                }
                if (!ok) {
                    // Abort: wait for the MMAs already issued before tensor memory is freed.
                    mma_commit<CTAS>(&st->drain);
                    mbar_wait(&st->drain, 0, nullptr, nullptr, limit);
                }
            }
            __syncwarp();
        } else if (PFU && warp >= 2) {
            // ------------------------------------------------------ converters
            // CTA pairs with in-ring conversion: six converter warps (2, 3 and
            // 12 .. 15) write each K block of this CTA's raw A (128 rows) and
            // raw B (128 rows), 64 bytes per row, into the MMA stage in the
            // operand type: a 16-byte piece i (row g = i / 4, piece p = i % 4)
            // becomes chunks 2p and 2p + 1 of row g, placed by the 128-byte
            // swizzle (chunk j of row g at j ^ (g & 7)).
            // The raw and MMA rings have their own depths and phases.  The pair's
            // MMAs read both CTAs' stages: each warp's arrival on the even CTA's
            // full barrier follows a proxy fence.
            if constexpr (PFU) {
                // Converter threads: warps 2, 3 and 12 .. 15 (192 threads); thread
                // ctid takes pieces ctid, ctid + 192, ... of each K block, four
                // loads in flight before their conversions and stores.
                constexpr int CT = 32 * (CONV_WARPS + 2);
                constexpr int PIECES = (kBM + C_::B_ROWS) * kRawRow / 16;
                constexpr int ITERS = (PIECES + CT - 1) / CT;
                const int ctid = warp < EPI_WARP0 ? int(threadIdx.x) - 64 : int(threadIdx.x) - 32 * C_::CONV_WARP0 + 64;
                int q = 0, r = 0;
                uint32_t qph = 0, rph = 0;
                bool ok = true;
                for (int t = cluster; t < args.num_vunits && ok; t += nclusters) {
                    const WorkRef wr = work_unit(t, args, C_::SUB);
                    for (int kb = wr.kb0; kb < wr.kb1; ++kb) {
                        if (!warp_wait(&st->rfull[r], rph, &st->abort, limit, lane) ||
                            !warp_wait(&st->empty[q], qph ^ 1u, &st->abort, limit, lane)) {
                            ok = false;
                            break;
                        }
                        // Every lane observes both completed phases before its accesses.
                        mbar_try_wait(&st->rfull[r], rph);
                        mbar_try_wait(&st->empty[q], qph ^ 1u);
                        const uint32_t raw = smem_u32(raw_ring) + uint32_t(r * C_::RAW_STAGE);
                        const uint32_t dst_a = smem_u32(a_ring) + uint32_t(q * C_::A_STAGE);
                        const uint32_t dst_b = smem_u32(b_ring) + uint32_t(q * C_::B_STAGE);
#pragma unroll
                        for (int it0 = 0; it0 < ITERS; it0 += 4) {
                            uint4 x[4];
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const int i = (it0 + u) * CT + ctid;
                                if (it0 + u < ITERS && i < PIECES) x[u] = ld_shared_v4(raw + uint32_t(i) * 16u);
                            }
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const int i = (it0 + u) * CT + ctid;
                                if (it0 + u >= ITERS || i >= PIECES) continue;
                                const int g = i >> 2, p = i & 3;
                                uint4 o0, o1;
                                if constexpr (KIND == Kind::F16)
                                    cvt_s8_f16_x16(x[u], o0, o1);
                                else
                                    cvt_s4_e4m3_x32(x[u], o0, o1);
                                const uint32_t row = g < kBM ? dst_a + uint32_t(g) * 128u : dst_b + uint32_t(g - kBM) * 128u;
                                st_shared_v4(row + (uint32_t((2 * p) ^ (g & 7)) << 4), o0.x, o0.y, o0.z, o0.w);
                                st_shared_v4(row + (uint32_t((2 * p + 1) ^ (g & 7)) << 4), o1.x, o1.y, o1.z, o1.w);
                            }
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            if (rank == 0)
                                mbar_arrive(&st->full[q]);
                            else
                                mbar_arrive_cluster(mapa_shared(smem_u32(&st->full[q]), leader));
                            mbar_arrive(&st->rempty[r]);
                        }
                        if (++q == STAGES) {
                            q = 0;
                            qph ^= 1u;
                        }
                        if (++r == C_::RSTAGES) {
                            r = 0;
                            rph ^= 1u;
                        }
                    }
                }
            }
            __syncwarp();
        } else if (GC && warp >= 2) {
            // ------------------------------------------------------ converters
            // Conversion in global memory: warps 2, 3 and 12 .. 15 of every CTA.
            if constexpr (GC) {
                const int cw = warp < 4 ? warp - 2 : warp - C_::CONV_WARP0 + 2;
                convert_global<KIND>(args, int(blockIdx.x) * kConvWarps + cw, int(gridDim.x) * kConvWarps, lane,
                                     &st->abort);
            }
            __syncwarp();
        }
    } else {
        // The epilogue warpgroups raise their register budget (16-warp layout).
        if constexpr (WIDE) regs_inc<kRegsHigh>();
        // ------------------------------------------------------ epilogue
        const int ew = warp - EPI_WARP0;    // epilogue warp 0 .. 7
        const int q = warp & 3;             // tensor-memory lane quarter
        const int h = ew >> 2;              // column half of the tile
        // The unit whose 4-byte C goes out by TMA stores (this cluster's last, or
        // none), and this warp's four C staging blocks in the idle ring.
        const int tma_t = (EPI == EPI_F32 && args.c_tma && cluster < args.num_vunits)
                              ? cluster + (args.num_vunits - 1 - cluster) / nclusters * nclusters
                              : -1;
        const uint32_t stg = smem_u32(smem) + uint32_t(ew) * uint32_t(kStageWarp);
        bool stg_pending = false;           // TMA stores may still be reading the blocks
        const uint32_t t_lane = tmem_base + (uint32_t(32 * q) << 16) + uint32_t(h * HALF);
        // Accumulator buffers are released on the issuing (even) CTA's barriers.
        auto release = [&](int b) {
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                if constexpr (CTAS == 1)
                    mbar_arrive(&st->acc_empty[b]);
                else
                    mbar_arrive_cluster(mapa_shared(smem_u32(&st->acc_empty[b]), leader));
            }
        };
        int abuf = 0;
        uint32_t aph = 0;
        bool ok = true;
        // In-ring conversion of K blocks [kb0, kb1) (the producer's and the MMA
        // issuer's sequence of stages): each thread converts (128 + BN) / 64
        // 16-byte raw pieces (row g = i / 4, piece p = i % 4 of 64 bytes) into
        // the 16-byte chunks 2p and 2p + 1 of row g of the MMA stage, placed
        // by the 128-byte swizzle (chunk j of row g at j ^ (g & 7)); the raw
        // reads are contiguous and each quarter-warp's writes cover eight
        // distinct chunks of two rows, so neither conflicts.  The writes reach
        // the tensor cores through a proxy fence before the stage's barrier.
        // (WIDE: all pieces of a thread in flight at once; the narrow form,
        // one piece at a time, serves while the int32 sums occupy registers.)
        int cs = 0;
        uint32_t cph = 0;
        auto convert = [&](int kb0, int kb1, auto wide) -> bool {
            constexpr bool WIDE = decltype(wide)::value;
            const int ctid = int(threadIdx.x) - 32 * EPI_WARP0;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!warp_wait(&st->rfull[cs], cph, &st->abort, limit, lane)) return false;
                if (!warp_wait(&st->empty[cs], cph ^ 1u, &st->abort, limit, lane)) return false;
                // Every lane observes both completed phases before its accesses.
                mbar_try_wait(&st->rfull[cs], cph);
                mbar_try_wait(&st->empty[cs], cph ^ 1u);
                const uint32_t raw = smem_u32(raw_ring) + uint32_t(cs * C_::RAW_STAGE);
                const uint32_t dst_a = smem_u32(a_ring) + uint32_t(cs * C_::A_STAGE);
                const uint32_t dst_b = smem_u32(b_ring) + uint32_t(cs * C_::B_STAGE);
                auto piece = [&](int it) {
                    const int i = it * 256 + ctid;
                    const int g = i >> 2, p = i & 3;
                    const uint4 x = ld_shared_v4(raw + uint32_t(i) * 16u);
                    uint4 o0, o1;
                    if constexpr (KIND == Kind::F16)
                        cvt_s8_f16_x16(x, o0, o1);
                    else
                        cvt_s4_e4m3_x32(x, o0, o1);
                    // Pieces 0 .. 511 are A's 128 rows (it = 0, 1), the rest B's.
                    const uint32_t row = it < 2 ? dst_a + uint32_t(g) * 128u : dst_b + uint32_t(g - kBM) * 128u;
                    st_shared_v4(row + (uint32_t((2 * p) ^ (g & 7)) << 4), o0.x, o0.y, o0.z, o0.w);
                    st_shared_v4(row + (uint32_t((2 * p + 1) ^ (g & 7)) << 4), o1.x, o1.y, o1.z, o1.w);
                };
                if constexpr (WIDE) {
#pragma unroll
                    for (int it = 0; it < (kBM + BN) / 64; ++it) piece(it);
                } else {
#pragma unroll 1
                    for (int it = 0; it < (kBM + BN) / 64; ++it) piece(it);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&st->full[cs]);
                    mbar_arrive(&st->rempty[cs]);
                }
                if (++cs == STAGES) {
                    cs = 0;
                    cph ^= 1u;
                }
            }
            return true;
        };
        if (CTAS == 2 && PAIRS == 1 && args.split_reduce && cluster < args.num_vunits) {
            // This cluster's last unit is the first K half of a split tile: zero
            // the tile's C (each warp its 32 x 128 slice) before the K loops run,
            // for both halves to add into.
            const int last = cluster + (args.num_vunits - 1 - cluster) / nclusters * nclusters;
            const WorkRef lw = work_unit(last, args, C_::SUB);
            if (lw.part == 1) {
                const int zrow = lw.mb * (kBM * CTAS) + int(rank) * kBM + 32 * q + lane;
                const int zcol = lw.nb * BN + h * HALF;
                if (zrow < args.M) {
                    uint32_t z[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) z[j] = 0u;
                    uint32_t *crow = reinterpret_cast<uint32_t *>(args.C) + int64_t(zrow) * args.ldc;
#pragma unroll
                    for (int c = 0; c < NCH; ++c) {
                        const int cc = zcol + 32 * c;
                        if (cc < args.N) store_32(crow + cc, z, args.N - cc, args.c_wide);
                    }
                }
                __threadfence();
                __syncwarp();
                if (lane == 0) st_release_gpu(args.split_count + ((lw.slot * CTAS + int(rank)) * 4 + q) * 2 + h, 1u);
            }
        }
        for (int t = cluster; t < args.num_vunits && ok; t += nclusters) {
            WorkRef wr = work_unit(t, args, C_::SUB);
            if constexpr (KS > 1) ksplit_range(wr, krank, KS);
            const int row = wr.mb * (kBM * CTAS) + int(rank) * kBM + 32 * q + lane;
            const int col0 = (wr.nb * PAIRS + int(pp)) * BN + h * HALF;
            if constexpr (INT_OUT) {
                const int nchunks = (wr.kb1 - wr.kb0 + args.kb_per_chunk - 1) / args.kb_per_chunk;
                // In-ring conversion of chunk c (its K blocks) precedes the fold
                // of chunk c, and the fold of chunk c precedes the conversion of
                // chunk c + 2, whose MMAs reuse chunk c's accumulator buffer:
                // chunks 0 and 1 are converted first (while the int32 sums below
                // hold nothing), then chunk c + 2 after each fold c.
                auto convert_chunk = [&](int c, auto wide) {
                    const int c0 = wr.kb0 + c * args.kb_per_chunk;
                    return convert(c0, min(wr.kb1, c0 + args.kb_per_chunk), wide);
                };
                if constexpr (FU && !PFU) {
                    if ((nchunks > 0 && !convert_chunk(0, std::true_type{})) ||
                        (nchunks > 1 && !convert_chunk(1, std::true_type{}))) {
                        ok = false;
                        break;
                    }
                }
                int32_t acc[HALF];
#pragma unroll
                for (int j = 0; j < HALF; ++j) acc[j] = 0;
                for (int ch = 0; ch < nchunks; ++ch) {
                    if (!warp_wait(&st->acc_full[abuf], aph, &st->abort, limit, lane)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
#pragma unroll
                    for (int c = 0; c < HALF / 16; ++c) {
                        uint32_t r[16];
                        tmem_ld_16cols(t_lane + uint32_t(abuf * BN + 16 * c), r);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 16; ++j) acc[16 * c + j] += __float2int_rn(__uint_as_float(r[j]));
                    }
                    release(abuf);
                    if (++abuf == 2) {
                        abuf = 0;
                        aph ^= 1u;
                    }
                    if constexpr (FU && !PFU) {
                        if (ch + 2 < nchunks && !convert_chunk(ch + 2, std::false_type{})) {
                            ok = false;
                            break;
                        }
                    }
                }
                if (!ok) break;
                if constexpr (KS > 1) {
                    // K-split cluster: the partial sums wait in the ring for the
                    // cluster's completion pass.
#pragma unroll
                    for (int c = 0; c < NCH; ++c)
                        put_partial<BN * 4>(smem_u32(smem), 32 * q + lane, h * (HALF / 4) + 8 * c,
                                    reinterpret_cast<const uint32_t(&)[32]>(acc[32 * c]));
                    continue;
                }
                // A split tile of int32 C: both K halves add into the zeroed C
                // by int32 TMA reductions (modulo 2^32, like every partial sum).
                const bool add = CTAS == 2 && PAIRS == 1 && wr.part != 0 && args.split_reduce;
                if (add) {
                    const int slice = ((wr.slot * CTAS + int(rank)) * 4 + q) * 2 + h;
                    if (!split_zeroed_wait(args.split_count + slice, &st->abort, limit, lane)) {
                        ok = false;
                        break;
                    }
                } else if (BN == kBN && PAIRS == 1 && wr.part != 0) {
                    // Sum of the two K halves, wrapping like every int32 partial sum.
                    const int slice = ((wr.slot * CTAS + int(rank)) * 4 + q) * 2 + h;
                    uint32_t *cnt = args.split_count + slice;
                    bool finish = split_other_done(cnt, lane);
                    if (!finish) {
                        float4 *mine = split_partial(args, slice, wr.part - 1);
#pragma unroll
                        for (int i = 0; i < HALF / 4; ++i)
                            mine[i * 32 + lane] = make_float4(__int_as_float(acc[4 * i]), __int_as_float(acc[4 * i + 1]),
                                                              __int_as_float(acc[4 * i + 2]), __int_as_float(acc[4 * i + 3]));
                        finish = split_publish(cnt, lane);
                    }
                    if (!finish) continue;
                    const float4 *other = split_partial(args, slice, 2 - wr.part);
#pragma unroll
                    for (int i = 0; i < HALF / 4; ++i) {
                        const float4 o = __ldcg(other + i * 32 + lane);
                        acc[4 * i] = int32_t(uint32_t(acc[4 * i]) + uint32_t(__float_as_int(o.x)));
                        acc[4 * i + 1] = int32_t(uint32_t(acc[4 * i + 1]) + uint32_t(__float_as_int(o.y)));
                        acc[4 * i + 2] = int32_t(uint32_t(acc[4 * i + 2]) + uint32_t(__float_as_int(o.z)));
                        acc[4 * i + 3] = int32_t(uint32_t(acc[4 * i + 3]) + uint32_t(__float_as_int(o.w)));
                    }
                }
                const int row0 = row - lane;  // first row of this warp's 32
                // Integer routes: TMA stores in single-wave launches (every unit
                // is its cluster's last); a per-unit choice, as the FP32 path
                // makes, costs this register-bound epilogue spills.
                const bool use_tma = add || (args.c_tma && args.num_vunits <= nclusters);
                if (args.out_mode == OUT_S32 && use_tma) {
#pragma unroll
                    for (int c = 0; c < NCH; ++c) {
                        const int cc = col0 + 32 * c;
                        if (cc < args.N)
                            tma_store_block(&tmC, stg + uint32_t(c * kStageC),
                                            reinterpret_cast<const uint32_t(&)[32]>(acc[32 * c]), lane, cc, row0,
                                            stg_pending && c == 0, add);
                    }
                    stg_pending = true;
                } else if (args.out_mode == OUT_S32) {
                    if (row < args.M) {
                        int32_t *crow = reinterpret_cast<int32_t *>(args.C) + int64_t(row) * args.ldc;
#pragma unroll
                        for (int c = 0; c < NCH; ++c) {
                            const int cc = col0 + 32 * c;
                            if (cc < args.N)
                                store_32(crow + cc, reinterpret_cast<const uint32_t(&)[32]>(acc[32 * c]), args.N - cc,
                                         args.c_wide);
                        }
                    }
                } else {
                    const bool tma_f32 = use_tma && args.out_mode == OUT_F32;
                    store_scaled_row<HALF>(args, row, col0, acc, &tmC, tma_f32, stg, lane, row0, stg_pending);
                    stg_pending = stg_pending || tma_f32;
                }
            } else {
                if (!warp_wait(&st->acc_full[abuf], aph, &st->abort, limit, lane)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                // This cluster's last unit: its epilogue is not hidden behind a
                // next tile, and the ring is idle once the unit has been
                // multiplied, so 4-byte C goes out by TMA stores staged there.
                const bool use_tma = t == tma_t;
                if constexpr (KS > 1) {
                    // K-split cluster: the partial sums (FP16 accumulators widened
                    // exactly to FP32) wait in the ring for the completion pass.
#pragma unroll
                    for (int c = 0; c < NCH; ++c) {
                        uint32_t r[32];
                        tmem_ld_32cols(t_lane + uint32_t(abuf * BN + 32 * c), r);
                        tmem_ld_wait();
                        if constexpr (EPI == EPI_F16ACC) {
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                r[e] = __float_as_uint(__half2float(__ushort_as_half(static_cast<uint16_t>(r[e]))));
                        }
                        put_partial<BN * 4>(smem_u32(smem), 32 * q + lane, h * (HALF / 4) + 8 * c, r);
                    }
                } else {
                    // A split tile of FP32 C: both K halves add into the zeroed C
                    // by FP32 TMA reductions (0 + a + b: the same bits in either
                    // order).
                    const bool add = CTAS == 2 && PAIRS == 1 && EPI == EPI_F32 && wr.part != 0 && args.split_reduce;
                    if (add) {
                        const int slice = ((wr.slot * CTAS + int(rank)) * 4 + q) * 2 + h;
                        ok = split_zeroed_wait(args.split_count + slice, &st->abort, limit, lane);
                    }
                    if (EPI == EPI_F32 && ((wr.part == 0 && use_tma) || add)) {
                        if (ok) {
#pragma unroll
                            for (int c = 0; c < NCH; ++c) {
                                uint32_t r[32];
                                tmem_ld_32cols(t_lane + uint32_t(abuf * BN + 32 * c), r);
                                tmem_ld_wait();
                                const int cc = col0 + 32 * c;
                                if (cc < args.N)
                                    tma_store_block(&tmC, stg + uint32_t(c * kStageC), r, lane, cc, row - lane,
                                                    stg_pending && c == 0, add);
                            }
                            stg_pending = true;
                        }
                    } else if (wr.part == 0) {
                        float *crow = reinterpret_cast<float *>(args.C) + int64_t(row) * args.ldc;
#pragma unroll
                        for (int c = 0; c < NCH; ++c) {
                            uint32_t r[32];
                            tmem_ld_32cols(t_lane + uint32_t(abuf * BN + 32 * c), r);
                            tmem_ld_wait();
                            const int cc = col0 + 32 * c;
                            if constexpr (EPI == EPI_F16ACC) {
                                if (row < args.M && cc < args.N)
                                    store_f16acc_32(reinterpret_cast<uint16_t *>(args.C) + int64_t(row) * args.ldc + cc, r,
                                                    args.N - cc, args.c_wide);
                            } else {
                                if (row < args.M && cc < args.N) store_32(crow + cc, r, args.N - cc, args.c_wide);
                            }
                        }
                    } else if constexpr (BN == kBN) {
                        // (Only 256-wide tiles are split in halves of K.)
                        const int slice = ((wr.slot * CTAS + int(rank)) * 4 + q) * 2 + h;
                        void *crow = nullptr;
                        if (row < args.M)
                            crow = static_cast<uint8_t *>(args.C) +
                                   (int64_t(row) * args.ldc + col0) * (EPI == EPI_F16ACC ? 2 : 4);
                        split_epilogue<EPI>(t_lane + uint32_t(abuf * BN), args.split_count + slice,
                                            split_partial(args, slice, wr.part - 1), split_partial(args, slice, 2 - wr.part),
                                            crow, args.N - col0, args.c_wide, lane);
                    }
                }
                release(abuf);
                if (++abuf == 2) {
                    abuf = 0;
                    aph ^= 1u;
                }
            }
        }
        // Every TMA store of C has read its staging block before the CTA exits
        // (the writes themselves complete with the grid).
        if (stg_pending && lane == 0) bulk_wait_group_read0();
        __syncwarp();
    }

    if constexpr (KS > 1) {
        // Every CTA's partial sums are in its ring (barrier release / acquire at
        // cluster scope); each completes its rows of the tile from all of them.
        // Peers read this CTA's ring until the second barrier, on which the
        // completing threads arrive after their last loads and every other
        // thread here.
        cluster_sync();
        tc_fence_before_sync();
        if (warp >= EPI_WARP0 && warp < EPI_WARP0 + EPI_WARPS && cluster < args.num_vunits) {
            const WorkRef wr = work_unit(cluster, args, C_::SUB);
            ksplit_complete<EPI, KS, BN>(args, wr.mb, wr.nb, krank, smem_u32(smem), warp - EPI_WARP0, lane);
        } else {
            cluster_arrive();
        }
        cluster_wait();
        tc_fence_after_sync();
    } else {
        tc_fence_before_sync();
        if constexpr (CL == 1)
            __syncthreads();
        else
            cluster_sync();
        tc_fence_after_sync();
    }
    if (warp == 1) tmem_dealloc<CTAS>(tmem_base, TMEM_COLS);
    if (args.clock_probe != nullptr && threadIdx.x == 0) {
        const uint64_t c1 = sm_clock64(), t1 = globaltimer_ns();
        atomicAdd(args.clock_probe + 0, static_cast<unsigned long long>(c1 - st->probe_c0));
        atomicAdd(args.clock_probe + 1, static_cast<unsigned long long>(t1 - st->probe_t0));
        atomicAdd(args.clock_probe + 2, 1ull);
    }
}

template <typename T>
__global__ void zero_fill_kernel(T *C, int64_t ldc, int M, int N) {
    const int64_t total = int64_t(M) * N;
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
         i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t r = i / N, c = i - r * N;
        C[r * ldc + c] = T(0);
    }
}

// Zeroes the split-tile counters of the GEMM launched next on the stream.
// Launched programmatically like the GEMM kernels: it waits for the previous
// kernel of the stream (an earlier user of the pool block) before writing, and
// lets the GEMM start its setup at once; the GEMM's own wait then orders its
// first counter access after these stores.  (A memset between the two kernels
// would end the overlap: ~5 us between them at N = 4096, against ~0.7 us.)
__global__ void __launch_bounds__(256) clear_words_kernel(uint32_t *p, int n, uint32_t *p2, int n2) {
    griddep_wait();
    griddep_launch_dependents();
    for (int i = int(threadIdx.x); i < n; i += int(blockDim.x)) p[i] = 0u;
    for (int i = int(threadIdx.x); i < n2; i += int(blockDim.x)) p2[i] = 0u;
}

// Zeroes n words at p and n2 at p2 (either count may be 0).
cudaError_t launch_clear_words(uint32_t *p, int n, uint32_t *p2, int n2, bool pdl, cudaStream_t stream) {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    std::memset(&cfg, 0, sizeof(cfg));
    std::memset(attr, 0, sizeof(attr));
    cfg.gridDim = dim3(1, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    cfg.attrs = attr;
    if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 1;
    }
    cudaError_t e = cudaLaunchKernelEx(&cfg, clear_words_kernel, p, n, p2, n2);
    if (e == cudaSuccess) note_launches(1);
    return e;
}

// The work list's tile coordinates (tile_coords), on the host.
void host_tile_coords(int t, const GemmArgs &a, int &mb, int &nb) {
    const int per_group = a.group_m * a.tiles_n;
    const int g = t / per_group;
    const int first_m = g * a.group_m;
    const int gsz = a.tiles_m - first_m < a.group_m ? a.tiles_m - first_m : a.group_m;
    const int r = t - g * per_group;
    mb = first_m + r % gsz;
    nb = r / gsz;
}

struct LaunchCache {
    int dev = -1;
    int max_clusters = 0;
};

struct LastLaunch {
    int grid = 0, cluster = 0, ksplit = 0, bn = 0;
};
thread_local LastLaunch g_last;

// Launch shape of one variant: dynamic shared memory, cluster dimension and
// (optionally) programmatic stream serialization.
template <Kind KIND, bool B_MN, int EPI, int CTAS, int SUBK, int KS, int BN, bool FU = false, int PAIRS = 1,
          bool GC = false>
void launch_config(cudaLaunchConfig_t &cfg, cudaLaunchAttribute (&attr)[2], bool pdl, cudaStream_t stream) {
    std::memset(&cfg, 0, sizeof(cfg));
    std::memset(attr, 0, sizeof(attr));
    cfg.blockDim = dim3(Cfg<CTAS, SUBK, BN, FU, GC>::THREADS_, 1, 1);
    cfg.dynamicSmemBytes = smem_bytes<CTAS, SUBK, BN, FU>();
    cfg.stream = stream;
    cfg.attrs = attr;
    int n = 0;
    if constexpr (CTAS * KS * PAIRS > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = CTAS * KS * PAIRS;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.numAttrs = n;
}

// Clusters of the variant that can be resident at once on the current device
// (cached per device; the shared-memory opt-in is set on first use).
template <Kind KIND, bool B_MN, int EPI, int CTAS, int SUBK, int KS, int BN, bool FU = false, int PAIRS = 1,
          bool GC = false>
cudaError_t cluster_capacity(int sms, int *out) {
    auto *fn = gemm_kernel<KIND, B_MN, EPI, CTAS, SUBK, KS, BN, FU, PAIRS, GC>;
    constexpr int CL = CTAS * KS * PAIRS;
    static thread_local LaunchCache cache;  // per device (re-queried when it changes)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev != cache.dev) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem_bytes<CTAS, SUBK, BN, FU>()));
        if (e != cudaSuccess) return e;
        int clusters = sms / CL;
        if constexpr (CL > 1) {
            cudaLaunchConfig_t cfg;
            cudaLaunchAttribute attr[2];
            launch_config<KIND, B_MN, EPI, CTAS, SUBK, KS, BN, FU, PAIRS, GC>(cfg, attr, false, nullptr);
            cfg.gridDim = dim3(CL * (sms / CL), 1, 1);
            int n = 0;
            e = cudaOccupancyMaxActiveClusters(&n, fn, &cfg);
            if (e != cudaSuccess) return e;
            if (n <= 0) return cudaErrorInvalidConfiguration;
            if (n < clusters) clusters = n;
        }
        cache.max_clusters = clusters;
        cache.dev = dev;
    }
    *out = cache.max_clusters;
    return cudaSuccess;
}

// Device address of g_clock_probe on the current device (cached per device
// and thread).
cudaError_t clock_probe_base(unsigned long long **out) {
    static thread_local int dev_cached = -1;
    static thread_local unsigned long long *addr = nullptr;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev != dev_cached) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_clock_probe);
        if (e != cudaSuccess) return e;
        addr = static_cast<unsigned long long *>(p);
        dev_cached = dev;
    }
    *out = addr;
    return cudaSuccess;
}

template <Kind KIND, bool B_MN, int EPI, int CTAS, int SUBK, int KS, int BN, bool FU = false, int PAIRS = 1,
          bool GC = false>
cudaError_t launch_one(const CUtensorMap &ta, const CUtensorMap &tb, const GemmArgs &args_in,
                       int sms, cudaMemPool_t pool, cudaStream_t stream) {
    auto *fn = gemm_kernel<KIND, B_MN, EPI, CTAS, SUBK, KS, BN, FU, PAIRS, GC>;
    int maxc = 0;
    cudaError_t e = cluster_capacity<KIND, B_MN, EPI, CTAS, SUBK, KS, BN, FU, PAIRS, GC>(sms, &maxc);
    if (e != cudaSuccess) return e;
    GemmArgs args = args_in;
    if constexpr (PAIRS == 2) {
        // Work units of two pairs: tile columns 2 nb and 2 nb + 1 of tile row mb
        // (the second is empty past N when the columns are odd).
        args.tiles_n = (args.tiles_n + 1) / 2;
        args.num_tiles = args.tiles_m * args.tiles_n;
    }
    if (KS > 1 && args.num_tiles > maxc) return cudaErrorInvalidConfiguration;  // one wave of clusters
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    launch_config<KIND, B_MN, EPI, CTAS, SUBK, KS, BN, FU, PAIRS, GC>(cfg, attr, args.pdl != 0, stream);
    // Work list: split the last wave's tiles in K when they fill at most half
    // of the clusters (a lone partial wave included).  The halves exchange
    // partial sums through a stream-ordered workspace from `pool`: a counter
    // per epilogue warp slice (zeroed here) and two slices of partial sums.
    GemmArgs a = args;
    a.clock_probe = nullptr;
    if (a.probe) {
        unsigned long long *base = nullptr;
        e = clock_probe_base(&base);
        if (e != cudaSuccess) return e;
        const int family = KIND == Kind::E4M3 ? 2 : EPI == EPI_INT ? 1 : 0;
        a.clock_probe = base + 3 * family;
    }
    // 32-byte C stores (whole L2 sectors) when C's base and row pitch allow them.
    const int64_t esize = (EPI == EPI_F16ACC || (EPI == EPI_INT && (a.out_mode == OUT_BF16 || a.out_mode == OUT_F16))) ? 2 : 4;
    a.c_wide = (reinterpret_cast<uintptr_t>(a.C) % 32 == 0 && (a.ldc * esize) % 32 == 0) ? 1 : 0;
    // 4-byte C (FP32, int32, scaled FP32) is written by TMA stores of 32 x 32
    // blocks staged in shared memory; 16-bit C by 16/32-byte stores per lane.
    CUtensorMap tc;
    std::memset(&tc, 0, sizeof(tc));
    a.c_tma = 0;
    const bool tma_c = esize == 4;
    const bool int_c = EPI == EPI_INT && a.out_mode == OUT_S32;
    // (A K-split cluster writes C from its completion pass, without TMA.)
    if (KS == 1 && tma_c && encode_tmap_c32(&tc, a.C, uint64_t(a.N), uint64_t(a.M), uint64_t(a.ldc), !int_c) == 0)
        a.c_tma = 1;
    // Split pair tiles of FP32 or int32 C add their halves into C by TMA
    // reductions (one-CTA tiles, split only when forced, exchange partials).
    const bool reduce = CTAS == 2 && a.split_reduce && a.c_tma && (EPI == EPI_F32 || int_c);
    a.split_reduce = 0;
    const int tail = a.num_tiles < maxc ? a.num_tiles : a.num_tiles % maxc;
    a.tail_split = 0;
    a.split_count = nullptr;
    a.split_part = nullptr;
    void *ws = nullptr;
    int split_words = 0;  // split-tile counters to zero before the launch
    // The split saves about half of a tile's K loop (~0.35 us per K block
    // under the power cap).  Adding the halves into C by TMA reductions costs
    // ~4 us after the last MMA; exchanging partial sums through the workspace
    // ~8-12 us (128 KiB in and out of each SM at its L2 write rate).  Measured
    // (interleaved A/B): with reductions the split gains from 64 K blocks for
    // the FP16 kind (FP16, INT8: N = 4096 -1% / -3.5%, N = 8192 -1.5% /
    // -2.2%) but loses at 64 blocks of the E4M3 kind (INT4, N = 8192: +1.2%);
    // with the exchange it loses at 64 blocks (FP16 N = 4096: +7%).  So the
    // threshold is split_min_kb K blocks (64 by default) with reductions on
    // the FP16 kind, twice that on the E4M3 kind or with the exchange.
    const int min_kb = a.split_min_kb * (reduce ? 1 : 2) * (KIND == Kind::E4M3 ? 2 : 1);
    if (!FU && PAIRS == 1 && KS == 1 && BN == kBN && pool != nullptr && a.split_ok && a.num_kb > SUBK &&
        a.num_kb >= min_kb &&
        tail > 0 && 2 * tail <= maxc) {
        const size_t slices = size_t(tail) * CTAS * EPI_WARPS;
        const size_t count_bytes = (slices * sizeof(uint32_t) + 255) / 256 * 256;
        const size_t bytes = count_bytes + (reduce ? 0 : slices * 2 * kSliceWords * sizeof(float));
        if (cudaMallocFromPoolAsync(&ws, bytes, pool, stream) == cudaSuccess) {
            split_words = int(count_bytes / sizeof(uint32_t));
            a.tail_split = tail;
            a.split_reduce = reduce ? 1 : 0;
            a.split_count = static_cast<uint32_t *>(ws);
            a.split_part = reduce ? nullptr : reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + count_bytes);
        } else {
            cudaGetLastError();  // no workspace: run the tail whole
            ws = nullptr;
        }
    }
    a.num_vunits = a.num_tiles + a.tail_split;
    // Conversion in global memory: every resident cluster is launched (CTAs
    // without a tile convert too), and the panels the first wave's tiles use
    // are converted first.
    const int clusters = GC ? maxc : (a.num_vunits < maxc ? a.num_vunits : maxc);
    int conv_words = 0;
    if constexpr (GC) {
        int max_mb = 0, max_nb = 0;
        const int wave = a.num_tiles < clusters ? a.num_tiles : clusters;
        for (int t = 0; t < wave; ++t) {
            int mb, nb;
            host_tile_coords(t, a, mb, nb);
            max_mb = mb > max_mb ? mb : max_mb;
            max_nb = nb > max_nb ? nb : max_nb;
        }
        const int pa = (a.M + kConvPanel - 1) / kConvPanel, pb = (a.N + kConvPanel - 1) / kConvPanel;
        a.conv_front_a = (max_mb + 1) * CTAS < pa ? (max_mb + 1) * CTAS : pa;
        a.conv_front_b = (max_nb + 1) * (BN / kConvPanel) < pb ? (max_nb + 1) * (BN / kConvPanel) : pb;
        conv_words = int(conv_counter_words(a.M, a.N, a.K));
    }
    if (split_words > 0 || conv_words > 0) {
        e = launch_clear_words(a.conv_count, conv_words, a.split_count, split_words, a.pdl != 0, stream);
        if (e != cudaSuccess) {
            if (ws != nullptr) cudaFreeAsync(ws, stream);
            return e;
        }
    }
    // Each cluster's last unit writes 4-byte C by TMA stores (or reductions)
    // staged in the idle ring (its epilogue is exposed); earlier units use
    // 32-byte stores, which leave the TMA engine to the operand loads while the
    // next tile runs.
    cfg.gridDim = dim3(CTAS * KS * PAIRS * clusters, 1, 1);
    e = cudaLaunchKernelEx(&cfg, fn, ta, tb, tc, a);
    if (e == cudaSuccess) {
        g_last.grid = CTAS * KS * PAIRS * clusters;
        g_last.cluster = CTAS * KS * PAIRS;
        g_last.ksplit = KS;
        g_last.bn = BN;
    }
    if (ws != nullptr) cudaFreeAsync(ws, stream);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Clusters of KS one-CTA tiles that fit one wave (the same for every variant:
// one 320-thread CTA with ~197 KB of shared memory per SM); 0 when that
// cluster shape cannot run.
int ksplit_capacity(int ks, int sms) {
    int cap = 0;
    cudaError_t e = cudaSuccess;
    if (ks == 8) e = cluster_capacity<Kind::F16, true, EPI_F32, 1, 1, 8, kBN>(sms, &cap);
    if (ks == 4) e = cluster_capacity<Kind::F16, true, EPI_F32, 1, 1, 4, kBN>(sms, &cap);
    if (ks == 2) e = cluster_capacity<Kind::F16, true, EPI_F32, 1, 1, 2, kBN>(sms, &cap);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return cap;
}

}  // namespace

ClusterCaps cluster_caps(int sms) {
    ClusterCaps c;
    c.c2 = ksplit_capacity(2, sms);
    c.c4 = ksplit_capacity(4, sms);
    c.c8 = ksplit_capacity(8, sms);
    return c;
}

void last_launch(int *grid, int *cluster, int *ksplit, int *tile_n) {
    *grid = g_last.grid;
    *cluster = g_last.cluster;
    *ksplit = g_last.ksplit;
    *tile_n = g_last.bn;
}

int pick_ksplit(int tiles, int num_kb, int knob, int sms) {
    if (knob == 1 || 2 * tiles > sms) return 1;
    return pick_ksplit_pure(tiles, num_kb, knob, sms, cluster_caps(sms));
}

int64_t conv_counter_words(int64_t M, int64_t N, int64_t K) {
    const int64_t slices = (K + kConvSlice - 1) / kConvSlice;
    return ((M + kConvPanel - 1) / kConvPanel + (N + kConvPanel - 1) / kConvPanel) * slices + 1;
}

size_t gemm_smem_bytes(int ctas) { return ctas == 2 ? smem_bytes<2, 2>() : smem_bytes<1, 1>(); }

// One-CTA launches of 256-wide tiles run as K-split clusters when pick_ksplit
// says so; args.bn = 64 / 128 selects the narrow one-CTA tiles.
cudaError_t launch_gemm(Kind kind, bool b_mn_major, int epi, int ctas, const CUtensorMap &ta,
                        const CUtensorMap &tb, const GemmArgs &args, int sms, cudaMemPool_t pool,
                        cudaStream_t stream) {
    const int bn = (ctas == 1 && args.bn != 0) ? args.bn : kBN;
    if (bn != kBN && bn != 64 && bn != 128) return cudaErrorInvalidValue;
    int ks = 1;
    if (ctas == 1 && bn == kBN) {
        ks = pick_ksplit(args.num_tiles, args.num_kb, args.ksplit, sms);
    } else if (ctas == 1 && (args.ksplit == 2 || args.ksplit == 4) && args.num_kb >= args.ksplit &&
               args.num_tiles <= ksplit_capacity(args.ksplit, sms)) {
        ks = args.ksplit;  // narrow tiles: the size (2 or 4) the caller chose
    }
#define PTC_LAUNCH(K, BMN, E)                                                                       \
    do {                                                                                            \
        if (bn == 64 && ks == 4) return launch_one<K, BMN, E, 1, 1, 4, 64>(ta, tb, args, sms, pool, stream); \
        if (bn == 64 && ks == 2) return launch_one<K, BMN, E, 1, 1, 2, 64>(ta, tb, args, sms, pool, stream); \
        if (bn == 128 && ks == 4) return launch_one<K, BMN, E, 1, 1, 4, 128>(ta, tb, args, sms, pool, stream); \
        if (bn == 128 && ks == 2) return launch_one<K, BMN, E, 1, 1, 2, 128>(ta, tb, args, sms, pool, stream); \
        if (bn == 64) return launch_one<K, BMN, E, 1, 1, 1, 64>(ta, tb, args, sms, pool, stream);   \
        if (bn == 128) return launch_one<K, BMN, E, 1, 1, 1, 128>(ta, tb, args, sms, pool, stream); \
        if (ks == 8) return launch_one<K, BMN, E, 1, 1, 8, kBN>(ta, tb, args, sms, pool, stream);   \
        if (ks == 4) return launch_one<K, BMN, E, 1, 1, 4, kBN>(ta, tb, args, sms, pool, stream);   \
        if (ks == 2) return launch_one<K, BMN, E, 1, 1, 2, kBN>(ta, tb, args, sms, pool, stream);   \
        return ctas == 1 ? launch_one<K, BMN, E, 1, 1, 1, kBN>(ta, tb, args, sms, pool, stream)     \
               : args.pairs == 2  ? launch_one<K, BMN, E, 2, 2, 1, kBN, false, 2>(ta, tb, args, sms, pool, stream) \
               : args.stage_kb == 1 ? launch_one<K, BMN, E, 2, 1, 1, kBN>(ta, tb, args, sms, pool, stream) \
                                    : launch_one<K, BMN, E, 2, 2, 1, kBN>(ta, tb, args, sms, pool, stream); \
    } while (0)
#define PTC_LAUNCH_FU(K)                                                                                \
    do {                                                                                                \
        if (ctas == 2) return launch_one<K, false, EPI_INT, 2, 1, 1, kBN, true>(ta, tb, args, sms, pool, stream); \
        if (bn == 64 && ks == 4) return launch_one<K, false, EPI_INT, 1, 1, 4, 64, true>(ta, tb, args, sms, pool, stream); \
        if (bn == 64 && ks == 2) return launch_one<K, false, EPI_INT, 1, 1, 2, 64, true>(ta, tb, args, sms, pool, stream); \
        if (bn == 128 && ks == 4) return launch_one<K, false, EPI_INT, 1, 1, 4, 128, true>(ta, tb, args, sms, pool, stream); \
        if (bn == 128 && ks == 2) return launch_one<K, false, EPI_INT, 1, 1, 2, 128, true>(ta, tb, args, sms, pool, stream); \
        if (bn == 64) return launch_one<K, false, EPI_INT, 1, 1, 1, 64, true>(ta, tb, args, sms, pool, stream);   \
        if (bn == 128) return launch_one<K, false, EPI_INT, 1, 1, 1, 128, true>(ta, tb, args, sms, pool, stream); \
        if (ks == 8) return launch_one<K, false, EPI_INT, 1, 1, 8, kBN, true>(ta, tb, args, sms, pool, stream);   \
        if (ks == 4) return launch_one<K, false, EPI_INT, 1, 1, 4, kBN, true>(ta, tb, args, sms, pool, stream);   \
        if (ks == 2) return launch_one<K, false, EPI_INT, 1, 1, 2, kBN, true>(ta, tb, args, sms, pool, stream);   \
        return launch_one<K, false, EPI_INT, 1, 1, 1, kBN, true>(ta, tb, args, sms, pool, stream);                \
    } while (0)
    if (kind == Kind::F16 && b_mn_major && epi == EPI_F32) PTC_LAUNCH(Kind::F16, true, EPI_F32);
    if (kind == Kind::F16 && b_mn_major && epi == EPI_F16ACC) PTC_LAUNCH(Kind::F16, true, EPI_F16ACC);
    if (args.conv != 0) {
        // Conversion in the GEMM kernel's converter warps: integer launches with
        // K-major B, 256-wide tiles, no K split (one CTA, or CTA pairs).
        if (b_mn_major || epi != EPI_INT || bn != kBN || args.pairs != 1) return cudaErrorInvalidValue;
        if (kind == Kind::F16)
            return ctas == 1 ? launch_one<Kind::F16, false, EPI_INT, 1, 1, 1, kBN, false, 1, true>(ta, tb, args, sms, pool, stream)
                             : launch_one<Kind::F16, false, EPI_INT, 2, 2, 1, kBN, false, 1, true>(ta, tb, args, sms, pool, stream);
        if (kind == Kind::E4M3)
            return ctas == 1 ? launch_one<Kind::E4M3, false, EPI_INT, 1, 1, 1, kBN, false, 1, true>(ta, tb, args, sms, pool, stream)
                             : launch_one<Kind::E4M3, false, EPI_INT, 2, 2, 1, kBN, false, 1, true>(ta, tb, args, sms, pool, stream);
        return cudaErrorInvalidValue;
    }
    if (args.in_ring != 0) {
        // In-ring conversion: integer launches with K-major B (one CTA per
        // tile, or CTA pairs with dedicated converter warps).
        if (b_mn_major || epi != EPI_INT) return cudaErrorInvalidValue;
        if (kind == Kind::F16) PTC_LAUNCH_FU(Kind::F16);
        if (kind == Kind::E4M3) PTC_LAUNCH_FU(Kind::E4M3);
        return cudaErrorInvalidValue;
    }
    if (kind == Kind::F16 && !b_mn_major && epi == EPI_INT) PTC_LAUNCH(Kind::F16, false, EPI_INT);
    if (kind == Kind::F16 && b_mn_major && epi == EPI_INT) PTC_LAUNCH(Kind::F16, true, EPI_INT);
    if (kind == Kind::E4M3 && !b_mn_major && epi == EPI_INT) PTC_LAUNCH(Kind::E4M3, false, EPI_INT);
#undef PTC_LAUNCH
#undef PTC_LAUNCH_FU
    return cudaErrorInvalidValue;
}

cudaError_t launch_zero_fill(void *C, int64_t ldc, int M, int N, int esize, int grid, cudaStream_t stream) {
    if (esize == 2)
        zero_fill_kernel<uint16_t><<<grid, 256, 0, stream>>>(static_cast<uint16_t *>(C), ldc, M, N);
    else
        zero_fill_kernel<uint32_t><<<grid, 256, 0, stream>>>(static_cast<uint32_t *>(C), ldc, M, N);
    return cudaGetLastError();
}

cudaError_t read_and_clear_clock_probe(unsigned long long out[9]) {
    unsigned long long v[3][3];
    cudaError_t e = cudaMemcpyFromSymbol(v, g_clock_probe, sizeof(v));
    if (e != cudaSuccess) return e;
    const unsigned long long zero[3][3] = {};
    e = cudaMemcpyToSymbol(g_clock_probe, zero, sizeof(zero));
    std::memcpy(out, v, sizeof(v));
    return e;
}

cudaError_t read_and_clear_error_word(uint32_t *out) {
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_error_word, sizeof(v));
    if (e != cudaSuccess) return e;
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero));
    *out = v;
    return e;
}

}  // namespace ptc
