// api.cu -- the C ABI of libptc (declared in include/ptc.h): argument checks,
// tensor maps, workspace, launches.  Host code only.
//
// Each call validates its arguments without touching CUDA, checks the device
// (compute capability 10.3), encodes TMA tensor maps for the operands, and
// launches on the caller's stream:
//   gemm_f16: one persistent tensor-core kernel (FP16 x FP16 -> FP32).
//   gemm_s8 : s8 -> f16 conversion of A and B into a stream-ordered workspace,
//             then the tensor-core kernel with exact chunked int32 folding.
//   gemm_s4 : packed s4 -> E4M3 conversion, then the same with E4M3 MMAs.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "ptc.h"

namespace {

using ptc::GemmArgs;
using ptc::Kind;

constexpr int64_t kMaxDim = int64_t(1) << 30;
constexpr uint64_t kDefaultWaitNs = 1000000000ull;  // 1 s per pipeline wait
constexpr int kMaxDevices = 64;

std::atomic<uint64_t> g_launches{0};
thread_local char g_msg[512];

// Tunables (process-wide).  Integer routes fold the FP32 partial sums into
// int32 every kb_per_chunk K blocks of 128 bytes; see gemm_tc.cu.
std::atomic<int> g_chunk_s8{16};  // 1024 K values: |partial| <= 1024 * 2^14 = 2^24
std::atomic<int> g_chunk_s4{64};  // 8192 K values: |partial| <= 8192 * 2^6  = 2^19
constexpr int kMaxChunkS8 = 16;   // 2^24 / (64 * 2^14): the longest exact INT8 fold
constexpr int kMaxChunkS4 = 2048; // 2^24 / (128 * 2^6): the longest exact INT4 fold
std::atomic<int> g_group_m{8};
std::atomic<int> g_l2_hint{0};
std::atomic<int> g_cta_pair{0};     // 0: by problem size, 1: one CTA per tile, 2: CTA pairs
std::atomic<int> g_tail_split{1};   // 1: split a short last wave in K
std::atomic<int> g_split_min_kb{64};
std::atomic<int> g_pair_stage_kb{2};  // CTA pairs: K blocks per ring stage
std::atomic<int> g_ksplit{0};         // K-split clusters: 0 by size, 1 never, 2 / 4 / 8 that size
std::atomic<int> g_tile_n{0};         // one-CTA tile width: 0 by size, 64 / 128 / 256 that width
std::atomic<int> g_split_reduce{1};   // split tiles of FP32 / int32 C: halves added by TMA reductions
std::atomic<int> g_pdl{1};            // programmatic stream serialization of the library's kernels
std::atomic<int> g_in_ring{1};        // integer routes: operands converted in the GEMM kernel's shared
                                      // memory where estimated faster (0: never, 2: on every one-CTA shape)
thread_local int g_last_conv = 0;     // operand conversion of this thread's last GEMM call
std::atomic<int> g_clock_probe{0};   // 1: GEMM kernels add to the clock record
std::atomic<int> g_multicast{0};     // 1: CTA-pair products run two pairs per cluster sharing A
std::atomic<int> g_conv_fused{0};    // 1: integer routes convert in the GEMM kernel's converter warps
std::atomic<int> g_pair_in_ring{0};  // integer routes on CTA pairs: 0 a separate conversion pass,
                                     // 2 conversion inside the pair kernel (dedicated converter warps)
std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};
std::atomic<int64_t> g_stall_tile{-1};

int fail_cuda(cudaError_t e, const char *what) {
    std::snprintf(g_msg, sizeof(g_msg), "CUDA call failed: %s: %s", what, cudaGetErrorString(e));
    cudaGetLastError();  // clear a sticky-free error so the next call starts clean
    return PTC_ERR_LAUNCH;
}

// ------------------------------------------------------------ device info
struct DevInfo {
    std::once_flag once;
    int ok = 0;      // 1: compute capability 10.3
    int sms = 0;
    cudaMemPool_t pool = nullptr;
    int pool_ok = 0;
};
DevInfo g_dev[kMaxDevices];

int current_device(int *dev_out, DevInfo **info_out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        std::snprintf(g_msg, sizeof(g_msg), "no usable current CUDA device");
        return PTC_ERR_DEVICE;
    }
    DevInfo &d = g_dev[dev];
    std::call_once(d.once, [&] {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return;
        }
        d.sms = sms;
        d.ok = (major == 10 && minor == 3 && sms > 0) ? 1 : 0;
        if (!d.ok) return;
        cudaMemPoolProps props;
        std::memset(&props, 0, sizeof(props));
        props.allocType = cudaMemAllocationTypePinned;
        props.handleTypes = cudaMemHandleTypeNone;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        if (cudaMemPoolCreate(&d.pool, &props) == cudaSuccess) {
            uint64_t keep = UINT64_MAX;  // keep freed workspace cached in the pool
            cudaMemPoolSetAttribute(d.pool, cudaMemPoolAttrReleaseThreshold, &keep);
            d.pool_ok = 1;
        } else {
            cudaGetLastError();
        }
    });
    if (!d.ok) {
        std::snprintf(g_msg, sizeof(g_msg), "device %d is not a compute capability 10.3 GPU", dev);
        return PTC_ERR_DEVICE;
    }
    *dev_out = dev;
    *info_out = &d;
    return PTC_OK;
}

// ------------------------------------------------------------ tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// 2-D row-major view: `inner` contiguous elements per row, `outer` rows,
// `pitch` bytes between rows; boxes of box_inner x box_outer elements with the
// 128-byte swizzle (or `swizzle`); out-of-range elements of a box read as zero.
int make_tmap(CUtensorMap *map, CUtensorMapDataType dt, const void *base, uint64_t inner,
              uint64_t outer, uint64_t pitch, uint32_t box_inner, uint32_t box_outer,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) {
        std::snprintf(g_msg, sizeof(g_msg), "cuTensorMapEncodeTiled unavailable");
        return PTC_ERR_LAUNCH;
    }
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {pitch};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        std::snprintf(g_msg, sizeof(g_msg), "cuTensorMapEncodeTiled failed (CUresult %d)", int(r));
        return PTC_ERR_LAUNCH;
    }
    return PTC_OK;
}

// ------------------------------------------------------------ validation
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void *a, uint64_t alen, const void *b, uint64_t blen) {
    const unsigned __int128 a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + blen && b0 < a0 + alen;
}

// Leading dimensions above 2^36 elements (256 GiB rows of 4-byte values, more
// than a GB300 holds) are rejected, as are sizes above 2^30.
constexpr int64_t kMaxLd = int64_t(1) << 36;

int check_ld(int64_t lda, int64_t ldb, int64_t ldc) {
    if (lda > kMaxLd || ldb > kMaxLd || ldc > kMaxLd) {
        std::snprintf(g_msg, sizeof(g_msg), "leading dimensions must be <= 2^36 elements");
        return PTC_ERR_INVALID;
    }
    return PTC_OK;
}

// Bytes spanned by `rows` rows of `cols` elements at `ld` elements pitch, for
// an element of `num`/`den` bytes (den = 2 for nibbles).  Sizes are at most
// 2^30 and pitches at most kMaxLd, so the product fits 128-bit arithmetic;
// the result saturates at 2^64 - 1.
uint64_t span_bytes(int64_t rows, int64_t cols, int64_t ld, int num, int den) {
    const __int128 elems = __int128(rows - 1) * ld + cols;
    const __int128 b = (elems * num + den - 1) / den;
    return b > __int128(UINT64_MAX) ? UINT64_MAX : uint64_t(b);
}

int check_sizes(int64_t M, int64_t N, int64_t K) {
    if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) {
        std::snprintf(g_msg, sizeof(g_msg), "sizes must satisfy 0 <= M, N, K <= 2^30");
        return PTC_ERR_INVALID;
    }
    const int64_t tiles = ((M + ptc::kBM - 1) / ptc::kBM) * ((N + ptc::kBN - 1) / ptc::kBN);
    if (tiles >= (int64_t(1) << 31)) {
        std::snprintf(g_msg, sizeof(g_msg), "too many output tiles");
        return PTC_ERR_INVALID;
    }
    return PTC_OK;
}

int fail(int code, const char *text) {
    std::snprintf(g_msg, sizeof(g_msg), "%s", text);
    return code;
}

// ------------------------------------------------------------ launches
// Launch shape: CTAs per output tile (1, or a pair on 256 x 256 tiles), the
// tile width of one-CTA tiles (256, 128 or 64 columns of 128 rows), and the
// K-split knob passed to the kernel launcher (1: no split; 2 / 4 / 8 that
// cluster size; 0 its size rule).
struct Shape {
    int ctas, bn, ks;
    bool ring = false;  // integer routes: operands converted inside the GEMM kernel
};

// Estimated SM clocks of one CTA's work in a single-wave launch, the quantity
// the automatic shape choice minimises (constants measured on GB300 with
// global-timer stamps per CTA, and fitted to the measured times of every
// shape at N = 512 .. 1536).  Per 128-byte K block: issuing its MMAs (~600
// clocks for 128 rows whatever the tile width: four K-steps, and the block's
// barrier round trip) or copying its operands (16 KiB of A plus bn rows of B
// at ~128 bytes per clock), whichever is longer; then the C tile leaving the
// SM (measured ~21
// bytes per clock end to end; the per-SM write path to L2 peaks at ~32),
// which is what makes 256-wide tiles slow when few SMs share a small
// product.  A K-split cluster instead writes its partial sums to shared
// memory, passes two cluster barriers and moves the partials and C between
// SMs: ~45 clocks per tile column.
int64_t est_clocks(int64_t num_kb, int bn, int ks, int esize) {
    const int64_t per_block = std::max<int64_t>(600, 128 + bn);
    const int64_t k_loop = (num_kb + ks - 1) / ks * per_block;
    return k_loop + (ks > 1 ? int64_t(45) * bn : int64_t(6) * bn * esize);
}

int64_t tile_count(int64_t M, int64_t N, int rows, int cols) {
    return ((M + rows - 1) / rows) * ((N + cols - 1) / cols);
}

// Operand conversion of the integer routes (conv 1: s8 -> binary16, 2: packed
// s4 -> E4M3), in the same SM clocks, fitted to the launch-shape sweep of
// both paths at N = 512 .. 2048 (CUDA-graph replays; the fit orders the two
// paths correctly for 70 of 72 single-wave shapes).  A separate pass costs
// ~2.7 us (its launch, its ramp, the GEMM's wait for it) plus its traffic
// (64 bytes read and 128 written per row and K block) at ~12 bytes per clock
// from L2.  In-ring conversion costs ~1.35 us before the first MMA plus, per
// K block of a CTA, what the eight converting warps add to the K loop (two
// per scheduler, latency-bound: ncu counts ~2400 instructions per K block of
// a 256-wide tile issued in 36% of the cycles): ~0.14 / 0.23 / 0.32 us for s8
// on 64 / 128 / 256-wide tiles, ~2.7 times that for s4, whose lookup takes
// more instructions per byte.  In ring only in single-wave launches.
int64_t pass_clocks(int64_t M, int64_t N, int64_t num_kb) { return 5100 + (M + N) * num_kb * 192 / 6300; }

int64_t ring_clocks(int64_t num_kb, int bn, int ks, int conv) {
    static const int64_t per_kb[2][3] = {{270, 440, 610}, {720, 1240, 1630}};
    const int w = bn == 64 ? 0 : bn == 128 ? 1 : 2;
    return 2560 + (num_kb + ks - 1) / ks * per_kb[conv == 2 ? 1 : 0][w];
}

}  // namespace

namespace ptc {
int pick_ksplit_pure(int tiles, int num_kb, int knob, int sms, const ClusterCaps &caps) {
    if (knob == 1 || 2 * tiles > sms) return 1;
    for (int ks = 8; ks >= 2; ks /= 2) {
        if ((knob != 0 && knob != ks) || num_kb < ks) continue;
        // The split costs ~1-1.5 us per call (partial sums to shared memory,
        // two cluster barriers, the reduction); a one-CTA K block takes
        // ~0.15 us, so by size it is taken when each CTA sheds 8 or more.
        const int shed = num_kb - (num_kb + ks - 1) / ks;
        if (knob == 0 && shed < 8) continue;
        if (tiles <= caps.of(ks)) return ks;
    }
    return 1;
}
}  // namespace ptc

namespace {

// Multi-wave products run on CTA pairs (256 x 256 tiles: a third fewer
// operand bytes per output).  A product whose 128 x 256 tiles fit one wave
// takes the shape of least estimated time among: narrow one-CTA tiles
// (128 x 128, 128 x 64) that still fit one wave, whole or in K-split
// clusters of 2 or 4; K-split clusters of 128 x 256 tiles (pick_ksplit_pure);
// and whole 128 x 256 tiles, which go to pairs for FP16 from 32 one-CTA tiles
// up (measured 4-10% faster at N = 1024 .. 2048 before narrow tiles existed;
// the integer routes were faster with one CTA per tile).  esize: bytes per C
// element; fpair / ftile / fks: the knobs cta_pair, tile_n and ksplit, which
// force parts of the choice; caps: the device's K-split cluster capacities.
// conv (integer routes that may convert in the ring: 1 s8, 2 packed s4; 0
// otherwise) adds to each one-CTA candidate the cheaper of the two operand
// conversions (a separate pass, or in-ring conversion in a single-wave
// launch); fring is the in_ring knob (0 never in ring, 1 by that estimate,
// 2 always on one-CTA shapes).  Pure (host arithmetic only).
Shape plan_shape(int64_t M, int64_t N, int64_t num_kb, int sms, bool f16, int esize, int fpair, int ftile,
                 int fks, const ptc::ClusterCaps &caps, int conv = 0, int fring = 0) {
    const int64_t pass = conv != 0 ? pass_clocks(M, N, num_kb) : 0;
    // Marks `sh` in-ring when that is allowed and estimated cheaper; returns
    // the conversion's estimated clocks.
    auto conversion = [&](Shape &sh, int64_t tiles) -> int64_t {
        sh.ring = false;
        if (conv == 0 || fring == 0 || sh.ctas != 1) return pass;
        if (fring == 2) {
            sh.ring = true;
            return 0;
        }
        if (tiles * sh.ks > sms) return pass;  // several tiles per CTA: the pass
        const int64_t r = ring_clocks(num_kb, sh.bn, sh.ks, conv);
        sh.ring = r < pass;
        return sh.ring ? r : pass;
    };
    if (fpair == 2) return {2, ptc::kBN, 1};
    if ((ftile == 64 || ftile == 128) && tile_count(M, N, ptc::kBM, ftile) <= (int64_t(1) << 20)) {
        Shape sh{1, ftile, (fks == 2 || fks == 4) ? fks : 1};
        conversion(sh, tile_count(M, N, ptc::kBM, ftile));
        return sh;
    }
    const int64_t t256 = tile_count(M, N, ptc::kBM, ptc::kBN);
    if (fpair == 1) {
        Shape sh{1, ptc::kBN, fks};
        Shape est = sh;  // the K-split the launcher will pick, for the estimate
        est.ks = (fks == 1 || 2 * t256 > sms) ? 1 : ptc::pick_ksplit_pure(int(t256), int(num_kb), fks, sms, caps);
        conversion(est, t256);
        sh.ring = est.ring;
        return sh;
    }
    if (t256 >= sms) return {2, ptc::kBN, 1};
    Shape best{1, ptc::kBN, 1};
    int64_t best_c = est_clocks(num_kb, ptc::kBN, 1, esize) + conversion(best, t256);
    if (fks != 1) {
        const int ks = ptc::pick_ksplit_pure(int(t256), int(num_kb), fks, sms, caps);
        if (ks > 1) {
            Shape sh{1, ptc::kBN, ks};
            const int64_t c = est_clocks(num_kb, ptc::kBN, ks, esize) + conversion(sh, t256);
            if (fks != 0 || c < best_c) {
                best = sh;
                best_c = fks != 0 ? 0 : c;
            }
        }
    }
    for (int bn : {128, 64}) {
        const int64_t tiles = tile_count(M, N, ptc::kBM, bn);
        if (ftile != 0 || tiles > sms) continue;
        // whole narrow tiles, or K-split clusters of 2 / 4 of them (at least
        // two K blocks per CTA; one with in-ring conversion, where the split
        // shortens the conversion too: measured fastest for INT4 at N = 512)
        for (int ks : {1, 2, 4}) {
            if (ks > 1 && (fks == 1 || (fks != 0 && fks != ks) || num_kb < ks || tiles > caps.of(ks)))
                continue;
            Shape sh{1, bn, ks};
            const int64_t conv_c = conversion(sh, tiles);
            if (ks > 1 && num_kb < 2 * ks && !sh.ring) continue;
            const int64_t c = est_clocks(num_kb, bn, ks, esize) + conv_c;
            if (c < best_c) {
                best = sh;
                best_c = c;
            }
        }
    }
    if (best.bn == ptc::kBN && best.ks == 1 && f16 && t256 >= 32) return {2, ptc::kBN, 1};
    return best;
}

Shape choose_shape(int64_t M, int64_t N, int64_t num_kb, int sms, bool f16, int esize, int conv = 0) {
    return plan_shape(M, N, num_kb, sms, f16, esize, g_cta_pair.load(), g_tile_n.load(), g_ksplit.load(),
                      ptc::cluster_caps(sms), conv, g_in_ring.load());
}

GemmArgs base_args(int64_t M, int64_t N, int64_t K, int k_elems_per_block, void *C, int64_t ldc,
                   const Shape &sh) {
    const int ctas = sh.ctas;
    GemmArgs a;
    std::memset(&a, 0, sizeof(a));
    a.C = C;
    a.ldc = ldc;
    a.M = int(M);
    a.N = int(N);
    a.K = int(K);
    const int64_t tile_m = int64_t(ptc::kBM) * ctas;
    a.tiles_m = int((M + tile_m - 1) / tile_m);
    a.bn = sh.ctas == 1 ? sh.bn : ptc::kBN;
    a.tiles_n = int((N + a.bn - 1) / a.bn);
    a.num_tiles = a.tiles_m * a.tiles_n;
    a.num_kb = int((K + k_elems_per_block - 1) / k_elems_per_block);
    a.kb_per_chunk = a.num_kb;
    a.group_m = g_group_m.load() > 0 ? g_group_m.load() : 1;
    a.stall_tile = int(g_stall_tile.exchange(-1));
    a.l2_hint = g_l2_hint.load();
    a.split_ok = g_tail_split.load();
    a.split_min_kb = g_split_min_kb.load();
    a.stage_kb = g_pair_stage_kb.load();
    a.ksplit = sh.ks;
    a.split_reduce = g_split_reduce.load();
    a.pdl = g_pdl.load();
    a.wait_limit_ns = g_wait_ns.load();
    a.probe = g_clock_probe.load();
    a.pairs = 1;
    return a;
}

int launch_gemm_checked(Kind kind, bool b_mn, int epi, int ctas, const CUtensorMap &ta,
                        const CUtensorMap &tb, const GemmArgs &args, const DevInfo &d,
                        cudaStream_t stream) {
    cudaError_t e = ptc::launch_gemm(kind, b_mn, epi, ctas, ta, tb, args, d.sms, d.pool_ok ? d.pool : nullptr, stream);
    if (e != cudaSuccess) return fail_cuda(e, "GEMM kernel launch");
    g_launches.fetch_add(1);
    return PTC_OK;
}

int zero_c(void *C, int64_t ldc, int64_t M, int64_t N, int esize, const DevInfo &d, cudaStream_t stream) {
    cudaError_t e = ptc::launch_zero_fill(C, ldc, int(M), int(N), esize, d.sms * 4, stream);
    if (e != cudaSuccess) return fail_cuda(e, "zero-fill launch");
    g_launches.fetch_add(1);
    return PTC_OK;
}

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

}  // namespace

namespace ptc {
void note_launches(uint64_t n) { g_launches.fetch_add(n); }
void set_message(const char *text) { std::snprintf(g_msg, sizeof(g_msg), "%s", text); }
int encode_tmap_c32(CUtensorMap *map, const void *C, uint64_t n, uint64_t m, uint64_t ldc, bool fp32) {
    // The element type matters to TMA reductions only (stores copy bits).
    return make_tmap(map, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_INT32, C, n, m, ldc * 4,
                     32, 32);
}
int encode_tmap_2d(CUtensorMap *map, bool one_byte, const void *base, uint64_t inner, uint64_t outer,
                   uint64_t pitch, uint32_t box_inner, uint32_t box_outer) {
    return make_tmap(map, one_byte ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                     base, inner, outer, pitch, box_inner, box_outer);
}
}  // namespace ptc

namespace {

// FP16 operands: validation, tensor maps, one kernel launch.  epi is
// EPI_F32 (FP32 accumulators, FP32 C) or EPI_F16ACC (FP16 accumulators, FP16 C).
int f16_gemm(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B, int64_t ldb,
             void *C, int64_t ldc, int epi, void *stream) {
    g_last_conv = 0;
    int rc = check_sizes(M, N, K);
    if (rc) return rc;
    if (M == 0 || N == 0) return PTC_OK;
    if ((rc = check_ld(K > 0 ? lda : 0, K > 0 ? ldb : 0, ldc))) return rc;
    const int eb = epi == ptc::EPI_F16ACC ? 2 : 4;
    if (!C || ldc < N) return fail(PTC_ERR_INVALID, "C is NULL or ldc < N");
    if (K > 0 && (!A || !B)) return fail(PTC_ERR_INVALID, "A or B is NULL");
    if (K > 0 && (lda < K || ldb < N)) return fail(PTC_ERR_INVALID, "lda < K or ldb < N");
    if (!aligned16(C) || (ldc * eb) % 16)
        return fail(PTC_ERR_ALIGN, "C must be 16-byte aligned with a row pitch that is a multiple of 16 bytes");
    if (K > 0 && (!aligned16(A) || !aligned16(B) || lda % 8 || ldb % 8))
        return fail(PTC_ERR_ALIGN, "A, B must be 16-byte aligned, lda % 8 == 0, ldb % 8 == 0");
    const uint64_t cbytes = span_bytes(M, N, ldc, eb, 1);
    if (K > 0 && (overlaps(C, cbytes, A, span_bytes(M, K, lda, 2, 1)) ||
                  overlaps(C, cbytes, B, span_bytes(K, N, ldb, 2, 1))))
        return fail(PTC_ERR_OVERLAP, "C overlaps A or B");

    int dev;
    DevInfo *d;
    if ((rc = current_device(&dev, &d))) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) return zero_c(C, ldc, M, N, eb, *d, s);

    const Shape sh = choose_shape(M, N, (K + 63) / 64, d->sms, true, eb);
    const int pairs = (sh.ctas == 2 && g_multicast.load() == 1) ? 2 : 1;
    CUtensorMap ta, tb;
    if ((rc = make_tmap(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, A, K, M, uint64_t(lda) * 2, 64, ptc::kBM / pairs)))
        return rc;
    if ((rc = make_tmap(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, B, N, K, uint64_t(ldb) * 2, 64, 64)))
        return rc;
    GemmArgs args = base_args(M, N, K, 64, C, ldc, sh);
    args.pairs = pairs;
    return launch_gemm_checked(Kind::F16, true, epi, sh.ctas, ta, tb, args, *d, s);
}

}  // namespace

extern "C" {

int gemm_f16(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B,
             int64_t ldb, float *C, int64_t ldc, void *stream) {
    g_msg[0] = 0;
    return f16_gemm(M, N, K, A, lda, B, ldb, C, ldc, ptc::EPI_F32, stream);
}

int gemm_f16_f16acc(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B,
                    int64_t ldb, void *C, int64_t ldc, void *stream) {
    g_msg[0] = 0;
    return f16_gemm(M, N, K, A, lda, B, ldb, C, ldc, ptc::EPI_F16ACC, stream);
}

}  // extern "C"

namespace {

// Bytes of one output element of an integer-route mode.
int out_bytes(int mode) { return (mode == ptc::OUT_BF16 || mode == ptc::OUT_F16) ? 2 : 4; }

// The integer routes: validation, operand conversion into a stream-ordered
// workspace, then the tensor-core kernel whose epilogue folds the FP32 chunk
// sums into int32 and writes int32 or scaled FP32 / BF16 / FP16.
//   s4 == false: INT8, lda / ldb in bytes; s4 == true: packed INT4, in nibbles.
int int_gemm(bool s4, int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B,
             int64_t ldb, void *C, int64_t ldc, int mode, const float *sa, const float *sb,
             void *stream) {
    g_last_conv = 0;
    int rc = check_sizes(M, N, K);
    if (rc) return rc;
    if (M == 0 || N == 0) return PTC_OK;
    if ((rc = check_ld(K > 0 ? lda : 0, K > 0 ? ldb : 0, ldc))) return rc;
    const int eb = out_bytes(mode);
    if (!C || ldc < N) return fail(PTC_ERR_INVALID, "C is NULL or ldc < N");
    if (K > 0 && (!A || !B)) return fail(PTC_ERR_INVALID, "A or B is NULL");
    if (K > 0 && (lda < K || ldb < K)) return fail(PTC_ERR_INVALID, "lda < K or ldb < K");
    if (s4 && K > 0 && ((lda & 1) || (ldb & 1)))
        return fail(PTC_ERR_INVALID, "lda, ldb must be even (counted in nibbles)");
    if (!aligned16(C) || (ldc * eb) % 16)
        return fail(PTC_ERR_ALIGN, "C must be 16-byte aligned with a row pitch that is a multiple of 16 bytes");
    const int pitch_mult = s4 ? 32 : 16;
    if (K > 0 && (!aligned16(A) || !aligned16(B) || lda % pitch_mult || ldb % pitch_mult))
        return fail(PTC_ERR_ALIGN, s4 ? "A, B must be 16-byte aligned, lda % 32 == 0, ldb % 32 == 0"
                                      : "A, B must be 16-byte aligned, lda % 16 == 0, ldb % 16 == 0");
    if ((sa && (reinterpret_cast<uintptr_t>(sa) & 3u)) || (sb && (reinterpret_cast<uintptr_t>(sb) & 3u)))
        return fail(PTC_ERR_ALIGN, "scale vectors must be 4-byte aligned");
    const uint64_t cbytes = span_bytes(M, N, ldc, eb, 1);
    const int den = s4 ? 2 : 1;
    if (K > 0 && (overlaps(C, cbytes, A, span_bytes(M, K, lda, 1, den)) ||
                  overlaps(C, cbytes, B, span_bytes(N, K, ldb, 1, den))))
        return fail(PTC_ERR_OVERLAP, "C overlaps A or B");
    if ((sa && overlaps(C, cbytes, sa, uint64_t(M) * 4)) || (sb && overlaps(C, cbytes, sb, uint64_t(N) * 4)))
        return fail(PTC_ERR_OVERLAP, "C overlaps a scale vector");

    int dev;
    DevInfo *d;
    if ((rc = current_device(&dev, &d))) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) return zero_c(C, ldc, M, N, eb, *d, s);

    const int k_elems = s4 ? 128 : 64;  // elements per 128-byte K block
    const int wsize = s4 ? 1 : 2;       // workspace bytes per element
    const int64_t ldw = round_up(K, k_elems);
    // In-ring conversion (chosen with the shape, for one-CTA shapes): the
    // kernel loads K blocks of the raw operands (64 bytes per row: 64 s8 or
    // 128 packed s4; zeros past K) and converts them in shared memory, with no
    // workspace and no separate pass.  Packed s4 needs an even K (no stray
    // high nibble).
    const int conv = s4 ? (K % 2 == 0 ? 2 : 0) : 1;
    Shape sh = choose_shape(M, N, ldw / k_elems, d->sms, false, eb, conv);
    // CTA pairs convert inside the kernel when the pair_in_ring knob says so.
    if (sh.ctas == 2 && conv != 0 && g_pair_in_ring.load() == 2) sh.ring = true;
    const int chunk = s4 ? g_chunk_s4.load() : g_chunk_s8.load();
    if (sh.ring) {
        const uint64_t kbytes = uint64_t(s4 ? K / 2 : K);
        CUtensorMap ta, tb;
        rc = make_tmap(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, kbytes, uint64_t(M), uint64_t(s4 ? lda / 2 : lda), 64,
                       ptc::kBM, CU_TENSOR_MAP_SWIZZLE_NONE);
        if (!rc)
            rc = make_tmap(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, kbytes, uint64_t(N), uint64_t(s4 ? ldb / 2 : ldb),
                           64, uint32_t(sh.bn / sh.ctas), CU_TENSOR_MAP_SWIZZLE_NONE);
        if (rc) return rc;
        GemmArgs args = base_args(M, N, K, k_elems, C, ldc, sh);
        args.kb_per_chunk = chunk > 0 ? chunk : 1;
        args.out_mode = mode;
        args.scale_a = sa;
        args.scale_b = sb;
        args.in_ring = 1;
        rc = launch_gemm_checked(s4 ? Kind::E4M3 : Kind::F16, false, ptc::EPI_INT, sh.ctas, ta, tb, args, *d, s);
        if (!rc) g_last_conv = 2;
        return rc;
    }
    if (!d->pool_ok) return fail(PTC_ERR_ALLOC, "workspace memory pool unavailable");

    // Workspace: A and B as rows of K in the MMA input type (binary16 for
    // INT8, E4M3 for INT4), pitch rounded to 128 bytes, blocks 1024-aligned.
    // With the conversion in the GEMM kernel (knob "conv_fused": 256-wide
    // tiles without a K split, one pair per cluster) the converter warps write
    // it, and the counters of converted pieces follow it.
    const int pairs = (sh.ctas == 2 && g_multicast.load() == 1) ? 2 : 1;
    const bool fused = g_conv_fused.load() == 1 && sh.bn == ptc::kBN && sh.ks <= 1 && pairs == 1 &&
                       ptc::conv_counter_words(M, N, K) < (int64_t(1) << 30);
    const int64_t a_bytes = round_up(M * ldw * wsize, 1024);
    const int64_t b_bytes = round_up(N * ldw * wsize, 1024);
    const int64_t c_bytes = fused ? round_up(ptc::conv_counter_words(M, N, K) * 4, 256) : 0;
    void *ws = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&ws, size_t(a_bytes + b_bytes + c_bytes), d->pool, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(PTC_ERR_ALLOC, "workspace allocation failed");
    }
    uint8_t *aw = static_cast<uint8_t *>(ws);
    uint8_t *bw = aw + a_bytes;
    const int cgrid = d->sms * 16;  // 16 CTAs per SM: measured 6% faster than 8 at N = 8192
    rc = PTC_OK;
    if (fused)
        e = cudaSuccess;
    else if (s4)
        e = ptc::launch_s4_to_e4m3_pair(static_cast<const uint8_t *>(A), lda / 2, int(M),
                                        static_cast<const uint8_t *>(B), ldb / 2, int(N), int(K), aw, bw,
                                        ldw, cgrid, s, g_pdl.load() != 0);
    else
        e = ptc::launch_s8_to_f16_pair(static_cast<const int8_t *>(A), lda, int(M),
                                       static_cast<const int8_t *>(B), ldb, int(N), int(K),
                                       reinterpret_cast<uint16_t *>(aw), reinterpret_cast<uint16_t *>(bw),
                                       ldw, cgrid, s, g_pdl.load() != 0);
    if (e != cudaSuccess)
        rc = fail_cuda(e, "operand conversion launch");
    else if (!fused)
        g_launches.fetch_add(1);
    const CUtensorMapDataType dt = s4 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap ta, tb;
    if (!rc) rc = make_tmap(&ta, dt, aw, K, M, uint64_t(ldw) * wsize, k_elems, ptc::kBM / pairs);
    if (!rc) rc = make_tmap(&tb, dt, bw, K, N, uint64_t(ldw) * wsize, k_elems, sh.bn / sh.ctas);
    if (!rc) {
        GemmArgs args = base_args(M, N, K, k_elems, C, ldc, sh);
        args.pairs = pairs;
        args.kb_per_chunk = chunk > 0 ? chunk : 1;
        args.out_mode = mode;
        args.scale_a = sa;
        args.scale_b = sb;
        if (fused) {
            args.conv = 1;
            args.conv_a = static_cast<const uint8_t *>(A);
            args.conv_b = static_cast<const uint8_t *>(B);
            args.conv_lda = s4 ? lda / 2 : lda;
            args.conv_ldb = s4 ? ldb / 2 : ldb;
            args.conv_wa = aw;
            args.conv_wb = bw;
            args.conv_ldw = ldw;
            args.conv_count = reinterpret_cast<uint32_t *>(bw + b_bytes);
        }
        rc = launch_gemm_checked(s4 ? Kind::E4M3 : Kind::F16, false, ptc::EPI_INT, sh.ctas, ta, tb, args, *d, s);
        if (!rc) g_last_conv = fused ? 3 : 1;
    }
    cudaFreeAsync(ws, s);
    return rc;
}

// INT8 with B row-major (K x N): A converted as for gemm_s8, B converted into
// K rows of N binary16 values, read by the MMAs as an MN-major operand (the
// same layout as gemm_f16's B).
int s8_rowb_gemm(int64_t M, int64_t N, int64_t K, const int8_t *A, int64_t lda, const int8_t *B, int64_t ldb,
                 int32_t *C, int64_t ldc, void *stream) {
    g_last_conv = 0;
    int rc = check_sizes(M, N, K);
    if (rc) return rc;
    if (M == 0 || N == 0) return PTC_OK;
    if ((rc = check_ld(K > 0 ? lda : 0, K > 0 ? ldb : 0, ldc))) return rc;
    if (!C || ldc < N) return fail(PTC_ERR_INVALID, "C is NULL or ldc < N");
    if (K > 0 && (!A || !B)) return fail(PTC_ERR_INVALID, "A or B is NULL");
    if (K > 0 && (lda < K || ldb < N)) return fail(PTC_ERR_INVALID, "lda < K or ldb < N");
    if (!aligned16(C) || (ldc * 4) % 16)
        return fail(PTC_ERR_ALIGN, "C must be 16-byte aligned with a row pitch that is a multiple of 16 bytes");
    if (K > 0 && (!aligned16(A) || !aligned16(B) || lda % 16 || ldb % 16))
        return fail(PTC_ERR_ALIGN, "A, B must be 16-byte aligned, lda % 16 == 0, ldb % 16 == 0");
    const uint64_t cbytes = span_bytes(M, N, ldc, 4, 1);
    if (K > 0 && (overlaps(C, cbytes, A, span_bytes(M, K, lda, 1, 1)) ||
                  overlaps(C, cbytes, B, span_bytes(K, N, ldb, 1, 1))))
        return fail(PTC_ERR_OVERLAP, "C overlaps A or B");

    int dev;
    DevInfo *d;
    if ((rc = current_device(&dev, &d))) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) return zero_c(C, ldc, M, N, 4, *d, s);
    if (!d->pool_ok) return fail(PTC_ERR_ALLOC, "workspace memory pool unavailable");

    const int64_t ldw_a = round_up(K, 64);  // binary16 elements per A row (128-byte multiple)
    const int64_t ldw_b = round_up(N, 64);  // binary16 elements per B row
    const int64_t a_bytes = round_up(M * ldw_a * 2, 1024);
    const int64_t b_bytes = round_up(K * ldw_b * 2, 1024);
    void *ws = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&ws, size_t(a_bytes + b_bytes), d->pool, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(PTC_ERR_ALLOC, "workspace allocation failed");
    }
    uint16_t *aw = static_cast<uint16_t *>(ws);
    uint16_t *bw = reinterpret_cast<uint16_t *>(static_cast<uint8_t *>(ws) + a_bytes);
    const int cgrid = d->sms * 16;  // 16 CTAs per SM: measured 6% faster than 8 at N = 8192
    rc = PTC_OK;
    e = ptc::launch_s8_to_f16(A, lda, int(M), int(K), aw, ldw_a, cgrid, s, g_pdl.load() != 0);
    if (e == cudaSuccess) {
        g_launches.fetch_add(1);
        e = ptc::launch_s8_to_f16(B, ldb, int(K), int(N), bw, ldw_b, cgrid, s, g_pdl.load() != 0);
        if (e == cudaSuccess) g_launches.fetch_add(1);
    }
    if (e != cudaSuccess) rc = fail_cuda(e, "operand conversion launch");
    const Shape sh = choose_shape(M, N, (K + 63) / 64, d->sms, false, 4);
    CUtensorMap ta, tb;
    if (!rc) rc = make_tmap(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, aw, K, M, uint64_t(ldw_a) * 2, 64, ptc::kBM);
    if (!rc) rc = make_tmap(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, bw, N, K, uint64_t(ldw_b) * 2, 64, 64);
    if (!rc) {
        GemmArgs args = base_args(M, N, K, 64, C, ldc, sh);
        const int ch = g_chunk_s8.load();
        args.kb_per_chunk = ch > 0 ? ch : 1;
        args.out_mode = ptc::OUT_S32;
        rc = launch_gemm_checked(Kind::F16, true, ptc::EPI_INT, sh.ctas, ta, tb, args, *d, s);
        if (!rc) g_last_conv = 1;
    }
    cudaFreeAsync(ws, s);
    return rc;
}

// ------------------------------------------------------------ host buffers
// Library-owned copy streams of one device (created on first use).
struct CopyStreams {
    std::once_flag once;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    int ok = 0;
};
CopyStreams g_copy[kMaxDevices];

int copy_streams(int dev, CopyStreams **out) {
    CopyStreams &c = g_copy[dev];
    std::call_once(c.once, [&] {
        if (cudaStreamCreateWithFlags(&c.h2d, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&c.d2h, cudaStreamNonBlocking) == cudaSuccess)
            c.ok = 1;
        else
            cudaGetLastError();
    });
    if (!c.ok) return fail(PTC_ERR_LAUNCH, "could not create the library's copy streams");
    *out = &c;
    return PTC_OK;
}

// Events of one host-buffer call; destroyed (lazily, by the driver) on return.
struct EventSet {
    cudaEvent_t ev[64];
    int n = 0;
    cudaError_t make(cudaEvent_t *e) {
        cudaError_t r = cudaEventCreateWithFlags(e, cudaEventDisableTiming);
        if (r == cudaSuccess) ev[n++] = *e;
        return r;
    }
    ~EventSet() {
        for (int i = 0; i < n; ++i) cudaEventDestroy(ev[i]);
    }
};

// One GEMM with host-resident A, B and C, pipelined over row panels of A / C:
//   copy stream 1: B, then the A panels (host -> device)
//   caller's stream: operand conversion (integer routes) and the tensor-core
//                    kernel of each panel as soon as its A panel has arrived
//   copy stream 2: each C panel (device -> host) as soon as its kernel is done
// Device buffers come from the library pool, stream-ordered on the caller's
// stream; everything runs after the work already queued on that stream, and
// the stream waits for the last copy.  prec: 0 FP16, 1 INT8, 2 packed INT4.
int host_gemm(int prec, int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B,
              int64_t ldb, void *C, int64_t ldc, void *stream) {
    g_last_conv = 0;
    int rc = check_sizes(M, N, K);
    if (rc) return rc;
    if (M == 0 || N == 0) return PTC_OK;
    if ((rc = check_ld(K > 0 ? lda : 0, K > 0 ? ldb : 0, ldc))) return rc;
    const bool f16 = prec == 0, s4 = prec == 2;
    if (!C || ldc < N) return fail(PTC_ERR_INVALID, "C is NULL or ldc < N");
    if (K > 0 && (!A || !B)) return fail(PTC_ERR_INVALID, "A or B is NULL");
    if (K > 0 && (lda < K || ldb < (f16 ? N : K))) return fail(PTC_ERR_INVALID, "lda or ldb below its minimum");
    if (s4 && K > 0 && ((lda & 1) || (ldb & 1)))
        return fail(PTC_ERR_INVALID, "lda, ldb must be even (counted in nibbles)");
    if (!aligned16(C) || ldc % 4) return fail(PTC_ERR_ALIGN, "C must be 16-byte aligned, ldc % 4 == 0");
    const int pitch_mult = f16 ? 8 : (s4 ? 32 : 16);
    if (K > 0 && (!aligned16(A) || !aligned16(B) || lda % pitch_mult || ldb % pitch_mult))
        return fail(PTC_ERR_ALIGN, "A, B must be 16-byte aligned with 16-byte row pitches");
    // Bytes per element x 2 (nibbles count half a byte).
    const int e2 = f16 ? 4 : (s4 ? 1 : 2);
    const uint64_t cbytes = span_bytes(M, N, ldc, 4, 1);
    if (K > 0 && (overlaps(C, cbytes, A, span_bytes(M, K, lda, e2, 2)) ||
                  overlaps(C, cbytes, B, f16 ? span_bytes(K, N, ldb, 2, 1) : span_bytes(N, K, ldb, e2, 2))))
        return fail(PTC_ERR_OVERLAP, "C overlaps A or B");

    int dev;
    DevInfo *d;
    if ((rc = current_device(&dev, &d))) return rc;
    if (!d->pool_ok) return fail(PTC_ERR_ALLOC, "workspace memory pool unavailable");
    CopyStreams *cs;
    if ((rc = copy_streams(dev, &cs))) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    // Device copies with 16-byte row pitches, plus the integer routes' workspace.
    const int64_t a_row = (K * e2 + 1) / 2, a_pitch = round_up(a_row > 0 ? a_row : 1, 16);
    const int64_t b_rows = f16 ? K : N, b_row = f16 ? N * 2 : (K * e2 + 1) / 2;
    const int64_t b_pitch = round_up(b_row > 0 ? b_row : 1, 16);
    const int64_t c_pitch = round_up(N * 4, 16);
    const int k_elems = f16 ? 64 : (s4 ? 128 : 64);
    const int wsize = s4 ? 1 : 2;
    const int64_t ldw = round_up(K > 0 ? K : 1, k_elems);
    int64_t off = 0;
    const int64_t off_a = off;
    off += round_up(M * a_pitch, 1024);
    const int64_t off_b = off;
    off += round_up(b_rows * b_pitch, 1024);
    const int64_t off_c = off;
    off += round_up(M * c_pitch, 1024);
    const int64_t off_wa = off;
    if (!f16) off += round_up(M * ldw * wsize, 1024);
    const int64_t off_wb = off;
    if (!f16) off += round_up(N * ldw * wsize, 1024);
    void *ws = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&ws, size_t(off), d->pool, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(PTC_ERR_ALLOC, "device buffers for host operands could not be allocated");
    }
    uint8_t *base = static_cast<uint8_t *>(ws);
    uint8_t *Ad = base + off_a, *Bd = base + off_b, *Cd = base + off_c;
    uint8_t *Wa = base + off_wa, *Wb = base + off_wb;

    // Row panels: 2048 rows (several waves of tiles each) once M allows four.
    const int64_t panel = (M >= 4 * 2048) ? 2048 : M;
    const int npanels = int((M + panel - 1) / panel);
    EventSet evs;
    cudaEvent_t ev_start, ev_b, ev_done;
    rc = PTC_OK;
    auto cuda = [&](cudaError_t r, const char *what) {
        if (rc == PTC_OK && r != cudaSuccess) rc = fail_cuda(r, what);
        return rc == PTC_OK;
    };
    if (npanels > 28) rc = fail(PTC_ERR_INVALID, "too many row panels");
    if (!cuda(evs.make(&ev_start), "event") || !cuda(evs.make(&ev_b), "event") ||
        !cuda(evs.make(&ev_done), "event")) {
        cudaFreeAsync(ws, s);
        return rc;
    }
    cuda(cudaEventRecord(ev_start, s), "event record");
    cuda(cudaStreamWaitEvent(cs->h2d, ev_start, 0), "stream wait");
    cuda(cudaStreamWaitEvent(cs->d2h, ev_start, 0), "stream wait");

    if (K == 0) {
        if (rc == PTC_OK) {
            cudaError_t r = ptc::launch_zero_fill(Cd, c_pitch / 4, int(M), int(N), 4, d->sms * 4, s);
            if (cuda(r, "zero-fill launch")) g_launches.fetch_add(1);
        }
        cuda(cudaMemcpy2DAsync(C, size_t(ldc) * 4, Cd, size_t(c_pitch), size_t(N) * 4, size_t(M),
                               cudaMemcpyDeviceToHost, s), "C copy to host");
        cudaFreeAsync(ws, s);
        return rc;
    }

    // B, then the A panels, host -> device.
    cuda(cudaMemcpy2DAsync(Bd, size_t(b_pitch), B, size_t(f16 ? ldb * 2 : (ldb * e2) / 2), size_t(b_row),
                           size_t(b_rows), cudaMemcpyHostToDevice, cs->h2d), "B copy to device");
    cuda(cudaEventRecord(ev_b, cs->h2d), "event record");
    cudaEvent_t ev_a[32], ev_c[32];
    for (int p = 0; p < npanels && rc == PTC_OK; ++p) {
        const int64_t r0 = p * panel, rows = std::min(panel, M - r0);
        if (!cuda(evs.make(&ev_a[p]), "event") || !cuda(evs.make(&ev_c[p]), "event")) break;
        const size_t apitch_host = size_t((lda * e2) / 2);
        cuda(cudaMemcpy2DAsync(Ad + r0 * a_pitch, size_t(a_pitch),
                               static_cast<const uint8_t *>(A) + r0 * apitch_host, apitch_host, size_t(a_row),
                               size_t(rows), cudaMemcpyHostToDevice, cs->h2d), "A copy to device");
        cuda(cudaEventRecord(ev_a[p], cs->h2d), "event record");
    }

    // Kernels on the caller's stream, panel by panel.
    cuda(cudaStreamWaitEvent(s, ev_b, 0), "stream wait");
    const int cgrid = d->sms * 16;  // 16 CTAs per SM: measured 6% faster than 8 at N = 8192
    if (!f16 && rc == PTC_OK) {
        cudaError_t r = s4 ? ptc::launch_s4_to_e4m3_pair(Bd, b_pitch, 0, Bd, b_pitch, int(N), int(K), Wa, Wb,
                                                          ldw, cgrid, s, g_pdl.load() != 0)
                           : ptc::launch_s8_to_f16_pair(reinterpret_cast<const int8_t *>(Bd), b_pitch, 0,
                                                        reinterpret_cast<const int8_t *>(Bd), b_pitch, int(N),
                                                        int(K), reinterpret_cast<uint16_t *>(Wa),
                                                        reinterpret_cast<uint16_t *>(Wb), ldw, cgrid, s, g_pdl.load() != 0);
        if (cuda(r, "operand conversion launch")) g_launches.fetch_add(1);
    }
    for (int p = 0; p < npanels && rc == PTC_OK; ++p) {
        const int64_t r0 = p * panel, rows = std::min(panel, M - r0);
        cuda(cudaStreamWaitEvent(s, ev_a[p], 0), "stream wait");
        const Shape sh = choose_shape(rows, N, (K + k_elems - 1) / k_elems, d->sms, f16, 4);
        CUtensorMap ta, tb;
        if (f16) {
            if (rc == PTC_OK)
                rc = make_tmap(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, Ad + r0 * a_pitch, K, rows, a_pitch, 64, ptc::kBM);
            if (rc == PTC_OK)
                rc = make_tmap(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, Bd, N, K, b_pitch, 64, 64);
        } else {
            uint8_t *wa = Wa + r0 * ldw * wsize;
            cudaError_t r =
                s4 ? ptc::launch_s4_to_e4m3_pair(Ad + r0 * a_pitch, a_pitch, int(rows), Ad, a_pitch, 0, int(K), wa,
                                                 wa, ldw, cgrid, s, g_pdl.load() != 0)
                   : ptc::launch_s8_to_f16_pair(reinterpret_cast<const int8_t *>(Ad + r0 * a_pitch), a_pitch,
                                                int(rows), reinterpret_cast<const int8_t *>(Ad), a_pitch, 0, int(K),
                                                reinterpret_cast<uint16_t *>(wa), reinterpret_cast<uint16_t *>(wa),
                                                ldw, cgrid, s, g_pdl.load() != 0);
            if (cuda(r, "operand conversion launch")) g_launches.fetch_add(1);
            const CUtensorMapDataType dt = s4 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
            if (rc == PTC_OK) rc = make_tmap(&ta, dt, wa, K, rows, uint64_t(ldw) * wsize, k_elems, ptc::kBM);
            if (rc == PTC_OK) rc = make_tmap(&tb, dt, Wb, K, N, uint64_t(ldw) * wsize, k_elems, sh.bn / sh.ctas);
        }
        if (rc != PTC_OK) break;
        GemmArgs args = base_args(rows, N, K, k_elems, Cd + r0 * c_pitch, c_pitch / 4, sh);
        if (!f16) {
            const int ch = s4 ? g_chunk_s4.load() : g_chunk_s8.load();
            args.kb_per_chunk = ch > 0 ? ch : 1;
            args.out_mode = ptc::OUT_S32;
        }
        rc = launch_gemm_checked(s4 ? Kind::E4M3 : Kind::F16, f16, f16 ? ptc::EPI_F32 : ptc::EPI_INT, sh.ctas, ta, tb,
                                 args, *d, s);
        cuda(cudaEventRecord(ev_c[p], s), "event record");
        // C panel, device -> host, once its kernel is done.
        cuda(cudaStreamWaitEvent(cs->d2h, ev_c[p], 0), "stream wait");
        cuda(cudaMemcpy2DAsync(static_cast<uint8_t *>(C) + r0 * ldc * 4, size_t(ldc) * 4, Cd + r0 * c_pitch,
                               size_t(c_pitch), size_t(N) * 4, size_t(rows), cudaMemcpyDeviceToHost, cs->d2h),
             "C copy to host");
    }
    // The caller's stream waits for the last copy; the buffers go back to the pool after it.
    cudaError_t r1 = cudaEventRecord(ev_done, cs->d2h);
    cudaError_t r2 = cudaStreamWaitEvent(s, ev_done, 0);
    cudaError_t r3 = cudaStreamWaitEvent(s, ev_b, 0);
    cuda(r1, "event record");
    cuda(r2, "stream wait");
    cuda(r3, "stream wait");
    cudaFreeAsync(ws, s);
    return rc;
}

int scaled_mode(int out_type) {
    switch (out_type) {
        case PTC_OUT_F32: return ptc::OUT_F32;
        case PTC_OUT_BF16: return ptc::OUT_BF16;
        case PTC_OUT_F16: return ptc::OUT_F16;
        default: return -1;
    }
}

}  // namespace

extern "C" {

int gemm_s8(int64_t M, int64_t N, int64_t K, const int8_t *A, int64_t lda, const int8_t *B,
            int64_t ldb, int32_t *C, int64_t ldc, void *stream) {
    g_msg[0] = 0;
    return int_gemm(false, M, N, K, A, lda, B, ldb, C, ldc, ptc::OUT_S32, nullptr, nullptr, stream);
}

int gemm_s8_b_rowmajor(int64_t M, int64_t N, int64_t K, const int8_t *A, int64_t lda, const int8_t *B,
                       int64_t ldb, int32_t *C, int64_t ldc, void *stream) {
    g_msg[0] = 0;
    return s8_rowb_gemm(M, N, K, A, lda, B, ldb, C, ldc, stream);
}

int gemm_s4(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B,
            int64_t ldb, int32_t *C, int64_t ldc, void *stream) {
    g_msg[0] = 0;
    return int_gemm(true, M, N, K, A, lda, B, ldb, C, ldc, ptc::OUT_S32, nullptr, nullptr, stream);
}

int gemm_s8_scaled(int64_t M, int64_t N, int64_t K, const int8_t *A, int64_t lda, const int8_t *B,
                   int64_t ldb, const float *scale_a, const float *scale_b, void *C, int64_t ldc,
                   int out_type, void *stream) {
    g_msg[0] = 0;
    const int mode = scaled_mode(out_type);
    if (mode < 0) return fail(PTC_ERR_INVALID, "out_type must be PTC_OUT_F32, PTC_OUT_BF16 or PTC_OUT_F16");
    return int_gemm(false, M, N, K, A, lda, B, ldb, C, ldc, mode, scale_a, scale_b, stream);
}

int gemm_s4_scaled(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B,
                   int64_t ldb, const float *scale_a, const float *scale_b, void *C, int64_t ldc,
                   int out_type, void *stream) {
    g_msg[0] = 0;
    const int mode = scaled_mode(out_type);
    if (mode < 0) return fail(PTC_ERR_INVALID, "out_type must be PTC_OUT_F32, PTC_OUT_BF16 or PTC_OUT_F16");
    return int_gemm(true, M, N, K, A, lda, B, ldb, C, ldc, mode, scale_a, scale_b, stream);
}

int gemm_f16_host(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B,
                  int64_t ldb, float *C, int64_t ldc, void *stream) {
    g_msg[0] = 0;
    return host_gemm(0, M, N, K, A, lda, B, ldb, C, ldc, stream);
}

int gemm_s8_host(int64_t M, int64_t N, int64_t K, const int8_t *A, int64_t lda, const int8_t *B,
                 int64_t ldb, int32_t *C, int64_t ldc, void *stream) {
    g_msg[0] = 0;
    return host_gemm(1, M, N, K, A, lda, B, ldb, C, ldc, stream);
}

int gemm_s4_host(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B,
                 int64_t ldb, int32_t *C, int64_t ldc, void *stream) {
    g_msg[0] = 0;
    return host_gemm(2, M, N, K, A, lda, B, ldb, C, ldc, stream);
}

int gemm_baseline(int variant, int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B,
                  int64_t ldb, void *C, int64_t ldc, void *stream) {
    g_msg[0] = 0;
    if (variant < PTC_BASELINE_F16_WMMA || variant > PTC_BASELINE_S4_LDMATRIX)
        return fail(PTC_ERR_INVALID, "unknown baseline variant");
    const ptc::Variant v = static_cast<ptc::Variant>(variant);
    int rc = check_sizes(M, N, K);
    if (rc) return rc;
    if (M == 0 || N == 0) return PTC_OK;
    if ((rc = check_ld(K > 0 ? lda : 0, K > 0 ? ldb : 0, ldc))) return rc;
    const bool f16 = v == ptc::BASE_F16_WMMA || v == ptc::BASE_F16_MMA || v == ptc::BASE_F16_LDM;
    const bool s4 = v == ptc::BASE_S4_WMMA || v == ptc::BASE_S4_MMA || v == ptc::BASE_S4_LDM;
    const int kmult = ptc::baseline_k_multiple(v);
    if (M % 32 || N % 64 || K % kmult || K == 0)
        return fail(PTC_ERR_INVALID, "baseline kernels need M % 32 == 0, N % 64 == 0 and K a positive multiple "
                                     "of 32 (FP16), 64 (INT8) or 128 (INT4)");
    if (!A || !B || !C) return fail(PTC_ERR_INVALID, "A, B or C is NULL");
    if (lda < K || ldb < (f16 ? N : K) || ldc < N) return fail(PTC_ERR_INVALID, "leading dimension below its minimum");
    if (s4 && ((lda & 1) || (ldb & 1))) return fail(PTC_ERR_INVALID, "lda, ldb must be even (counted in nibbles)");
    const int64_t lda_b = f16 ? lda * 2 : (s4 ? lda / 2 : lda);
    const int64_t ldb_b = f16 ? ldb * 2 : (s4 ? ldb / 2 : ldb);
    if (!aligned16(A) || !aligned16(B) || lda_b % 16 || ldb_b % 16)
        return fail(PTC_ERR_ALIGN, "A, B must be 16-byte aligned with 16-byte row pitches");
    if ((reinterpret_cast<uintptr_t>(C) & 31u) || ldc % 8)
        return fail(PTC_ERR_ALIGN, "C must be 32-byte aligned, ldc % 8 == 0");
    const uint64_t cbytes = span_bytes(M, N, ldc, 4, 1);
    const int64_t a_row_bytes = f16 ? K * 2 : (s4 ? (K + 1) / 2 : K);
    if (overlaps(C, cbytes, A, span_bytes(M, a_row_bytes, lda_b, 1, 1)) ||
        overlaps(C, cbytes, B, f16 ? span_bytes(K, N * 2, ldb_b, 1, 1) : span_bytes(N, a_row_bytes, ldb_b, 1, 1)))
        return fail(PTC_ERR_OVERLAP, "C overlaps A or B");
    int dev;
    DevInfo *d;
    if ((rc = current_device(&dev, &d))) return rc;
    cudaError_t e = ptc::launch_baseline(v, A, lda_b, B, ldb_b, C, ldc, int(M), int(N), int(K),
                                         static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda(e, "baseline kernel launch");
    g_launches.fetch_add(1);
    return PTC_OK;
}

const char *gemm_status_string(int status) {
    static const char *names[] = {"PTC_OK",           "PTC_ERR_INVALID: invalid argument",
                                  "PTC_ERR_ALIGN: misaligned pointer or row pitch",
                                  "PTC_ERR_OVERLAP: C overlaps an input",
                                  "PTC_ERR_DEVICE: no compute capability 10.3 device",
                                  "PTC_ERR_LAUNCH: CUDA call failed",
                                  "PTC_ERR_TIMEOUT: a kernel pipeline wait timed out",
                                  "PTC_ERR_ALLOC: workspace allocation failed"};
    thread_local char buf[640];
    const char *base = (status >= 0 && status <= 7) ? names[status] : "unknown status";
    if (status != PTC_OK && g_msg[0])
        std::snprintf(buf, sizeof(buf), "%s (%s)", base, g_msg);
    else
        std::snprintf(buf, sizeof(buf), "%s", base);
    return buf;
}

int gemm_poll_device_error(void) {
    int dev;
    DevInfo *d;
    int rc = current_device(&dev, &d);
    if (rc) return rc;
    uint32_t w = 0;
    cudaError_t e = ptc::read_and_clear_error_word(&w);
    if (e != cudaSuccess) return fail_cuda(e, "reading the device error word");
    return w ? PTC_ERR_TIMEOUT : PTC_OK;
}

uint64_t ptc_kernel_launch_count(void) { return g_launches.load(); }

int ptc_clock_probe_read(uint64_t *cycles, uint64_t *ns, uint64_t *ctas) {
    if (!cycles || !ns || !ctas) return fail(PTC_ERR_INVALID, "NULL pointer");
    int dev;
    DevInfo *d;
    int rc = current_device(&dev, &d);
    if (rc) return rc;
    unsigned long long v[9];
    cudaError_t e = ptc::read_and_clear_clock_probe(v);
    if (e != cudaSuccess) return fail_cuda(e, "reading the clock record");
    for (int f = 0; f < 3; ++f) {
        cycles[f] = v[3 * f];
        ns[f] = v[3 * f + 1];
        ctas[f] = v[3 * f + 2];
    }
    return PTC_OK;
}

int ptc_debug_set_wait_limit(uint64_t timeout_ns, int64_t stall_tile) {
    g_wait_ns.store(timeout_ns ? timeout_ns : kDefaultWaitNs);
    g_stall_tile.store(stall_tile);
    return PTC_OK;
}

int ptc_plan_shape(int64_t M, int64_t N, int64_t K, int prec, int sms, int cap2, int cap4, int cap8, int *ctas,
                   int *tile_n, int *ksplit, int *in_ring) {
    if (!ctas || !tile_n || !ksplit) return fail(PTC_ERR_INVALID, "NULL pointer");
    if (prec < 0 || prec > 2 || sms <= 0 || cap2 < 0 || cap4 < 0 || cap8 < 0 || M <= 0 || N <= 0 || K <= 0)
        return fail(PTC_ERR_INVALID, "precision, SM count, capacities or sizes out of range");
    int rc = check_sizes(M, N, K);
    if (rc) return rc;
    ptc::ClusterCaps caps;
    caps.c2 = cap2;
    caps.c4 = cap4;
    caps.c8 = cap8;
    const int64_t num_kb = (K + (prec == 2 ? 127 : 63)) / (prec == 2 ? 128 : 64);
    const int conv = prec == 1 ? 1 : (prec == 2 && K % 2 == 0) ? 2 : 0;
    Shape sh = plan_shape(M, N, num_kb, sms, prec == 0, 4, g_cta_pair.load(), g_tile_n.load(), g_ksplit.load(),
                          caps, conv, g_in_ring.load());
    // what the launcher then runs for one-CTA tiles
    if (sh.ctas == 1 && sh.bn == ptc::kBN) {
        sh.ks = ptc::pick_ksplit_pure(int(tile_count(M, N, ptc::kBM, ptc::kBN)), int(num_kb), sh.ks, sms, caps);
    } else if (sh.ctas == 1 && sh.ks > 1 &&
               (num_kb < sh.ks || tile_count(M, N, ptc::kBM, sh.bn) > caps.of(sh.ks))) {
        sh.ks = 1;
    }
    *ctas = sh.ctas;
    *tile_n = sh.bn;
    *ksplit = sh.ks < 1 ? 1 : sh.ks;
    if (in_ring) *in_ring = sh.ring ? 1 : 0;
    return PTC_OK;
}

int ptc_last_launch(int *grid, int *cluster, int *ksplit, int *tile_n) {
    if (!grid || !cluster || !ksplit || !tile_n) return fail(PTC_ERR_INVALID, "NULL pointer");
    ptc::last_launch(grid, cluster, ksplit, tile_n);
    return PTC_OK;
}

int ptc_last_conversion(int *mode) {
    if (!mode) return fail(PTC_ERR_INVALID, "NULL pointer");
    *mode = g_last_conv;
    return PTC_OK;
}

int ptc_set_tuning(const char *key, int64_t value) {
    if (!key) return fail(PTC_ERR_INVALID, "key is NULL");
    // Fold lengths stay within exactness: every FP32 partial sum of a chunk is
    // an integer of magnitude <= 2^24 (s8: 64 values of |ab| <= 2^14 per K
    // block, so at most 16 blocks; E4M3 route: 128 values of |ab| <= 2^6, at
    // most 2048 blocks).
    if (std::strcmp(key, "s8_chunk_kb") == 0) {
        if (value > 0 && value % 2 == 0 && value <= kMaxChunkS8) {
            g_chunk_s8.store(int(value));
            return PTC_OK;
        }
        return fail(PTC_ERR_INVALID, "s8_chunk_kb must be even and in 2 .. 16 (exact FP32 partial sums)");
    }
    if (std::strcmp(key, "s4_chunk_kb") == 0) {
        if (value > 0 && value % 2 == 0 && value <= kMaxChunkS4) {
            g_chunk_s4.store(int(value));
            return PTC_OK;
        }
        return fail(PTC_ERR_INVALID, "s4_chunk_kb must be even and in 2 .. 2048 (exact FP32 partial sums)");
    }
    if (std::strcmp(key, "group_m") == 0 && value > 0 && value < (1 << 20)) {
        g_group_m.store(int(value));
        return PTC_OK;
    }
    if (std::strcmp(key, "l2_hint") == 0 && value >= 0 && value <= 3) {
        g_l2_hint.store(int(value));
        return PTC_OK;
    }
    if (std::strcmp(key, "tail_split") == 0 && (value == 0 || value == 1)) {
        g_tail_split.store(int(value));
        return PTC_OK;
    }
    if (std::strcmp(key, "pair_stage_kb") == 0 && (value == 1 || value == 2)) {
        g_pair_stage_kb.store(int(value));
        return PTC_OK;
    }
    if (std::strcmp(key, "split_min_kb") == 0 && value >= 2 && value <= (1 << 20)) {
        g_split_min_kb.store(int(value));
        return PTC_OK;
    }
    if (std::strcmp(key, "ksplit") == 0 && (value == 0 || value == 1 || value == 2 || value == 4 || value == 8)) {
        g_ksplit.store(int(value));
        return PTC_OK;
    }
    if (std::strcmp(key, "split_reduce") == 0 && (value == 0 || value == 1)) {
        g_split_reduce.store(int(value));
        return PTC_OK;
    }
    if (std::strcmp(key, "tile_n") == 0 && (value == 0 || value == 64 || value == 128 || value == 256)) {
        g_tile_n.store(int(value));
        return PTC_OK;
    }
    if (std::strcmp(key, "pdl") == 0 && (value == 0 || value == 1)) {
        g_pdl.store(int(value));
        return PTC_OK;
    }
    if (std::strcmp(key, "in_ring") == 0 && value >= 0 && value <= 2) {
        g_in_ring.store(int(value));
        return PTC_OK;
    }
    if (std::strcmp(key, "multicast") == 0 && (value == 0 || value == 1)) {
        g_multicast.store(int(value));
        return PTC_OK;
    }
    if (std::strcmp(key, "conv_fused") == 0 && (value == 0 || value == 1)) {
        g_conv_fused.store(int(value));
        return PTC_OK;
    }
    if (std::strcmp(key, "pair_in_ring") == 0 && (value == 0 || value == 2)) {
        g_pair_in_ring.store(int(value));
        return PTC_OK;
    }
    if (std::strcmp(key, "clock_probe") == 0 && (value == 0 || value == 1)) {
        g_clock_probe.store(int(value));
        return PTC_OK;
    }
    if (std::strcmp(key, "cta_pair") == 0 && value >= 0 && value <= 2) {
        g_cta_pair.store(int(value));
        return PTC_OK;
    }
    return fail(PTC_ERR_INVALID, "unknown tuning key or value out of range");
}

}  // extern "C"
