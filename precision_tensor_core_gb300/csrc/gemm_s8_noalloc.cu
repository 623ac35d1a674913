// gemm_s8_noalloc.cu -- the INT8 GEMM for callers that cannot allocate
// device memory.
//
// gemm_s8 needs scratch memory: A and B are rewritten as binary16 before the
// tensor-core kernel reads them, and that workspace comes from a memory pool
// at call time.  Some callers cannot let a library allocate: a host
// application whose own allocator has reserved the GPU's memory and forbids
// any other allocation, or a latency-bound path where a device allocation may
// block or fail at an arbitrary moment.  gemm_s8_noalloc runs the same two
// conversion kernels and the same tensor-core kernel, with the workspace taken
// from a fixed array in device global memory that the library's module
// defines.  It makes no allocation of any kind on any call.
//
// The array (kScratchBytes) is part of the library's device image: every GPU
// that loads the library holds it until the process exits.  Host code cannot
// use the array's name as a device address (on the host it names a stand-in),
// so the first call on each device, with that device current, asks the
// runtime for the array's device address with cudaGetSymbolAddress and keeps
// it; later calls on that device reuse it.  Make that first call before any
// stream capture begins.  Under CUDA's default lazy module loading, that first
// lookup is also what loads the library's device code onto the GPU and
// commits the array's memory: make the first call (or run with
// CUDA_MODULE_LOADING=EAGER) before the application's allocator reserves the
// device's memory.  A failed set-up is not remembered: the next call on that
// device tries again.
//
// All calls share the one array, and it keeps whatever the last call wrote.
// Nothing has to start at zero: each call writes every workspace element its
// tensor-core kernel reads before reading it (elements outside the matrix are
// zero-filled by the tensor-memory-access unit, not read from the array).
// Calls whose kernels overlap on the GPU (different streams, or several host
// threads) race on the array and give wrong results: serialise them.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "ptc.h"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;  // 32 MiB
static __device__ __align__(256) uint8_t g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
constexpr int kChunkKb = 8;        // 512 K values per fold: |partial| <= 2^23, exact in FP32
constexpr int kGroupM = 16;
constexpr uint64_t kWaitNs = 1000000000ull;

struct DeviceScratch {
    std::atomic<int> ok{0};  // set once the set-up below has succeeded
    int sms = 0;
    void *ptr = nullptr;  // device address of g_scratch on this device
};
DeviceScratch g_dev[kMaxDevices];
std::mutex g_setup;

// With the device current: check it and look up the scratch array's device
// address.  Done once per device on success; a failure is reported to the
// caller and retried by the next call.
int device_scratch(DeviceScratch **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        ptc::set_message("no usable current CUDA device");
        return PTC_ERR_DEVICE;
    }
    DeviceScratch &d = g_dev[dev];
    if (!d.ok.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(g_setup);
        if (!d.ok.load(std::memory_order_relaxed)) {
            char why[160];
            int major = 0, minor = 0, sms = 0;
            if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
                cudaGetLastError();
                std::snprintf(why, sizeof(why), "device %d attributes unavailable", dev);
                ptc::set_message(why);
                return PTC_ERR_DEVICE;
            }
            if (!(major == 10 && minor == 3 && sms > 0)) {
                std::snprintf(why, sizeof(why), "device %d is not a compute capability 10.3 GPU", dev);
                ptc::set_message(why);
                return PTC_ERR_DEVICE;
            }
            void *p = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
            if (e != cudaSuccess || p == nullptr) {
                std::snprintf(why, sizeof(why),
                              "cudaGetSymbolAddress of the scratch array failed (retried on the next call): %s",
                              cudaGetErrorString(e));
                cudaGetLastError();
                ptc::set_message(why);
                return PTC_ERR_DEVICE;
            }
            d.sms = sms;
            d.ptr = p;
            d.ok.store(1, std::memory_order_release);
        }
    }
    *out = &d;
    return PTC_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void *a, uint64_t alen, const void *b, uint64_t blen) {
    const unsigned __int128 a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + blen && b0 < a0 + alen;
}

// Bytes spanned by `rows` rows of `cols` elements of `esize` bytes at a pitch
// of `ld` elements (sizes <= 2^30, pitches <= 2^36: exact in 128 bits).
uint64_t span(int64_t rows, int64_t cols, int64_t ld, int esize) {
    return uint64_t((__int128(rows - 1) * ld + cols) * esize);
}

int reject(int code, const char *text) {
    ptc::set_message(text);
    return code;
}

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

}  // namespace

extern "C" int gemm_s8_noalloc(int64_t M, int64_t N, int64_t K, const int8_t *A, int64_t lda,
                               const int8_t *B, int64_t ldb, int32_t *C, int64_t ldc,
                               void *stream) {
    ptc::set_message("");
    // The same argument contract as gemm_s8.
    const int64_t kMaxDim = int64_t(1) << 30;
    if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return reject(PTC_ERR_INVALID, "sizes must satisfy 0 <= M, N, K <= 2^30");
    if (M == 0 || N == 0) return PTC_OK;
    if (!C || ldc < N) return reject(PTC_ERR_INVALID, "C is NULL or ldc < N");
    if (K > 0 && (!A || !B)) return reject(PTC_ERR_INVALID, "A or B is NULL");
    if (K > 0 && (lda < K || ldb < K)) return reject(PTC_ERR_INVALID, "lda < K or ldb < K");
    const int64_t kMaxLd = int64_t(1) << 36;
    if (ldc > kMaxLd || (K > 0 && (lda > kMaxLd || ldb > kMaxLd)))
        return reject(PTC_ERR_INVALID, "leading dimensions must be <= 2^36 elements");
    if (!aligned16(C) || ldc % 4) return reject(PTC_ERR_ALIGN, "C must be 16-byte aligned, ldc % 4 == 0");
    if (K > 0 && (!aligned16(A) || !aligned16(B) || lda % 16 || ldb % 16))
        return reject(PTC_ERR_ALIGN, "A, B must be 16-byte aligned, lda % 16 == 0, ldb % 16 == 0");
    const uint64_t cbytes = span(M, N, ldc, 4);
    if (K > 0 && (overlaps(C, cbytes, A, span(M, K, lda, 1)) || overlaps(C, cbytes, B, span(N, K, ldb, 1))))
        return reject(PTC_ERR_OVERLAP, "C overlaps A or B");

    // Workspace layout of gemm_s8: A then B as binary16 rows of K, pitch
    // rounded up to 64 values (128 bytes), each block 1024-byte aligned.
    const int64_t ldw = round_up(K > 0 ? K : 1, 64);
    const int64_t a_bytes = round_up(M * ldw * 2, 1024);
    const int64_t b_bytes = round_up(N * ldw * 2, 1024);
    if (K > 0 && a_bytes + b_bytes > int64_t(kScratchBytes)) {
        char text[200];
        std::snprintf(text, sizeof(text),
                      "problem needs %lld bytes of workspace, above the %lld-byte static scratch "
                      "of gemm_s8_noalloc ((M+N) * roundup(K,64) * 2 must fit); use gemm_s8",
                      static_cast<long long>(a_bytes + b_bytes), static_cast<long long>(kScratchBytes));
        return reject(PTC_ERR_INVALID, text);
    }

    DeviceScratch *d = nullptr;
    int rc = device_scratch(&d);
    if (rc) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (K == 0) {
        if ((e = ptc::launch_zero_fill(C, ldc, int(M), int(N), 4, d->sms * 4, s)) != cudaSuccess) {
            cudaGetLastError();
            return reject(PTC_ERR_LAUNCH, cudaGetErrorString(e));
        }
        ptc::note_launches(1);
        return PTC_OK;
    }

    uint16_t *aw = static_cast<uint16_t *>(d->ptr);
    uint16_t *bw = reinterpret_cast<uint16_t *>(static_cast<uint8_t *>(d->ptr) + a_bytes);
    const int cgrid = d->sms * 16;  // 16 CTAs per SM: measured 6% faster than 8 at N = 8192
    if ((e = ptc::launch_s8_to_f16(A, lda, int(M), int(K), aw, ldw, cgrid, s)) != cudaSuccess) {
        cudaGetLastError();
        return reject(PTC_ERR_LAUNCH, cudaGetErrorString(e));
    }
    ptc::note_launches(1);
    if ((e = ptc::launch_s8_to_f16(B, ldb, int(N), int(K), bw, ldw, cgrid, s)) != cudaSuccess) {
        cudaGetLastError();
        return reject(PTC_ERR_LAUNCH, cudaGetErrorString(e));
    }
    ptc::note_launches(1);

    CUtensorMap ta, tb;
    if ((rc = ptc::encode_tmap_2d(&ta, false, aw, K, M, uint64_t(ldw) * 2, 64, ptc::kBM))) return rc;
    if ((rc = ptc::encode_tmap_2d(&tb, false, bw, K, N, uint64_t(ldw) * 2, 64, ptc::kBN))) return rc;
    ptc::GemmArgs args;
    std::memset(&args, 0, sizeof(args));
    args.C = C;
    args.ldc = ldc;
    args.M = int(M);
    args.N = int(N);
    args.K = int(K);
    args.tiles_m = int((M + ptc::kBM - 1) / ptc::kBM);
    args.bn = ptc::kBN;
    args.tiles_n = int((N + ptc::kBN - 1) / ptc::kBN);
    args.num_tiles = args.tiles_m * args.tiles_n;
    args.num_kb = int((K + 63) / 64);
    args.kb_per_chunk = kChunkKb;
    args.group_m = kGroupM;
    args.stall_tile = -1;
    args.l2_hint = 0;
    args.out_mode = ptc::OUT_S32;
    args.scale_a = nullptr;
    args.scale_b = nullptr;
    args.wait_limit_ns = kWaitNs;
    if ((e = ptc::launch_gemm(ptc::Kind::F16, false, ptc::EPI_INT, 1, ta, tb, args, d->sms, nullptr, s)) != cudaSuccess) {
        cudaGetLastError();
        return reject(PTC_ERR_LAUNCH, cudaGetErrorString(e));
    }
    ptc::note_launches(1);
    return PTC_OK;
}
