/*
 * ptc.h -- C ABI of libptc: dense tensor-core matrix products C = A.B on one
 * NVIDIA GB300 (sm_103), in the three precisions of "Hand-Written PTX
 * Tensor-Core GEMM Kernels: A Multi-Precision Study on NVIDIA L4"
 * (Borowski & Osinski):
 *
 *   gemm_f16  FP16 operands, FP32 accumulation, FP32 result
 *             (section IV-A and Table VI: FP16 family with f32 accumulators;
 *             section IV-A's ~537 MB working set at N = 8192 is two FP16
 *             operands plus an FP32 C)
 *   gemm_s8   INT8 operands, INT32 accumulation, INT32 result (section IV-B)
 *   gemm_s4   packed INT4 operands, INT32 accumulation, INT32 result
 *             (section IV-C, Listings 1-2: mma ... .s32.s4.s4.s32)
 *
 * All three compute C <- A.B exactly as the plain sum over k, with C
 * overwritten and no scaling, bias or dequantisation (section VI "Scope":
 * INT32 accumulations without in-kernel dequantization or scaling).  The
 * paper's problems are square (section III-B, N = 512 ... 8192); general
 * M, N, K >= 0 are accepted.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - A, B, C are DEVICE pointers owned by the caller (any allocator).  The
 *   library keeps no pointer after the call returns.
 * - Sizes and leading dimensions are counted in ELEMENTS (for packed INT4:
 *   in 4-bit elements, i.e. nibbles).
 * - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every call
 *   is asynchronous on that stream and never synchronises the host.  Errors
 *   raised by the device after launch surface at the caller's next
 *   synchronisation, or through gemm_poll_device_error().
 * - The call runs on the calling thread's current CUDA device, which must be
 *   a compute-capability 10.3 GPU (GB300).  There is no CPU fallback: any
 *   unsupported case returns an error code and computes nothing.
 * - M == 0 or N == 0: no-op, returns PTC_OK (pointers may be NULL).
 *   K == 0: C is filled with zeros (the empty sum), A and B are not read.
 * - Return value: PTC_OK (0) on success, else one of the PTC_ERR_* codes below.
 *   Arguments are checked in this order, before any CUDA call:
 *     PTC_ERR_INVALID  negative or too-large size (each of M, N, K must be
 *                      <= 2^30, and C must have fewer than 2^31 output tiles
 *                      of 128 x 256), NULL pointer where data is needed, a leading
 *                      dimension below its minimum or above 2^36 elements
 *                      (the operands' when K > 0, C's always), an odd INT4
 *                      leading dimension
 *     PTC_ERR_ALIGN    a base pointer not 16-byte aligned, or a row pitch in
 *                      bytes that is not a multiple of 16
 *     PTC_ERR_OVERLAP  C's byte range intersects A's or B's
 *   and then, at execution:
 *     PTC_ERR_DEVICE   no current device, or it is not compute capability 10.3
 *     PTC_ERR_ALLOC    the stream-ordered workspace could not be obtained
 *     PTC_ERR_LAUNCH   a CUDA runtime or driver call failed (text available
 *                      from gemm_status_string(PTC_ERR_LAUNCH) on this thread)
 *     PTC_ERR_TIMEOUT  (device side, reported by gemm_poll_device_error) a
 *                      pipeline wait inside a kernel exceeded its time limit;
 *                      the kernel stopped early and C is incomplete
 */
#ifndef PTC_H
#define PTC_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PTC_OK 0
#define PTC_ERR_INVALID 1
#define PTC_ERR_ALIGN 2
#define PTC_ERR_OVERLAP 3
#define PTC_ERR_DEVICE 4
#define PTC_ERR_LAUNCH 5
#define PTC_ERR_TIMEOUT 6
#define PTC_ERR_ALLOC 7

/*
 * FP16 GEMM: C[M x N] (float32) = A[M x K] (binary16) . B[K x N] (binary16),
 * products accumulated in FP32 on the tensor cores.
 *   A  row-major, element (i,k) at A[i*lda + k]; lda >= K, lda % 8 == 0
 *   B  row-major, element (k,j) at B[k*ldb + j]; ldb >= N, ldb % 8 == 0
 *      (the paper's FP16 kernels load B with ldmatrix .trans, Table VI)
 *   C  row-major, element (i,j) at C[i*ldc + j]; ldc >= N, ldc % 4 == 0
 * Accuracy: each element is the FP32 tensor-core sum of exact products; it is
 * not bitwise reproducible against a sequential sum.
 */
int gemm_f16(int64_t M, int64_t N, int64_t K,
             const void *A, int64_t lda,
             const void *B, int64_t ldb,
             float *C, int64_t ldc,
             void *stream);

/*
 * FP16 GEMM with FP16 accumulators: C[M x N] (binary16) = A . B, the tensor
 * cores accumulating in binary16 (the paper's fp16_ptx_fp16acc variant,
 * section IV-A and Table VI: f16 accumulators instead of f32).  A and B as
 * gemm_f16; C row-major binary16 with ldc >= N and ldc % 8 == 0.  Each output
 * is the binary16 running sum of the products, so its error grows with K:
 * the bound the tests use is |C - sum| <= (ceil(K/16) + 1) * 2^-10 *
 * sum_k |A_ik B_kj| + ceil(K/16) * 2^-24.  Values beyond the binary16 range
 * become infinities.
 */
int gemm_f16_f16acc(int64_t M, int64_t N, int64_t K,
                    const void *A, int64_t lda,
                    const void *B, int64_t ldb,
                    void *C, int64_t ldc,
                    void *stream);

/*
 * INT8 GEMM: C[M x N] (int32) = A[M x K] (int8) . B[K x N] (int8), exact.
 *   A  row-major,    element (i,k) at A[i*lda + k]; lda >= K, lda % 16 == 0
 *   B  column-major, element (k,j) at B[j*ldb + k]; ldb >= K, ldb % 16 == 0
 *      (K-contiguous "non-transposed" B of the paper's .row.col MMAs;
 *      section IV-D shows a transposed B collapses coalescing)
 *   C  row-major, element (i,j) at C[i*ldc + j];    ldc >= N, ldc % 4 == 0
 * Result: bit-exact sum_k A_ik B_kj, wrapped modulo 2^32 if it leaves the
 * int32 range (unreachable for K <= 131072).
 * A and B are first converted into a stream-ordered device workspace of about
 * 2*(M+N)*K bytes, taken from and returned to a library-owned memory pool on
 * `stream`; small products (one wave of one-CTA tiles with few K blocks each)
 * instead convert each K block inside the GEMM kernel's shared memory and use
 * no workspace (tuning key "in_ring").
 */
int gemm_s8(int64_t M, int64_t N, int64_t K,
            const int8_t *A, int64_t lda,
            const int8_t *B, int64_t ldb,
            int32_t *C, int64_t ldc,
            void *stream);

/*
 * INT8 GEMM with B row-major: as gemm_s8, except
 *   B  row-major (K x N), element (k,j) at B[k*ldb + j]; ldb >= N, ldb % 16 == 0
 * The paper's ablation of a transposed B ("Hand-Written PTX Tensor-Core GEMM
 * Kernels: A Multi-Precision Study on NVIDIA L4", section IV-D) found this
 * orientation far slower for its cp.async / ldmatrix kernel; here B is
 * converted into K rows of N binary16 values and read by the tensor cores as
 * an MN-major operand (the layout gemm_f16 reads), so the orientation costs
 * only the conversion of a differently shaped B.  Workspace: about
 * 2*(M*K + K*N) bytes from the library pool, stream-ordered on `stream`.
 */
int gemm_s8_b_rowmajor(int64_t M, int64_t N, int64_t K,
                       const int8_t *A, int64_t lda,
                       const int8_t *B, int64_t ldb,
                       int32_t *C, int64_t ldc,
                       void *stream);

/*
 * Packed INT4 GEMM: C[M x N] (int32) = A[M x K] (s4) . B[K x N] (s4), exact.
 * Two signed 4-bit values per byte, element 2t of a row in bits 0..3 of byte
 * t and element 2t+1 in bits 4..7 (low nibble = even k); Listing 1 addresses
 * A's byte (row, k) at row*(K/2) + k/2.
 *   A  row-major,    element (i,k) in byte A[i*lda/2 + k/2]; lda >= K,
 *                    lda even, lda % 32 == 0 (16-byte row pitch)
 *   B  column-major, element (k,j) in byte B[j*ldb/2 + k/2]; ldb >= K,
 *                    ldb even, ldb % 32 == 0
 *   C  row-major int32, ldc >= N, ldc % 4 == 0
 * Odd K is allowed: the high nibble of a row's last byte is then ignored.
 * Result: bit-exact sum_k A_ik B_kj (|C| <= 64*K, no overflow for K < 2^25).
 * Uses a stream-ordered device workspace of about (M+N)*K bytes, or converts
 * inside the GEMM kernel, as gemm_s8 (in-kernel conversion needs an even K).
 */
int gemm_s4(int64_t M, int64_t N, int64_t K,
            const void *A, int64_t lda,
            const void *B, int64_t ldb,
            int32_t *C, int64_t ldc,
            void *stream);

/*
 * Integer GEMM with a dequantising epilogue.  The paper leaves scaling out of
 * its kernels ("INT32 accumulations without in-kernel dequantization or
 * scaling", section VI "Scope"); this is the per-channel-scaled form such
 * INT8 / INT4 products take in quantised LLM inference (section V), built on
 * the same exact integer sums:
 *
 *   acc[i][j] = sum_k A_ik B_kj                (exact, wrapped to int32)
 *   C[i][j]   = out( rn(rn(rn(float(acc)) * scale_a[i]) * scale_b[j]) )
 *
 * in FP32 with round-to-nearest-even at each step, in that order and without
 * fused multiply-add, then rounded to nearest-even into the output type
 * (PTC_OUT_F32: no further rounding).  scale_a (M floats) and scale_b
 * (N floats) are device pointers, 4-byte aligned; NULL means all ones.
 * K == 0 writes +0 everywhere.  A, B, lda, ldb as gemm_s8 (INT8) and gemm_s4
 * (packed INT4, nibbles); C row-major with ldc >= N elements of the output
 * type and a row pitch that is a multiple of 16 bytes.  Errors as gemm_s8,
 * plus PTC_ERR_INVALID for an unknown out_type and PTC_ERR_OVERLAP when C
 * overlaps a scale vector.
 */
#define PTC_OUT_F32 0
#define PTC_OUT_BF16 1
#define PTC_OUT_F16 2

int gemm_s8_scaled(int64_t M, int64_t N, int64_t K,
                   const int8_t *A, int64_t lda,
                   const int8_t *B, int64_t ldb,
                   const float *scale_a, const float *scale_b,
                   void *C, int64_t ldc, int out_type,
                   void *stream);

int gemm_s4_scaled(int64_t M, int64_t N, int64_t K,
                   const void *A, int64_t lda,
                   const void *B, int64_t ldb,
                   const float *scale_a, const float *scale_b,
                   void *C, int64_t ldc, int out_type,
                   void *stream);

/*
 * gemm_s8 without any memory allocation.  The paper has no counterpart: it is
 * an addition for callers that cannot let a library allocate device memory,
 * such as an application whose own allocator has reserved the GPU's memory
 * and forbids other allocations, or a latency-bound path where an allocation
 * could block or fail at an arbitrary moment.
 * Same arguments, layouts, result and errors as gemm_s8; the binary16
 * workspace lives in a fixed 32 MiB array in the library's device image
 * (held on every GPU that loads the library until the process exits) instead
 * of the memory pool.  The workspace must fit:
 *     (M + N) * roundup(K, 64) * 2 bytes <= 32 MiB   (e.g. M = N = K = 2048),
 * otherwise the call returns PTC_ERR_INVALID and launches nothing.
 * The first call on each device (with that device current) looks up the
 * array's device address with cudaGetSymbolAddress; make it before any stream
 * capture begins.  Under CUDA's default lazy module loading that first lookup
 * also loads the library's device code and commits the array's 32 MiB on the
 * GPU, so make the first call (or set CUDA_MODULE_LOADING=EAGER) before the
 * application's own allocator reserves the device's memory; later calls
 * allocate nothing.  If that set-up fails the call returns PTC_ERR_DEVICE and
 * the next call tries it again.  Every call uses the same array: calls whose
 * kernels overlap on the GPU (other streams, other host threads) race on it
 * and give wrong results, so serialise them.
 */
int gemm_s8_noalloc(int64_t M, int64_t N, int64_t K,
                    const int8_t *A, int64_t lda,
                    const int8_t *B, int64_t ldb,
                    int32_t *C, int64_t ldc,
                    void *stream);

/*
 * The same three products with HOST-resident operands and result: A, B and C
 * are host pointers (pinned memory from cudaHostAlloc / cudaHostRegister gives
 * asynchronous copies; pageable memory works but its copies are staged
 * synchronously by the driver).  Layouts, leading dimensions and errors as
 * gemm_f16 / gemm_s8 / gemm_s4 (host pointers must also be 16-byte aligned).
 * Asynchronous on `stream`: the call enqueues the work and returns; A and B
 * must stay unchanged and C unread until `stream` has completed.  The work is
 * pipelined over row panels of 2048 rows once M >= 8192: B and the A panels
 * are copied to the device on a library-owned stream, each panel's kernels
 * run on `stream` as soon as its operands arrived, and each C panel is copied
 * back on a second library-owned stream as soon as it is done, so the two
 * copy directions and the tensor cores work at the same time.  All of it is
 * ordered after the work already queued on `stream`, and `stream` waits for
 * the last copy.  Device buffers come from the library's stream-ordered pool.
 * The paper has no counterpart (its matrices are device-resident).
 */
int gemm_f16_host(int64_t M, int64_t N, int64_t K,
                  const void *A, int64_t lda,
                  const void *B, int64_t ldb,
                  float *C, int64_t ldc,
                  void *stream);

int gemm_s8_host(int64_t M, int64_t N, int64_t K,
                 const int8_t *A, int64_t lda,
                 const int8_t *B, int64_t ldb,
                 int32_t *C, int64_t ldc,
                 void *stream);

int gemm_s4_host(int64_t M, int64_t N, int64_t K,
                 const void *A, int64_t lda,
                 const void *B, int64_t ldb,
                 int32_t *C, int64_t ldc,
                 void *stream);

/*
 * The paper's own kernel families on GB300, as same-precision baselines for
 * its speedup definitions (section III-A, III-B: every PTX kernel is compared
 * with the WMMA kernel of its precision, and quantised kernels with the FP16
 * WMMA kernel).  Eight warps per block, 16 x 16 warp tiles (block tile
 * 32 x 64), two cp.async stages, then:
 *   PTC_BASELINE_F16_WMMA  WMMA m16n16k16, FP16 -> FP32      (fp16_wmma)
 *   PTC_BASELINE_F16_MMA   mma.sync m16n8k16, FP16 -> FP32   (fp16_ptx_mma)
 *   PTC_BASELINE_S8_WMMA   WMMA m16n16k16, s8 -> s32         (int8_wmma)
 *   PTC_BASELINE_S8_MMA    mma.sync m16n8k32, s8 -> s32      (int8_ptx_mma_k32)
 *   PTC_BASELINE_S4_WMMA   WMMA m8n8k32, s4 -> s32           (int4_wmma)
 *   PTC_BASELINE_S4_MMA    mma.sync m16n8k64, s4 -> s32      (int4_ptx_mma_k64)
 *   PTC_BASELINE_F16_LDMATRIX, PTC_BASELINE_S8_LDMATRIX, PTC_BASELINE_S4_LDMATRIX
 *                          the three mma.sync kernels with their fragments
 *                          loaded by ldmatrix (A: .x4, B: .x2; FP16 B with
 *                          .trans), the fragment path of the paper's fastest
 *                          INT8 / INT4 kernels (Table VI, Listing 2); the
 *                          *_MMA variants pack fragments from scalar 32-bit
 *                          shared loads (the paper's manual-pack family)
 * Operands and C have the layouts of gemm_f16 / gemm_s8 / gemm_s4 (C FP32 for
 * the FP16 variants, int32 otherwise).  Restrictions of these simple kernels:
 * M % 32 == 0, N % 64 == 0, K a positive multiple of 32 (FP16), 64 (INT8) or
 * 128 (INT4); C 32-byte aligned with ldc % 8 == 0.  They are comparison
 * points, not the fast path; integer results are exact, FP16 results are FP32
 * tensor-core sums.
 */
#define PTC_BASELINE_F16_WMMA 0
#define PTC_BASELINE_F16_MMA 1
#define PTC_BASELINE_S8_WMMA 2
#define PTC_BASELINE_S8_MMA 3
#define PTC_BASELINE_S4_WMMA 4
#define PTC_BASELINE_S4_MMA 5
#define PTC_BASELINE_F16_LDMATRIX 6
#define PTC_BASELINE_S8_LDMATRIX 7
#define PTC_BASELINE_S4_LDMATRIX 8

int gemm_baseline(int variant, int64_t M, int64_t N, int64_t K,
                  const void *A, int64_t lda,
                  const void *B, int64_t ldb,
                  void *C, int64_t ldc,
                  void *stream);

/* Human-readable text of a status code.  For PTC_ERR_LAUNCH the text of the
 * failing CUDA call on the calling thread is appended.  Never NULL; the
 * string stays valid until the next call on the same thread. */
const char *gemm_status_string(int status);

/* Reads and clears the device-side error word of the current device that the
 * GEMM kernels set when a pipeline wait times out.  Synchronises the device.
 * Returns PTC_OK when no kernel reported an error, PTC_ERR_TIMEOUT when one
 * did, PTC_ERR_DEVICE / PTC_ERR_LAUNCH when the device cannot be queried. */
int gemm_poll_device_error(void);

/* Number of kernels this library has launched in this process (all devices,
 * all threads).  Lets callers count the GPU work behind a sequence of calls. */
uint64_t ptc_kernel_launch_count(void);

/* Clock record of the GEMM kernels (tuning key "clock_probe" = 1 turns it on):
 * thread 0 of every CTA of a GEMM kernel launched while it is on adds the SM
 * clock cycles (%clock64) and the global-timer nanoseconds between its start
 * of work and its exit, and 1, to the record of its kernel family, so that
 * cycles / ns is the mean SM clock (GHz) the tensor-core kernels ran at.
 * Families: [0] FP16 operands (gemm_f16, gemm_f16_f16acc), [1] the INT8
 * route, [2] the INT4 route.  Fills cycles[3], ns[3], ctas[3] for the current
 * device, then clears the record.  Synchronises the device.  The timing
 * methodology of the study (wall-clock times of repeated launches, section
 * III-B of "Hand-Written PTX Tensor-Core GEMM Kernels: A Multi-Precision Study
 * on NVIDIA L4") leaves the clock implicit; this makes it explicit.  Returns
 * PTC_OK, PTC_ERR_INVALID for a NULL pointer, PTC_ERR_DEVICE, or
 * PTC_ERR_LAUNCH. */
int ptc_clock_probe_read(uint64_t *cycles, uint64_t *ns, uint64_t *ctas);

/* Test hook, not for production use.  Sets the pipeline-wait time limit (in
 * nanoseconds, 0 restores the default of one second) and, when stall_tile >= 0,
 * makes the next launched GEMM kernel withhold the operands of output tile
 * `stall_tile`, so that the wait for them runs out and the kernel reports
 * PTC_ERR_TIMEOUT through gemm_poll_device_error().  stall_tile = -2 makes the
 * converter warps of the next integer launch with conversion in the GEMM
 * kernel (tuning key "conv_fused") withhold the first piece they would
 * convert, so that the producers waiting for it run out.  The stall applies to
 * one launch only.  Returns PTC_OK. */
int ptc_debug_set_wait_limit(uint64_t timeout_ns, int64_t stall_tile);

/* The launch shape the library would choose for an M x N x K product of
 * precision `prec` (0 FP16, 1 INT8, 2 INT4; 4-byte C) on a device with `sms`
 * SMs on which cap2 / cap4 / cap8 thread-block clusters of 2 / 4 / 8 one-CTA
 * tiles fit at once, under the current tuning knobs: *ctas = 1 or 2 (CTA
 * pairs on 256 x 256 tiles), *tile_n = output columns per tile (256, 128,
 * 64), *ksplit = CTAs sharing one tile's K range (1 = none), and, when
 * in_ring is not NULL, *in_ring = 1 if the integer operands would be
 * converted inside the GEMM kernel (0: a separate pass, or FP16).  Host-only
 * arithmetic (no device is touched), for inspecting and testing the
 * automatic choice.  Returns PTC_OK, or PTC_ERR_INVALID for a NULL pointer
 * (other than in_ring) or an argument out of range (sizes must be positive). */
int ptc_plan_shape(int64_t M, int64_t N, int64_t K, int prec, int sms, int cap2, int cap4, int cap8, int *ctas,
                   int *tile_n, int *ksplit, int *in_ring);

/* Launch shape of the last GEMM kernel the calling thread launched through
 * this library: *grid = CTAs launched, *cluster = CTAs per thread-block
 * cluster (1; 2 for CTA pairs; KS for K-split clusters), *ksplit = CTAs that
 * share one output tile's K range (1 when the tiles are not split that way),
 * *tile_n = output columns per tile (256, or 128 / 64 for narrow one-CTA
 * tiles).  All zero before the first launch.  Host-side only (no device
 * work).  Returns PTC_OK, or PTC_ERR_INVALID when a pointer is NULL. */
int ptc_last_launch(int *grid, int *cluster, int *ksplit, int *tile_n);

/* Operand conversion of the calling thread's last GEMM call through this
 * library: *mode = 0 none (FP16 operands, a call that launched nothing, or no
 * call yet), 1 a separate conversion pass into a workspace, 2 conversion
 * inside the GEMM kernel's shared memory, 3 conversion into the workspace by
 * the GEMM kernel's converter warps (tuning key "conv_fused").  Host-side
 * only.  Returns PTC_OK,
 * or PTC_ERR_INVALID when the pointer is NULL. */
int ptc_last_conversion(int *mode);

/* Tuning and test knobs, process-wide.  Returns PTC_OK, or PTC_ERR_INVALID for
 * an unknown key or a value out of range.  Keys:
 *   "group_m"      output-tile rows per raster group of the persistent
 *                  scheduler (L2 reuse), default 8
 *   "s8_chunk_kb"  INT8 route: K blocks (64 values each) whose FP32 partial
 *                  sum is folded into int32 at a time, default 16 (1024
 *                  values: |partial| <= 2^24, so every FP32 partial sum is an
 *                  exactly representable integer); at most 16
 *   "s4_chunk_kb"  INT4 route: K blocks (128 values each) per fold, default 64
 *                  (8192 values: |partial| <= 2^19); at most 2048 (2^24)
 *                  Both fold lengths must be even (CTA pairs stage two K
 *                  blocks at a time); odd values, and values above the
 *                  exactness limits (which could let an FP32 partial sum
 *                  round), return PTC_ERR_INVALID.
 *   "l2_hint"      L2 eviction policy of operand loads: 0 (default) none;
 *                  1 A evict-last / B evict-first; 2 A evict-last; 3 both
 *                  evict-normal (all measured slower than 0 on GB300)
 *   "cta_pair"     0 (default): clusters of two CTAs sharing 256 x 256
 *                  tiles (tcgen05 cta_group::2) once 128 x 256 one-CTA tiles
 *                  would fill the SMs, and for FP16 whole 128 x 256 tiles
 *                  from 32 one-CTA tiles up; otherwise one CTA per tile (see
 *                  "tile_n" and "ksplit" for the shapes of small products);
 *                  1: always one CTA per 128 x 256 tile; 2: always CTA
 *                  pairs.  Results do not depend on the choice except
 *                  through the FP16 summation order.
 *   "tail_split"   1 (default): when K spans enough K blocks (see
 *                  "split_min_kb") and the last wave of output tiles would
 *                  occupy at most half of the CTAs (or CTA pairs), each tile
 *                  of that wave runs as two units over the two halves of K on
 *                  two CTAs (or pairs), whose partial sums are added (see
 *                  "split_reduce"), so that the tail takes about half the
 *                  time.  The workspace (flags, or up to ~20 MB of partial
 *                  sums) is stream-ordered from the library pool.  0: never.
 *                  Integer results do not depend on the choice; FP16 results
 *                  of split tiles differ by the summation order (the sum of
 *                  two FP32 half sums).
 *   "split_reduce" 1 (default): a split tile of FP32 or int32 C is zeroed
 *                  by its first half's CTAs when the kernel starts and both
 *                  halves add their partial sums into it by TMA reductions
 *                  (in FP32, 0 + a + b: the same bits in either order); only
 *                  a flag per epilogue warp slice is kept in the workspace.
 *                  0: the halves exchange partial sums through the
 *                  workspace and one of them writes C (always the case for
 *                  FP16 C and the scaled outputs).
 *   "pair_stage_kb" CTA pairs: K blocks per shared-memory ring stage, 2
 *                  (default: 3 stages of 64 KiB per CTA) or 1 (7 stages of
 *                  32 KiB).  Results do not depend on the choice.
 *   "split_min_kb" K blocks (64 values FP16 / INT8, 128 INT4) below which no
 *                  tile is split, default 64; doubled for INT4 and for
 *                  tiles whose halves exchange partial sums (split_reduce 0,
 *                  FP16 C, scaled outputs), as measured: the split saves
 *                  about half a tile's K loop and costs ~4 us per call with
 *                  TMA reductions, ~10 us with the exchange; 2 or more.
 *   "ksplit"       small problems: when 128 x 256 one-CTA tiles would fill at
 *                  most half of the SMs in one wave, each tile runs on a
 *                  thread-block cluster of KS CTAs that share its K blocks
 *                  (about 1/KS each) and add their partial sums through
 *                  distributed shared memory, in rank order.  0 (default):
 *                  the largest KS of 8, 4, 2 whose clusters fit one wave with
 *                  at least one K block per CTA; 2, 4 or 8: only that KS
 *                  (one CTA per tile when it does not fit); 1: never (the
 *                  "cta_pair" rule decides alone).  Integer results do not
 *                  depend on the choice; FP16 results differ by the summation
 *                  order (a rank-ordered sum of KS FP32 partial sums), and
 *                  FP16-accumulator results are rounded to binary16 once,
 *                  from that FP32 sum.  No workspace is used.
 *   "tile_n"       output tile width: 0 (default) chooses by size; 64 or
 *                  128: one CTA per 128 x 64 / 128 x 128 tile; 256: only
 *                  128 x 256 one-CTA tiles (with or without K-split
 *                  clusters) and 256 x 256 CTA-pair tiles.
 *                  By size, a product whose 128 x 256 tiles would occupy
 *                  fewer CTAs than there are SMs (one wave) takes, among
 *                  narrow tiles that still fit one wave, K-split clusters and
 *                  whole 128 x 256 tiles, the shape with the least estimated
 *                  time: each SM writes C to L2 at ~32 bytes per clock, so
 *                  narrow tiles spread a small product's output over more
 *                  SMs.  Results do not depend on the choice.
 *   "pdl"          1 (default): kernels are launched with programmatic
 *                  stream serialization, so that a kernel can start (set up
 *                  barriers and tensor memory) while the previous kernel of
 *                  the stream finishes; it waits for that kernel before its
 *                  first global-memory access.  0: plain stream order.
 *   "pair_in_ring" gemm_s8 / gemm_s4 on CTA pairs (products whose 128 x 256
 *                  tiles would fill the SMs): 0 (default) converts the
 *                  operands in a separate pass; 2 converts each K block of the
 *                  raw operands inside the pair kernel, by six dedicated
 *                  converter warps per CTA.  Measured on GB300 at N = 8192,
 *                  the in-kernel route is ~3x slower (the conversion and the
 *                  proxy fence that publishes each converted block take
 *                  longer than the block's MMAs), so it is not the default.
 *                  Results do not depend on the choice.
 *   "conv_fused"   gemm_s8 / gemm_s4 (and their scaled forms) on 256-wide tiles
 *                  without a K split that would use the separate conversion
 *                  pass: 0 (default) keeps the pass; 1 converts the operands
 *                  into the same workspace inside the GEMM kernel, by six
 *                  converter warps per CTA (16-warp CTAs; CTAs without a tile
 *                  convert too), panel slice by panel slice in the order the
 *                  tiles need them, each slice loaded once its counter holds
 *                  all its pieces.  Measured on GB300 it is slower than the
 *                  pass (N = 8192: INT8 673 against 625 us, INT4 392 against
 *                  325 us; N = 2048: 31 against 21 us): the converter warps'
 *                  loads in flight limit their rate, and their HBM traffic
 *                  slows the GEMM's operand loads.  Results do not depend on
 *                  the choice.
 *   "multicast"    CTA-pair products (256 x 256 tiles): 0 (default) one pair
 *                  per thread-block cluster; 1 two pairs per cluster of four
 *                  CTAs, computing adjacent tile columns of one tile row and
 *                  sharing A by TMA multicast (each CTA loads half of its 128
 *                  A rows into its own shared memory and its counterpart's in
 *                  the other pair), which cuts the operand bytes the SMs read
 *                  from L2 by a quarter (not the bytes each SM receives).
 *                  Clusters of four fit 144 of the 152 SMs, and the
 *                  last-wave K split is not used.  Measured on GB300 it is
 *                  no faster (N = 8192: FP16 +3.9%, INT8 +2.2%, INT4 -1.0%
 *                  time; N = 4096 and 6144 within +-4%), so it is off by
 *                  default.  The in-kernel pair conversion ("pair_in_ring" 2)
 *                  keeps one pair per cluster.  Results do not depend on the
 *                  choice.
 *   "clock_probe"  0 (default) or 1: GEMM kernels add their SM cycles and
 *                  nanoseconds to the clock record (ptc_clock_probe_read)
 *   "in_ring"      gemm_s8 / gemm_s4 (and their scaled forms) on one-CTA
 *                  shapes may load K blocks of the raw operands and convert
 *                  them to the MMA input type in the GEMM kernel's shared
 *                  memory (the epilogue warps, idle during the K loop, do
 *                  it), with no workspace and no separate kernel.  1
 *                  (default): where estimated faster than a separate pass
 *                  (single-wave launches with few K blocks per CTA: small
 *                  products such as N = 512); 0: never; 2: on every one-CTA
 *                  shape.  Results do not depend on the choice.
 * No accepted value of any key changes an INT8 or INT4 result. */
int ptc_set_tuning(const char *key, int64_t value);

#ifdef __cplusplus
}
#endif

#endif /* PTC_H */
