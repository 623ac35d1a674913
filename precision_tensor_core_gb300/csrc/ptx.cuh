// ptx.cuh -- sm_103a device primitives written as inline PTX: mbarriers with
// bounded waits, TMA tiled loads, tensor-memory allocation, tcgen05 MMA,
// commit and tensor-memory loads, and the shared-memory matrix / instruction
// descriptors the MMA consumes.
//
// These replace the SM89 primitives of "Hand-Written PTX Tensor-Core GEMM
// Kernels: A Multi-Precision Study on NVIDIA L4": cp.async 16-byte copies with
// commit_group/wait_group (section II-B, Listing 1) become TMA bulk tensor
// copies completing on mbarriers; ldmatrix fragment loads (Listing 2) vanish
// because tcgen05.mma reads its operands straight from shared memory through
// descriptors; register accumulators become tensor-memory columns.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace ptc {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint64_t sm_clock64() {
    uint64_t c;
    asm volatile("mov.u64 %0, %%clock64;" : "=l"(c));
    return c;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Makes barrier initialisation visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Error word codes written by kernels (match PTC_ERR_TIMEOUT in ptc.h).
constexpr uint32_t kErrTimeout = 6;

// Shared abort state of one CTA.
struct AbortState {
    volatile uint32_t flag;  // nonzero once any role of this CTA gave up
};

// Waits until the phase with the given parity of `bar` has completed.
// Returns false (without waiting further) when this CTA was told to abort, or
// when `limit_ns` elapsed; in the latter case it raises the CTA's abort flag
// and records kErrTimeout in `err_word`.  With ab == nullptr (used while
// draining after an abort) neither the flag nor the error word is touched.
// Never spins unbounded.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, AbortState *ab,
                                          uint32_t *err_word, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 15u) == 0) {
            if (ab != nullptr && ab->flag) return false;
            if (globaltimer_ns() - t0 > limit_ns) {
                if (ab != nullptr) {
                    ab->flag = 1;
                    atomicCAS(err_word, 0u, kErrTimeout);
                }
                return false;
            }
        }
    }
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled bulk tensor load global -> shared, completion signalled on `bar`
// as transaction bytes.  x is the innermost (contiguous) coordinate.
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, uint64_t *bar,
                                            int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// ---------------------------------------------------------------- TMA stores
// Generic-proxy writes to shared memory made visible to the async proxy
// (the TMA engine, the tensor cores) before a bulk copy or an MMA reads them.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t saddr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(saddr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void st_shared_v4(uint32_t saddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(saddr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// 2-D tiled bulk tensor store shared -> global of one box at (x, y); elements
// of the box outside the tensor are not written.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t smem_src, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_src), "r"(x), "r"(y)
                 : "memory");
}

// TMA reduction of a 2-D box from shared memory into global memory: each
// element of the box is added (in the tensor map's element type: FP32 with
// round-to-nearest-even, or 32-bit integers modulo 2^32) to the global
// element at (x + i, y + j); elements outside the tensor are skipped.
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap *map, uint32_t smem_src, int32_t x, int32_t y) {
    asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(smem_src), "r"(x), "r"(y)
                 : "memory");
}

// Orders this thread's view of global memory written through the generic
// proxy (ordinary stores, here made visible to it by an acquire) before its
// later asynchronous-proxy (TMA) accesses of global memory.
// Orders this thread's generic-proxy writes (any state space) before later
// async-proxy accesses: used before a CTA pair's tensor cores read shared
// memory that threads of either CTA wrote.
__device__ __forceinline__ void fence_proxy_async_all() {
    asm volatile("fence.proxy.async;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until the source shared memory of every committed bulk store has been read.
__device__ __forceinline__ void bulk_wait_group_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Wait until every committed bulk store has completed.
__device__ __forceinline__ void bulk_wait_group0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ---------------------------------------------------------------- clusters
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address, in the shared::cluster window, of the variable at shared::cta
// address `saddr` in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

// All threads of all CTAs of the cluster.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                     "memory");
}

// The two halves of cluster_sync, for work between them (every thread of
// the cluster arrives once, then waits).
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 16 bytes from shared::cluster address `addr` (this CTA's or a peer's).
__device__ __forceinline__ uint4 ld_shared_cluster_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// Arrive on an mbarrier given by its shared::cluster address (own or peer CTA).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}

// 2-D tiled TMA load multicast into the shared memory of every CTA of
// `cta_mask` (same offset in each) in a cluster of CTA pairs: the completion
// of each destination's copy is signalled on the mbarrier at the offset of
// `bar_cluster_addr` in the even CTA of that destination's pair (measured on
// GB300: each pair leader's barrier received exactly its pair's bytes).
__device__ __forceinline__ void tma_load_2d_pair_mc(void *smem_dst, const CUtensorMap *map,
                                                    uint32_t bar_cluster_addr, int32_t x, int32_t y,
                                                    uint16_t cta_mask) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
        ".cta_group::2 [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster_addr), "h"(cta_mask)
        : "memory");
}

// 2-D tiled TMA load into this CTA's shared memory whose completion is
// signalled on an mbarrier of either CTA of the pair (shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void *smem_dst, const CUtensorMap *map,
                                                 uint32_t bar_cluster_addr, int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster_addr)
        : "memory");
}

// ---------------------------------------------------------------- dependent launches
// A kernel launched with programmatic stream serialization may start while
// the kernel before it in the stream is still running: griddep_wait blocks
// until that kernel has completed and its memory operations are visible, so
// every global-memory access of the kernel comes after it.  Without a
// programmatic predecessor it returns at once.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Lets the next kernel in the stream (if launched programmatically) start
// once every CTA of this grid has called this or exited; it still waits for
// this grid's completion before touching memory.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- L2 policies
// 64-bit L2 cache policies for the .L2::cache_hint operand of bulk copies.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// As tma_load_2d / tma_load_2d_pair, with an L2 eviction policy.
__device__ __forceinline__ void tma_load_2d_hint(void *smem_dst, const CUtensorMap *map, uint64_t *bar,
                                                 int32_t x, int32_t y, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d_pair_hint(void *smem_dst, const CUtensorMap *map,
                                                      uint32_t bar_cluster_addr, int32_t x, int32_t y,
                                                      uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster_addr), "l"(policy)
        : "memory");
}

// ---------------------------------------------------------------- tcgen05
// CTAS = 1: one CTA owns its tensor memory and issues its own MMAs.
// CTAS = 2: a CTA pair; allocation is collective over one warp of each CTA,
// MMAs issued by the even CTA read operands from both CTAs' shared memory and
// write accumulators into both CTAs' tensor memory.
//
// Tensor-memory allocation: executed by one full warp (of each CTA of the
// group).  The base address (lane 0, first column) is written to shared memory.
template <int CTAS>
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
    if constexpr (CTAS == 1)
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(dst)),
                     "r"(ncols)
                     : "memory");
    else
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(dst)),
                     "r"(ncols)
                     : "memory");
}

template <int CTAS>
__device__ __forceinline__ void tmem_relinquish() {
    if constexpr (CTAS == 1)
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    else
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

template <int CTAS>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    if constexpr (CTAS == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                     : "memory");
    else
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                     : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] . B[smem desc], FP16 operands (KIND_F8 = false) or
// E4M3 operands (KIND_F8 = true, kind::f8f6f4), FP32 accumulators.
template <int CTAS, bool KIND_F8>
__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                    uint32_t idesc, uint32_t accumulate) {
#define PTC_MMA(GROUP, KINDS)                                                              \
    asm volatile(                                                                          \
        "{\n\t.reg .pred p;\n\t"                                                       \
        "setp.ne.b32 p, %4, 0;\n\t"                                                      \
        "tcgen05.mma.cta_group::" GROUP ".kind::" KINDS " [%0], %1, %2, %3, p;\n\t}" ::"r"( \
            d_tmem),                                                                       \
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)                              \
        : "memory")
    if constexpr (CTAS == 1 && !KIND_F8)
        PTC_MMA("1", "f16");
    else if constexpr (CTAS == 1 && KIND_F8)
        PTC_MMA("1", "f8f6f4");
    else if constexpr (CTAS == 2 && !KIND_F8)
        PTC_MMA("2", "f16");
    else
        PTC_MMA("2", "f8f6f4");
#undef PTC_MMA
}

// Arrives once on `bar` (this CTA) when every tcgen05 operation issued so far
// by this thread has completed.
template <int CTAS>
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    if constexpr (CTAS == 1)
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                smem_u32(bar))
            : "memory");
    else
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                smem_u32(bar))
            : "memory");
}

// CTA pair: arrives once on the mbarrier at the same shared-memory offset in
// every CTA of `cta_mask` when this thread's tcgen05 operations completed.
__device__ __forceinline__ void mma_commit_pair(uint64_t *bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

// Loads 32 consecutive 32-bit columns of one tensor-memory lane per thread
// (warp w % 4 may address lanes 32*(w%4) .. +31 only).
__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// Loads 16 consecutive 32-bit columns of one tensor-memory lane per thread.
__device__ __forceinline__ void tmem_ld_16cols(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- registers
// Per-warpgroup register budget (all four warps of the warpgroup execute the
// same instruction): .dec returns registers to the CTA's pool, .inc waits
// until the pool holds enough and takes them.  The budgets of the CTA's
// warpgroups must sum to at most the registers it was launched with.  ptxas
// allocates the code that an instruction dominates within its budget.
template <uint32_t N>
__device__ __forceinline__ void regs_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// ---------------------------------------------------------------- descriptors
// Shared-memory matrix descriptor (tcgen05 form):
//   bits  0-13  start address >> 4
//   bits 16-29  leading-dimension byte offset >> 4
//   bits 32-45  stride-dimension byte offset >> 4
//   bits 46-47  descriptor version (1 for tcgen05)
//   bits 49-51  base offset (0: swizzle atoms are 1024-byte aligned)
//   bit  52     leading-dimension mode (0: byte offset)
//   bits 61-63  swizzle mode (2 = 128-byte swizzle)
// With the 128-byte swizzle a K-major operand is rows of 128 bytes, eight rows
// (one 1024-byte atom) apart by the stride offset; an MN-major operand is
// 64 two-byte elements of M/N per 128-byte row, K rows 128 bytes apart, 8-row
// groups `sbo` apart and 64-element M/N atoms `lbo` apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                    uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor for kind::f16 and kind::f8f6f4 (dense):
//   bits  4-5   D format (0 = F16, 1 = F32)
//   bits  7-9   A format, bits 10-12 B format (kind::f16: 0 = F16;
//               kind::f8f6f4: 0 = E4M3)
//   bit  15     A major (0 = K-major), bit 16 B major (1 = MN-major)
//   bits 17-22  N >> 3, bits 24-28 M >> 4
__host__ __device__ constexpr uint32_t instr_desc(uint32_t dfmt, uint32_t afmt, uint32_t bfmt, bool b_mn_major,
                                                  int m, int n) {
    return (dfmt << 4) | (afmt << 7) | (bfmt << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

}  // namespace ptc
