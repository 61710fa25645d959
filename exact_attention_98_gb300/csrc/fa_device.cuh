// Device primitives for sm_103a written as inline PTX: mbarriers with bounded
// waits, TMA tile loads, tensor-memory allocation, tcgen05 MMAs and
// tensor-memory loads/stores.  Everything the attention kernels need from the
// hardware goes through this file.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "exp2_poly_coeffs.h"

#if FA_EXP2_POLY_DEGREE != 3
#error "exp2_poly() evaluates a degree-3 polynomial; refit or update it"
#endif

namespace fa {

// ---------------------------------------------------------------------------
// Device status word (owned by the API translation unit and passed to every
// kernel by pointer).  A bounded wait that expires records FA_ERR_TIMEOUT (4)
// in the low byte and the wait-site code in bits 8..23; the first writer wins.
// ---------------------------------------------------------------------------
constexpr unsigned int kStatusTimeout = 4u;
// A correct kernel never waits this long on one pipeline event.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;
// Limit for the clean-up waits on the give-up path (copies and MMAs in flight).
constexpr unsigned long long kDrainLimitNs = 200000000ull;

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Where a CTA records a give-up: its shared abort flag and the global word.
struct WaitCtl {
  volatile int* abort_flag;  // shared memory, 0 = running
  unsigned int* status;      // global status word
};

__device__ __forceinline__ void record_status(unsigned int* status, unsigned int code,
                                              unsigned int site) {
  atomicCAS(status, 0u, code | (site << 8));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// The same test with acquire semantics at cluster scope: for a barrier that
// threads of the other CTA of a pair arrive on.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

template <bool kCluster>
__device__ __forceinline__ bool mbar_try_wait_scoped(uint32_t bar, uint32_t parity) {
  if constexpr (kCluster) return mbar_try_wait_cluster(bar, parity);
  else return mbar_try_wait(bar, parity);
}

// Waits for the phase with the given parity to complete.  Gives up when the
// CTA-wide abort flag is raised or after `limit_ns`; on expiry it records the
// site in the status word and raises the abort flag so that every other role
// of the CTA leaves its loop too.  Returns false when it gave up.  kCluster:
// acquire at cluster scope (arrivals from the other CTA of a pair).
template <bool kCluster = false>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const WaitCtl& ctl,
                                          unsigned int site,
                                          unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait_scoped<kCluster>(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_scoped<kCluster>(bar, parity)) return true;
    if ((it & 15u) == 0u) {
      if (*ctl.abort_flag) return false;
      if (globaltimer() - t0 > limit_ns) {
        *ctl.abort_flag = 1;
        record_status(ctl.status, kStatusTimeout, site);
        return false;
      }
    }
  }
}

// mbar_wait for a whole converged warp: every lane waits and the result is
// made warp-uniform, so that a warp whose lanes run the same loop (the MMA
// issuers, whose tcgen05 instructions are issued by one elected lane) stays
// converged even on the give-up path.
template <bool kCluster = false>
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, const WaitCtl& ctl,
                                               unsigned int site,
                                               unsigned long long limit_ns = kWaitLimitNs) {
  return __all_sync(0xffffffffu, mbar_wait<kCluster>(bar, parity, ctl, site, limit_ns));
}

// Clean-up wait on the give-up path: ignores the abort flag, bounded by
// kDrainLimitNs, records nothing.  Used to let this CTA's own TMA copies and
// MMAs finish before it frees tensor memory and exits.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kDrainLimitNs) return false;
  }
  return true;
}

// Programmatic dependent launch: blocks until the kernels this grid depends
// on (the stream's earlier work) have completed and their memory operations
// are visible.  Every kernel launched by launch_dependent() calls it before
// its first access to data that earlier work produces or may still read.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---------------------------------------------------------------------------
// CTA pairs: a cluster of two CTAs on one TPC that share each MMA
// (tcgen05 cta_group::2).  Rank 0 issues the MMAs; operands and accumulators
// live at the same shared- and tensor-memory addresses in both CTAs.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// The shared::cluster address of this CTA's shared-memory address `addr` in
// the CTA of the cluster with rank `rank`.
__device__ __forceinline__ uint32_t cluster_smem(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Every thread of both CTAs: release this CTA's prior writes, acquire the
// other's.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// Arrival on a barrier of the other CTA of a pair (shared::cluster address)
// with the default semantics of mbarrier.arrive (release at CTA scope), the
// form tcgen05 pipelines use to hand data a thread has finished writing
// (tensor memory after tcgen05.wait::st and tcgen05.fence::before_thread_sync,
// or shared memory after fence.proxy.async) to the CTA that issues the pair's
// MMAs.  In the pair backward, arrivals with a cluster-scope release
// (mbarrier.arrive.release.cluster) measured 600-1300 cycles each on the
// arriving warp, and the kernel 1.5x slower with them.
__device__ __forceinline__ void mbar_arrive_peer(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

// ---------------------------------------------------------------------------
// TMA (non-multicast tiled loads)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

// A tile into this CTA's shared memory whose completion is counted on a
// barrier of either CTA of the pair (cluster address `cluster_bar`).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t cluster_bar, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".cta_group::2 [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(cluster_bar)
      : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Bulk tensor reduction: adds a shared-memory tile into global memory (fp32
// add performed at L2), tracked by this thread's bulk-async group.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, uint32_t src, int c0,
                                                  int c1, int c2) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
      " [%0, {%2, %3, %4}], [%1];" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1,
                                             int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group"
      " [%0, {%2, %3, %4}], [%1];" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Waits until at most N of this thread's bulk groups are incomplete.
template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Named barrier over `count` threads (id 1..15; id 0 is __syncthreads).
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Named barrier that also returns the AND of `v` over its `count` threads, so
// that they go on (or leave a loop) together.
__device__ __forceinline__ bool named_bar_and(int id, int count, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}
// Arrival on a named barrier without waiting: how a warp that leaves a loop
// early releases the warps already waiting in that loop's bar.sync.
__device__ __forceinline__ void named_bar_arrive(int id, int count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (tensor core / TMA) reads of the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Tensor memory
// ---------------------------------------------------------------------------
// Executed by one whole warp.  Writes the allocated base address into smem.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

// Pair forms: one warp of each CTA of the pair executes them together; the
// same columns are allocated (freed) in both CTAs' tensor memory.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32-byte global store (one whole L2 sector per thread); `p` must be 32-byte
// aligned.
__device__ __forceinline__ void st_global_v8(void* p, uint32_t a0, uint32_t a1, uint32_t a2,
                                             uint32_t a3, uint32_t a4, uint32_t a5, uint32_t a6,
                                             uint32_t a7) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a0),
               "r"(a1), "r"(a2), "r"(a3), "r"(a4), "r"(a5), "r"(a6), "r"(a7)
               : "memory");
}

// TMEM address: lane in bits 31..16, column in bits 15..0.
__device__ __forceinline__ uint32_t tmem_addr(uint32_t base, uint32_t lane, uint32_t col) {
  return base + (lane << 16) + col;
}

// 32 lanes x 32 columns of 32 bit: thread t of the warp gets 32 consecutive
// columns of lane (warp's lane quarter + t).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// Waits for this thread's outstanding tcgen05.ld.  The registers are passed
// through the asm so that no use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait16(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 MMA (kind::f16, bf16 inputs, fp32 accumulator in tensor memory)
// ---------------------------------------------------------------------------
// Instruction descriptor: D fp32 (bits 4-5 = 1), A and B bf16 (bits 7-9 and
// 10-12 = 1), A/B major-ness (bit 15 / 16: 0 = K-major, 1 = MN-major),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn_major,
                                                      bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Instruction descriptor for tcgen05.mma kind::f8f6f4 with A and B both
// e4m3 (format 0 in bits 7-9 and 10-12) and an fp32 accumulator; the other
// fields as for kind::f16.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N, bool a_mn_major,
                                                      bool b_mn_major) {
  return (1u << 4) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand:
// start address >> 4 (bits 0-13), leading byte offset >> 4 (16-29), stride
// byte offset >> 4 (32-45), descriptor version 1 (46-47), swizzle mode
// 128B = 2 (61-63).  Base offset 0: every swizzle atom is 1024-byte aligned.
//   K-major operand:  rows of 128 B (64 bf16 along K), SBO = distance between
//                     groups of 8 rows; LBO unused.
//   MN-major operand: rows of 128 B (64 bf16 along M/N) per K index, SBO =
//                     distance between groups of 8 K indices, LBO = distance
//                     between 64-wide blocks along M/N.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}

// Shared-memory matrix descriptor for a K-major operand without swizzle:
// 8-row x 16-byte core matrices; LBO = distance between the two core
// matrices along K (one MMA's K = 16), SBO = distance between groups of 8
// rows.  Layout type 0.
__device__ __forceinline__ uint64_t sdesc_plain(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  return d;
}

// Every MMA and commit form below comes in two flavours.  kWarp = false: the
// calling thread issues it.  kWarp = true: a whole converged warp executes the
// call and elect.sync picks the one lane that issues it (the same lane every
// time, so its commits track its own MMAs); the warp's loop, waits and
// operand arithmetic then run as ordinary warp-uniform code.
#define FA_MMA_ASM(kWarp, INSTR, ...)                                                  \
  do {                                                                                 \
    if constexpr (kWarp)                                                               \
      asm volatile("{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\t"          \
                   "setp.ne.b32 p, %4, 0;\n\t@e " INSTR "\n\t}" ::__VA_ARGS__          \
                   : "memory");                                                        \
    else                                                                               \
      asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t" INSTR "\n\t}" ::__VA_ARGS__ \
                   : "memory");                                                        \
  } while (0)

// D[tmem] (+)= A[smem] * B[smem]
template <bool kWarp = false>
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  FA_MMA_ASM(kWarp, "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;", "r"(d_tmem),
             "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// D[tmem] (+)= A[tmem] * B[smem]
template <bool kWarp = false>
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  FA_MMA_ASM(kWarp, "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;", "r"(d_tmem),
             "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// Pair forms (cta_group::2, issued by rank 0): M = 256 rows, 128 from each
// CTA's A (shared or tensor memory at the same address in both) into each
// CTA's D; B is split along N, the first N/2 columns in rank 0's shared
// memory and the rest in rank 1's, both at the descriptor's address.
template <bool kWarp = false>
__device__ __forceinline__ void mma_ss_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  FA_MMA_ASM(kWarp, "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;", "r"(d_tmem),
             "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}
template <bool kWarp = false>
__device__ __forceinline__ void mma_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  FA_MMA_ASM(kWarp, "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;", "r"(d_tmem),
             "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// The same two forms for 8-bit operands (kind::f8f6f4: K = 32 per MMA).
template <bool kWarp = false>
__device__ __forceinline__ void mma_ss_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  FA_MMA_ASM(kWarp, "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;", "r"(d_tmem),
             "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}
template <bool kWarp = false>
__device__ __forceinline__ void mma_ts_f8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  FA_MMA_ASM(kWarp, "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;", "r"(d_tmem),
             "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}
#undef FA_MMA_ASM

// Arrives once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
template <bool kWarp = false>
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  if constexpr (kWarp)
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
        : "memory");
  else
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// Pair form: arrives once on the barrier at shared::cluster address
// `cluster_bar` (this CTA's own address, or one from cluster_smem() for the
// other CTA of the pair) when the pair MMAs this thread issued so far have
// completed.  A barrier in each CTA takes one commit each.
template <bool kWarp = false>
__device__ __forceinline__ void mma_commit_pair(uint32_t cluster_bar) {
  if constexpr (kWarp)
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
            cluster_bar)
        : "memory");
  else
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            cluster_bar)
        : "memory");
}

// ---------------------------------------------------------------------------
// Small numeric helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2_mufu(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Four floats -> four e4m3 (round to nearest even, saturating at +-448),
// the first in the low byte.
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  const __nv_fp8x2_e4m3 lo(make_float2(a, b));
  const __nv_fp8x2_e4m3 hi(make_float2(c, d));
  return static_cast<uint32_t>(lo.__x) | (static_cast<uint32_t>(hi.__x) << 16);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Software exp2 on the FMA pipe: 2^x = 2^n * p(f), n = round(x), f = x - n in
// [-1/2, 1/2], p the fitted polynomial of exp2_poly_coeffs.h.  Adding
// 1.5 * 2^23 rounds x to an integer held in the low mantissa bits of t, so
// (bits(t) << 23) is n << 23 modulo 2^32 and one integer add scales p by 2^n.
// x is clamped to [-125, 127] so the result stays a normal float.
__device__ __forceinline__ float exp2_poly(float x) {
  x = fminf(fmaxf(x, -125.0f), 127.0f);
  const float kRound = 12582912.0f;  // 1.5 * 2^23
  const float t = __fadd_rn(x, kRound);
  const float n = __fsub_rn(t, kRound);
  const float f = __fsub_rn(x, n);
  float p = fmaf(FA_EXP2_POLY_C3, f, FA_EXP2_POLY_C2);
  p = fmaf(p, f, FA_EXP2_POLY_C1);
  p = fmaf(p, f, 1.0f);
  return __uint_as_float(__float_as_uint(p) + (__float_as_uint(t) << 23));
}

// ---------------------------------------------------------------------------
// Packed fp32 pairs (f32x2 instructions of sm_100+): one instruction works on
// two fp32 values held in a 64-bit register pair.
// ---------------------------------------------------------------------------
using f32x2 = unsigned long long;

__device__ __forceinline__ f32x2 f2_pack(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(f32x2 v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f32x2 f2_add(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 f2_mul(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// max of three fp32 values in one instruction (sm_100+)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// exp2_poly on a pair, the arithmetic in f32x2 instructions.  Inputs are at
// most 2^8 here (the softmax's stale-max bound), so only the low clamp stays.
__device__ __forceinline__ void exp2_poly2(float x0, float x1, float& y0, float& y1) {
  const f32x2 x = f2_pack(fmaxf(x0, -125.0f), fmaxf(x1, -125.0f));
  const f32x2 kRound = f2_pack(12582912.0f, 12582912.0f);
  const f32x2 kNegRound = f2_pack(-12582912.0f, -12582912.0f);
  const f32x2 kMinus1 = f2_pack(-1.0f, -1.0f);
  const f32x2 t = f2_add(x, kRound);
  const f32x2 n = f2_add(t, kNegRound);
  const f32x2 f = f2_fma(n, kMinus1, x);
  f32x2 p = f2_fma(f2_pack(FA_EXP2_POLY_C3, FA_EXP2_POLY_C3), f,
                   f2_pack(FA_EXP2_POLY_C2, FA_EXP2_POLY_C2));
  p = f2_fma(p, f, f2_pack(FA_EXP2_POLY_C1, FA_EXP2_POLY_C1));
  p = f2_fma(p, f, f2_pack(1.0f, 1.0f));
  float p0, p1, t0, t1;
  f2_unpack(p, p0, p1);
  f2_unpack(t, t0, t1);
  y0 = __uint_as_float(__float_as_uint(p0) + (__float_as_uint(t0) << 23));
  y1 = __uint_as_float(__float_as_uint(p1) + (__float_as_uint(t1) << 23));
}

// Keeps later uses of r[] after an earlier wait (the asm statements are not
// reordered with each other).
__device__ __forceinline__ void reg_fence(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31]));
}

// Register reallocation between warpgroups (executed by all threads of a
// warpgroup).  The callers' shares must add up to at most the registers the
// CTA was launched with; the launchers check the compiled register count.
template <int N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ void reg_fence16(uint32_t (&r)[16]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]));
}

// Moves this warpgroup from the launch allocation `kFrom` to `kTo` registers
// per thread with the instruction that goes that way: setmaxnreg.dec to a
// count above the current one (or .inc to one below) is an illegal
// instruction.
template <int kTo, int kFrom>
__device__ __forceinline__ void regs_set() {
  static_assert(kTo % 8 == 0 && kTo >= 24 && kTo <= 256, "setmaxnreg count");
  if constexpr (kTo > kFrom) regs_inc<kTo>();
  else if constexpr (kTo < kFrom) regs_dec<kTo>();
}

__device__ __forceinline__ int warp_id() { return threadIdx.x >> 5; }
__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }

}  // namespace fa
