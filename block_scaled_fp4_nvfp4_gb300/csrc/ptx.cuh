// Thin inline-PTX wrappers for the sm_103a features the GEMM uses: mbarriers,
// TMA (tensor and bulk copies), L2 cache policies and the tcgen05 tensor-core
// family (tensor memory alloc, scale copy, block-scaled MMA, commit, load).
// Each wrapper is one instruction with its operands; the semantics are the
// PTX ISA's.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace nvfp4 {
namespace ptx {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// True once the phase with the given parity has completed.
// try_wait with acquire at cluster scope, for barriers that other CTAs of
// the cluster arrive on (mbar_arrive_remote).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// ---------------------------------------------------------------- L2 policy
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled store shared -> global (rows/columns outside the map are clipped).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y,
                                             int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(x), "r"(y), "r"(z)
      : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until at most N bulk groups are still in flight (writes complete).
template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Make generic-proxy shared-memory writes visible to the async proxy (TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// The same for global memory: a bulk copy after this reads what the thread's
// generic-proxy accesses (e.g. an acquire of a flag) made visible.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}


// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Tensor memory -> registers: each thread of the warp reads its lane, 32
// consecutive 32-bit columns.
__device__ __forceinline__ void tmem_load_32cols(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_load_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Orders later uses of 32 tcgen05.ld destination registers after the
// preceding tcgen05.wait::ld (volatile asm statements keep their order).
__device__ __forceinline__ void reg_fence32(uint32_t* r) {
  asm volatile("" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}

// ---------------------------------------------------------------- misc
// Programmatic dependent launch (no-ops when the launch did not opt in).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// L2 prefetches (no shared-memory destination, no completion tracking).  L2
// is the coherence point for global memory, so a prefetch issued before a
// preceding kernel finished writing the same bytes only costs bandwidth: the
// real loads, issued after griddepcontrol.wait, see the final values.
__device__ __forceinline__ void prefetch_tile_l2_3d(const CUtensorMap* map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Flag word in global memory: acquire load / release store at GPU scope.
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(int* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Invalidate one 128-byte L2 line without writing it back (its contents
// become undefined).  `p` must be 128-byte aligned.
__device__ __forceinline__ void discard_l2(const void* p) {
  asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

// ---------------------------------------------------------------- warp-issued forms
// The whole warp executes these with warp-uniform operands; elect.sync picks
// one lane (the same lowest lane every time for a full warp) to issue.  Keeping
// the warp converged lets the operands stay in uniform registers, which the
// tcgen05 and TMA instructions read.
__device__ __forceinline__ void mbar_arrive_expect_tx_elect(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d_elect(uint32_t dst, const CUtensorMap* map, int x, int y,
                                                  int z, uint32_t bar, uint64_t policy) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;\n\t}" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void bulk_load_elect(uint32_t dst, const void* src, uint32_t bytes,
                                                uint32_t bar, uint64_t policy) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;\n\t}" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tc_commit_elect(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}

// One MMA k-block in one instruction group under a single elect.sync: the
// scale-atom copies into tensor memory (SFA, then NSFB atoms of SFB) and the
// block-scaled MMA that reads them.  `CG` is the cta_group (1 or 2).
#define NVFP4_CP(CG, T, D) "@e tcgen05.cp.cta_group::" #CG ".32x128b.warpx4 [%" #T "], %" #D ";\n\t"
#define NVFP4_MMA(CG) \
  "@e tcgen05.mma.cta_group::" #CG ".kind::mxf4nvf4.block_scale.block16 [%4], %5, %6, %7, [%8], [%9], p;\n\t"
template <int CG, int NSFB>
__device__ __forceinline__ void tc_kblock_elect(uint32_t sfa_t, uint64_t sfa_d, uint32_t sfb_t, uint64_t sfb_d,
                                                uint32_t sfb_t2, uint64_t sfb_d2, uint32_t d_tmem, uint64_t a_desc,
                                                uint64_t b_desc, uint32_t idesc, uint32_t sfa_mma, uint32_t sfb_mma,
                                                uint32_t accumulate) {
  static_assert((CG == 1 || CG == 2) && (NSFB == 1 || NSFB == 2), "variants");
  if constexpr (CG == 1 && NSFB == 1)
    asm volatile("{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %10, 0;\n\telect.sync _|e, 0xffffffff;\n\t" NVFP4_CP(1, 0, 1)
                     NVFP4_CP(1, 2, 3) NVFP4_MMA(1) "}" ::"r"(sfa_t),
                 "l"(sfa_d), "r"(sfb_t), "l"(sfb_d), "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_mma),
                 "r"(sfb_mma), "r"(accumulate), "r"(sfb_t2), "l"(sfb_d2)
                 : "memory");
  else if constexpr (CG == 1 && NSFB == 2)
    asm volatile("{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %10, 0;\n\telect.sync _|e, 0xffffffff;\n\t" NVFP4_CP(1, 0, 1)
                     NVFP4_CP(1, 2, 3) NVFP4_CP(1, 11, 12) NVFP4_MMA(1) "}" ::"r"(sfa_t),
                 "l"(sfa_d), "r"(sfb_t), "l"(sfb_d), "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_mma),
                 "r"(sfb_mma), "r"(accumulate), "r"(sfb_t2), "l"(sfb_d2)
                 : "memory");
  else if constexpr (CG == 2 && NSFB == 1)
    asm volatile("{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %10, 0;\n\telect.sync _|e, 0xffffffff;\n\t" NVFP4_CP(2, 0, 1)
                     NVFP4_CP(2, 2, 3) NVFP4_MMA(2) "}" ::"r"(sfa_t),
                 "l"(sfa_d), "r"(sfb_t), "l"(sfb_d), "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_mma),
                 "r"(sfb_mma), "r"(accumulate), "r"(sfb_t2), "l"(sfb_d2)
                 : "memory");
  else
    asm volatile("{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %10, 0;\n\telect.sync _|e, 0xffffffff;\n\t" NVFP4_CP(2, 0, 1)
                     NVFP4_CP(2, 2, 3) NVFP4_CP(2, 11, 12) NVFP4_MMA(2) "}" ::"r"(sfa_t),
                 "l"(sfa_d), "r"(sfb_t), "l"(sfb_d), "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_mma),
                 "r"(sfb_mma), "r"(accumulate), "r"(sfb_t2), "l"(sfb_d2)
                 : "memory");
}
#undef NVFP4_CP
#undef NVFP4_MMA

// ---------------------------------------------------------------- clusters
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// All threads of every CTA of the cluster (hardware barrier; every CTA of a
// cluster is co-scheduled, so it completes once each CTA arrives).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 3-D tiled load delivered to the same shared-memory offset of every CTA in
// `cta_mask`; each destination CTA's mbarrier at `bar` counts the bytes.
__device__ __forceinline__ void tma_load_3d_mc_elect(uint32_t dst, const CUtensorMap* map, int x, int y,
                                                     int z, uint32_t bar, uint64_t policy,
                                                     uint16_t cta_mask) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6, %7;\n\t}" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "h"(cta_mask), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void bulk_load_mc_elect(uint32_t dst, const void* src, uint32_t bytes,
                                                   uint32_t bar, uint64_t policy, uint16_t cta_mask) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4, %5;\n\t}" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "h"(cta_mask), "l"(policy)
      : "memory");
}

// Commit whose arrival lands on the mbarrier at `bar` in every CTA of `cta_mask`.
__device__ __forceinline__ void tc_commit_mc_elect(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}

// ---------------------------------------------------------------- 2-SM pairs
// tcgen05 with cta_group::2: one thread of the pair's even CTA (the leader)
// issues for both CTAs; shared-memory descriptors and tensor-memory addresses
// name the same offsets in each CTA.  A kernel uses one cta_group throughout,
// so a pair kernel also allocates with cta_group::2 (one warp of each CTA).

// Address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Arrive on an mbarrier of any CTA of the cluster (shared::cluster address)
// with the default CTA-scope release.  For arrivals that publish no ordinary
// memory writes -- that this CTA's ring is idle, or that this thread's
// tensor-memory reads are complete (tcgen05.wait::ld) -- a cluster-scope
// release is not needed, and on GB300 it costs about a microsecond per
// arrival (it waits for the thread's outstanding memory traffic).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// One thread arms a local barrier with a transaction byte count and arrives.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// Counts `bytes` of the current phase's transactions as done without any
// data: for copies a barrier was armed for but that were never issued.
__device__ __forceinline__ void mbar_complete_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// 32-bit load / store of shared memory of any CTA of the cluster
// (shared::cluster address from mapa_shared).
__device__ __forceinline__ uint32_t ld_shared_cluster(uint32_t cluster_addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(cluster_addr) : "memory");
  return v;
}
__device__ __forceinline__ void st_shared_cluster(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// Bulk copy from this CTA's shared memory into the shared memory of a CTA of
// the cluster; the destination CTA's mbarrier (shared::cluster address)
// counts the bytes.  Addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_copy_to_cluster(uint32_t dst_cluster, uint32_t src, uint32_t bytes,
                                                     uint32_t bar_cluster) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   dst_cluster),
               "r"(src), "r"(bytes), "r"(bar_cluster)
               : "memory");
}

__device__ __forceinline__ void tmem_alloc2(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish2() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Tiled loads into this CTA's shared memory whose bytes are counted on an
// mbarrier that may live in the peer CTA (`bar` is a shared::cluster address).
__device__ __forceinline__ void tma_load_3d_pair_elect(uint32_t dst, const CUtensorMap* map, int x, int y,
                                                       int z, uint32_t bar, uint64_t policy) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;\n\t}" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d_pair_elect(uint32_t dst, const CUtensorMap* map, int x, int y,
                                                       uint32_t bar, uint64_t policy) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;\n\t}" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// Commit of the pair's MMAs and copies; the arrival lands on the mbarrier at
// `bar` in every CTA of `cta_mask`.
__device__ __forceinline__ void tc_commit2_mc_elect(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}

}  // namespace ptx
}  // namespace nvfp4
