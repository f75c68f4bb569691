// Persistent, warp-specialised NVFP4 block-scaled GEMM for sm_103a.
//
// One CTA per SM walks a static list of work units (output tile, K range) of
// all groups.  Inside a CTA (256 threads):
//   warps 0-2   TMA producers: per 256-wide k-tile warp 0 arms the stage's
//               "full" mbarrier and copies the A tile (128 rows x 128 B) and
//               its scale slab, warp 1 the B tile (BN rows x 128 B, or this
//               CTA's half of it when two CTAs share it), warp 2 the B scale
//               slabs;
//   warp 3      MMA issuer (one elected lane): per MMA k-block its scale atoms
//               into tensor memory with tcgen05.cp, then one
//               tcgen05.mma.kind::mxf4nvf4.block_scale.block16 (128 x BN x 64,
//               or 256 x BN x 64 over a CTA pair) into a tensor-memory
//               accumulator; one commit per k-tile frees the stage;
//   warps 4-7   epilogue, one per 32-lane tensor-memory sub-partition:
//               tcgen05.ld of the accumulator (one row per thread), fp32 ->
//               fp16 (RNE), 64B-swizzled staging and TMA stores of 32 x 32
//               boxes (rows past M and columns past N are clipped).
// Stream-K segments of a tile either exchange fp32 partials through
// distributed shared memory (the tile's segments form one cluster) or write
// them to a workspace where the last segment to arrive sums them; both sum in
// segment (k) order, so results are deterministic.
//
// The warp roles and the mbarrier ring follow the structure of the pages'
// kernels ("nvfp4 group gemm, submission 407526", grouped_kernel; "nvfp4 gemm,
// submission 125598", kernel); the persistent unit loop, split-K, the
// double-buffered accumulator, the scale-slot ring, the TMA-store epilogue and
// the bounded waits are this library's own.
//
// Every wait is bounded (Waiter below).  When one runs out the CTA records a
// status code, stops issuing, waits for its own copies and MMAs in flight,
// frees its tensor memory and exits.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "descriptors.h"
#include "gemm_params.h"
#include "ptx.cuh"
#include "schedule.h"

namespace nvfp4 {

namespace {

constexpr int kMaxStages = 8;

struct SmemCtl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t epi_gather;
  uint64_t epi_bcast;
  uint64_t mma_drain;
  uint64_t red_go;    // cluster reduction: every CTA of the cluster may now be written
  uint64_t red_full;    // cluster reduction: every peer's slice of this CTA's columns landed
  uint64_t part_full;   // pair stream-K: the other segment's partial landed in the ring
  uint32_t tmem_base;
  volatile int abort;
  int last_flag;
  // Copy bookkeeping for the drain after an abort: per producer warp and
  // stage, the last use (the warp's k-tile count) it issued copies for and
  // the bytes those copies deliver to each destination barrier; warp 0's
  // arming of each stage (use and armed byte count); in reduce clusters,
  // whether red_full was armed and, per epilogue warp, which ranks its part
  // of this CTA's partial went to.
  int rec_use[kProducerWarps][kMaxStages];
  uint32_t rec_bytes[kProducerWarps][kMaxStages];
  int arm_use[kMaxStages];
  uint32_t arm_bytes[kMaxStages];
  int red_armed;
  uint32_t red_sent[kEpiWarps];  // per epilogue warp: ranks its part of the partial went to
  uint32_t part_armed;   // bytes part_full was armed with
  uint32_t part_issued;  // bytes of partial copies issued
  uint32_t peer_abort[4];  // abort flags the cluster's CTAs published here (index = rank)
};

// Bounded mbarrier wait.  Returns false if the CTA is aborting or the limit
// ran out (then the abort flag and the device status word are set).
struct Waiter {
  volatile int* abort_flag;
  int* status;
  unsigned long long timeout_ns;

  // kCluster: acquire at cluster scope (the phase was completed by arrivals
  // that release writes made by other CTAs of the cluster).
  template <bool kCluster = false>
  __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity, int code) const {
    auto test = [&]() {
      return kCluster ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity);
    };
    if (test()) return true;
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t i = 1;; ++i) {
      if (test()) return true;
      if ((i & 7u) == 0) {
        if (*abort_flag) return false;
        if (ptx::globaltimer() - t0 > timeout_ns) {
          *abort_flag = 1;
          atomicCAS(status, 0, code);
          return false;
        }
      }
    }
  }

  // Used only while shutting down after an abort: waits for the CTA's own
  // asynchronous work, bounded by the same limit, ignoring the abort flag.
  __device__ __forceinline__ bool drain(uint32_t bar, uint32_t parity) const {
    const uint64_t t0 = ptx::globaltimer();
    while (!ptx::mbar_try_wait(bar, parity)) {
      if (ptx::globaltimer() - t0 > timeout_ns) return false;
    }
    return true;
  }
};

// Every lane polls the barrier; the vote makes the outcome warp-uniform and
// reconverges the warp (a lane that saw the phase complete just as another one
// gave up still aborts with it).
template <bool kCluster = false>
__device__ __forceinline__ bool warp_wait(const Waiter& W, uint32_t bar, uint32_t parity, int code) {
  const bool ok = W.template wait<kCluster>(bar, parity, code);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);  // round to nearest even
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float4 ld_shared_v4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

}  // namespace

template <int BN, int CL, int MODE>
__global__ void __launch_bounds__(kNumThreads, 1) nvfp4_gemm_kernel(const __grid_constant__ GemmParams p) {
  constexpr bool P2 = MODE == kModePair;
  constexpr bool kMc = MODE == kModeMulticast;
  constexpr bool kRed = MODE == kModeReduce;
  using Cfg = TileCfg<BN, P2>;
  static_assert(MODE == kModeSingle ? CL == 1 : (kRed ? (CL == 2 || CL == 4) : CL == 2), "cluster size");
  // CL == 2: the two CTAs of a cluster run tiles with the same B columns
  // (m-tiles 2q and 2q+1).  Without P2 each loads half of every B tile and
  // of the B scale slabs and multicasts it to both, halving B's L2 -> SM
  // traffic.  With P2 the pair runs one 256 x BN tile as 2-SM MMAs
  // (tcgen05 cta_group::2, issued by the even CTA): each CTA keeps only its
  // half of B in shared memory, the tensor cores exchange the halves, and
  // every copy of both CTAs is counted on the leader's "full" barrier.
  constexpr uint16_t kPeers = static_cast<uint16_t>((1u << CL) - 1u);
  constexpr int kBHalfRows = (kMc || P2) ? BN / 2 : BN;  // B rows each CTA of a sharing pair loads
  constexpr int kStages = Cfg::kStages;
  static_assert(kStages <= kMaxStages, "stage ring too deep");

  extern __shared__ uint8_t dsmem_raw[];
  __shared__ SmemCtl ctl;

  const uint32_t raw = ptx::smem_addr(dsmem_raw);
  const uint32_t smem_base = (raw + 1023u) & ~1023u;  // 128B-swizzled tiles need 1024-B alignment
  const uint32_t epi_base = smem_base + kStages * Cfg::kStageBytes;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int crank = CL > 1 ? static_cast<int>(ptx::cluster_ctarank()) : 0;
  // Work is dealt per cluster when the cluster shares tiles (multicast, pair)
  // and per CTA when its CTAs are the segments of one tile (reduce).
  const int unit = kRed ? static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x) / CL;
  const int units = kRed ? static_cast<int>(gridDim.x) : static_cast<int>(gridDim.x) / CL;
  const int wrank = kRed ? 0 : crank;  // rank passed to the work cursor
  const int brow = (kMc || P2) ? crank * kBHalfRows : 0;  // first B row of the tile this CTA loads

  auto full_bar = [&](int s) { return ptx::smem_addr(&ctl.full[s]); };
  auto empty_bar = [&](int s) { return ptx::smem_addr(&ctl.empty[s]); };
  auto acc_full_bar = [&](int b) { return ptx::smem_addr(&ctl.acc_full[b]); };
  auto acc_empty_bar = [&](int b) { return ptx::smem_addr(&ctl.acc_empty[b]); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), kMc ? CL : 1);  // released by the MMAs of every CTA that reads it
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(acc_full_bar(b), 1);
      ptx::mbar_init(acc_empty_bar(b), kEpiWarps * (P2 ? 2 : 1));  // pairs: both CTAs' epilogues
    }
    ptx::mbar_init(ptx::smem_addr(&ctl.epi_gather), kEpiWarps);
    ptx::mbar_init(ptx::smem_addr(&ctl.epi_bcast), 1);
    ptx::mbar_init(ptx::smem_addr(&ctl.mma_drain), 1);
    ptx::mbar_init(ptx::smem_addr(&ctl.red_go), CL);                 // one arrival per CTA of the cluster
    ptx::mbar_init(ptx::smem_addr(&ctl.red_full), 1);  // armed with the peers' bytes
    ptx::mbar_init(ptx::smem_addr(&ctl.part_full), 1);
    ctl.abort = 0;
    ctl.last_flag = 0;
    for (int s = 0; s < kMaxStages; ++s) {
      for (int w = 0; w < kProducerWarps; ++w) {
        ctl.rec_use[w][s] = -1;
        ctl.rec_bytes[w][s] = 0;
      }
      ctl.arm_use[s] = -1;
      ctl.arm_bytes[s] = 0;
    }
    ctl.red_armed = 0;
    for (int w = 0; w < kEpiWarps; ++w) ctl.red_sent[w] = 0;
    ctl.part_armed = 0;
    ctl.part_issued = 0;
    for (int r = 0; r < 4; ++r) ctl.peer_abort[r] = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int g = 0; g < p.sched.num_groups; ++g) {
      ptx::prefetch_tensormap(&p.tmA[g]);
      ptx::prefetch_tensormap(&p.tmB[g]);
      ptx::prefetch_tensormap(&p.tmC[g]);
      if constexpr (P2) {
        ptx::prefetch_tensormap(&p.tmSFA[g]);
        ptx::prefetch_tensormap(&p.tmSFB[g]);
      }
    }
  }
  if (warp == kMmaWarp) {
    if constexpr (P2) {
      ptx::tmem_alloc2(ptx::smem_addr(&ctl.tmem_base), Cfg::kTmemCols);
      ptx::tmem_relinquish2();
    } else {
      ptx::tmem_alloc(ptx::smem_addr(&ctl.tmem_base), Cfg::kTmemCols);
      ptx::tmem_relinquish();
    }
  }
  ptx::tc_fence_before_sync();
  __syncthreads();
  if constexpr (CL > 1) ptx::cluster_sync();  // peers' barriers exist before any multicast
  ptx::tc_fence_after_sync();
  const uint32_t tmem = ctl.tmem_base;

  // Programmatic dependent launch: everything above overlaps the previous
  // kernel on the stream, and so does each role's set-up below (its work
  // list, the first tile's addresses -- loads from the parameter block whose
  // latency would otherwise sit between the previous kernel's end and the
  // first copy).  Only global memory must wait for the previous kernel: the
  // producers wait right before their first copy and the epilogue before its
  // first store; the MMA warp touches shared and tensor memory only and never
  // waits.  Optionally (prefetch_ktiles > 0) one thread asks L2 for the first
  // k-tiles this CTA will load before that wait.
  if (warp == 0 && lane == 0 && p.prefetch_ktiles > 0) {
    WorkCursor pc;
    work_begin(p.sched, unit, units, pc, wrank);
    Work pw;
    int left = p.prefetch_ktiles;
    while (left > 0 && work_next(p.sched, unit, units, pc, pw)) {
      const size_t atoms = static_cast<size_t>(p.sched.ktiles[pw.g]) * 4;
      const uint8_t* sfa = p.sfa[pw.g] + (static_cast<size_t>(pw.l) * p.sf_rows_a[pw.g] + pw.tm) * atoms * kSfAtomBytes;
      const int sfb_block0 = pw.tn * BN / 128;
      const uint8_t* sfb = p.sfb[pw.g] + (static_cast<size_t>(pw.l) * p.sf_rows_b[pw.g] + sfb_block0) * atoms * kSfAtomBytes;
      for (int kt = pw.kt0; kt < pw.kt1 && left > 0; ++kt, --left) {
        ptx::prefetch_tile_l2_3d(&p.tmA[pw.g], kt * kBKBytes, pw.tm * kBM, pw.l);
        ptx::prefetch_tile_l2_3d(&p.tmB[pw.g], kt * kBKBytes, pw.tn * BN + brow, pw.l);
        ptx::prefetch_l2(sfa + static_cast<size_t>(kt) * kSfSlabBytes, kSfSlabBytes);
        if (sfb_block0 < p.sf_rows_b[pw.g]) ptx::prefetch_l2(sfb + static_cast<size_t>(kt) * kSfSlabBytes, kSfSlabBytes);
      }
    }
  }
  ptx::griddep_launch_dependents();

  const Waiter W{&ctl.abort, p.status, p.timeout_ns};

  // Counted drain after an abort, run by one thread of each CTA once every
  // warp of the cluster has stopped issuing.  For each stage it takes the last
  // use any producer warp issued copies for (its own warps' and, where copies
  // signal this CTA's barrier from the peer -- B multicast, 2-SM pairs -- the
  // peer's records, read through distributed shared memory).  If that phase
  // is still open it makes the phase completable by exactly the bytes that
  // were issued: it adds the arrival and byte count warp 0 did not make, or
  // counts as done the bytes armed for but never issued; then it waits
  // (bounded) for the phase, i.e. for every issued copy to have landed.  The
  // reduction clusters' partial exchange is drained the same way.
  auto drain_after_abort = [&]() {
    auto peer_word = [&](const void* local, int rank) {
      return ptx::ld_shared_cluster(ptx::mapa_shared(ptx::smem_addr(local), static_cast<uint32_t>(rank)));
    };
    if (!P2 || crank == 0) {  // a pair's copies all signal the leader's barriers
      for (int s = 0; s < kStages; ++s) {
        int use = ctl.arm_use[s];
        for (int w = 0; w < kProducerWarps; ++w) use = ctl.rec_use[w][s] > use ? ctl.rec_use[w][s] : use;
        int peer_use[kProducerWarps];
        uint32_t peer_bytes[kProducerWarps];
        for (int w = 0; w < kProducerWarps; ++w) {
          peer_use[w] = -1;
          peer_bytes[w] = 0;
          if ((P2 || (kMc && w > 0)) && CL == 2) {  // peer warps whose copies land here
            peer_use[w] = static_cast<int>(peer_word(&ctl.rec_use[w][s], crank ^ 1));
            peer_bytes[w] = peer_word(&ctl.rec_bytes[w][s], crank ^ 1);
            use = peer_use[w] > use ? peer_use[w] : use;
          }
        }
        if (use < 0) continue;
        const uint32_t parity = static_cast<uint32_t>(use / kStages) & 1u;
        const uint32_t bar = full_bar(s);
        if (ptx::mbar_try_wait(bar, parity)) continue;  // complete: nothing of it in flight
        uint32_t issued = 0;
        for (int w = 0; w < kProducerWarps; ++w) {
          if (ctl.rec_use[w][s] == use) issued += ctl.rec_bytes[w][s];
          if (peer_use[w] == use) issued += peer_bytes[w];
        }
        if (ctl.arm_use[s] == use) {
          if (ctl.arm_bytes[s] > issued) ptx::mbar_complete_tx(bar, ctl.arm_bytes[s] - issued);
        } else {
          ptx::mbar_arrive_expect_tx(bar, issued);
        }
        W.drain(bar, parity);
      }
    }
    if (ctl.part_armed) {
      const uint32_t bar = ptx::smem_addr(&ctl.part_full);
      if (!ptx::mbar_try_wait(bar, 0)) {
        if (ctl.part_armed > ctl.part_issued) ptx::mbar_complete_tx(bar, ctl.part_armed - ctl.part_issued);
        W.drain(bar, 0);
      }
    }
    if constexpr (kRed) {
      constexpr uint32_t kSlotBytes = BN / CL * kBM * 4;
      constexpr uint32_t kWarpPart = kSlotBytes / kEpiWarps;
      uint32_t got = 0;  // bytes the peers' warps sent into this CTA's receive slots
      for (int r = 0; r < CL; ++r)
        if (r != crank)
          for (int w = 0; w < kEpiWarps; ++w)
            if ((peer_word(&ctl.red_sent[w], r) >> crank) & 1u) got += kWarpPart;
      const uint32_t bar = ptx::smem_addr(&ctl.red_full);
      if ((ctl.red_armed || got) && !ptx::mbar_try_wait(bar, 0)) {
        const uint32_t expected = (CL - 1) * kSlotBytes;
        if (ctl.red_armed) {
          if (expected > got) ptx::mbar_complete_tx(bar, expected - got);
        } else {
          ptx::mbar_arrive_expect_tx(bar, got);
        }
        W.drain(bar, 0);
      }
    }
  };

  if (warp < kProducerWarps) {
    // ------------------------------------------------------------ producers
    // Three producer warps fill every stage together: warp 0 arms the stage's
    // barrier with the whole byte count and loads A and its scales, warp 1
    // loads B, warp 2 the B scale slabs.  Splitting the copies shortens the
    // time from a stage's release to its refill, which bounds the ring's
    // throughput (the barrier's byte count may briefly go negative when
    // another warp's bytes land first; the phase still needs warp 0's
    // arrival).  Measured on GB300 against two warps (B and its slabs on one):
    // 8192^3 as 2-SM pairs 177 -> 172 us, the two-group workload 27.7 -> 27.4
    // us, the others unchanged.  Within a warp every lane runs the loop with
    // warp-uniform values and one elected lane issues each copy (see the
    // *_elect wrappers).
    const uint64_t pol_stream = ptx::policy_evict_first();
    const uint64_t pol_keep = ptx::policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    int count = 0;
    bool ok = true;
    bool dep_done = false;  // griddepcontrol.wait passed
    const int skip_at = blockIdx.x == 0 ? p.debug_skip_ktile : -1;
    const uint32_t full0 = full_bar(0), empty0 = empty_bar(0);
    [[maybe_unused]] uint32_t lfull0 = 0;
    if constexpr (P2) lfull0 = ptx::mapa_shared(full0, 0);
    WorkCursor cur;
    work_begin(p.sched, unit, units, cur, wrank);
    Work x;
    bool any_item = false;
    while (ok && work_next(p.sched, unit, units, cur, x)) {
      any_item = true;
      const CUtensorMap* mapA = &p.tmA[x.g];
      const CUtensorMap* mapB = &p.tmB[x.g];
      const uint64_t polA = p.a_streams[x.g] ? pol_stream : pol_keep;
      const uint64_t polB = p.a_streams[x.g] ? pol_keep : pol_stream;
      const size_t atoms_per_block = static_cast<size_t>(p.sched.ktiles[x.g]) * 4;
      const uint8_t* sfa = p.sfa[x.g] +
          (static_cast<size_t>(x.l) * p.sf_rows_a[x.g] + x.tm) * atoms_per_block * kSfAtomBytes;
      const int sfb_block0 = x.tn * BN / 128;  // 128-row scale block holding the tile's first row
      const uint8_t* sfb = p.sfb[x.g] +
          (static_cast<size_t>(x.l) * p.sf_rows_b[x.g] + sfb_block0) * atoms_per_block * kSfAtomBytes;
      int nsfb = p.sf_rows_b[x.g] - sfb_block0;
      nsfb = nsfb < Cfg::kSfbBlocks ? nsfb : Cfg::kSfbBlocks;
      // pair copies of the scale slabs: rows of 256 B in the 2-D scale maps
      const int sfa_row = static_cast<int>(atoms_per_block / 4 * 8) * (x.l * p.sf_rows_a[x.g] + x.tm);
      const int sfb_row = static_cast<int>(atoms_per_block / 4 * 8) * (x.l * p.sf_rows_b[x.g] + sfb_block0);
      const uint32_t stage_tx =
          Cfg::kABytes + Cfg::kBBytes + kSfSlabBytes + static_cast<uint32_t>(nsfb) * kSfSlabBytes;
      for (int kt = x.kt0; kt < x.kt1; ++kt) {
        if (!warp_wait(W, empty0 + 8u * stage, phase ^ 1u, kStatusTimeoutProducer)) {
          ok = false;
          break;
        }
        const uint32_t sA = smem_base + stage * Cfg::kStageBytes;
        const uint32_t sB = sA + Cfg::kABytes;
        const uint32_t sSFA = sB + Cfg::kBBytes;
        const uint32_t sSFB = sSFA + kSfSlabBytes;
        if (!dep_done) {
          ptx::griddep_wait();  // the previous kernel's writes are visible from here on
          dep_done = true;
        }
        if (count == skip_at) {
          // test-only: nothing issued, nothing in flight, nothing recorded
        } else {
          const uint32_t fb = full0 + 8u * stage;
          if constexpr (P2) {
            // Every copy of both CTAs lands on the leader's barrier, armed by
            // the leader with both CTAs' bytes.  Both B scale slabs go to each
            // CTA (each tensor core scales all BN columns); a slab past the
            // last 128-row block reads other scales or zeros, harmless since
            // those B rows are zero-filled and their columns are not stored.
            const uint32_t lfb = lfull0 + 8u * stage;
            if (warp == 0) {
              if (crank == 0) ptx::mbar_arrive_expect_tx_elect(fb, 2u * Cfg::kStageBytes);
              ptx::tma_load_3d_pair_elect(sA, mapA, kt * kBKBytes, x.tm * kBM, x.l, lfb, polA);
              ptx::tma_load_2d_pair_elect(sSFA, &p.tmSFA[x.g], 0, sfa_row + kt * 8, lfb, polA);
            } else if (warp == 1) {
              ptx::tma_load_3d_pair_elect(sB, mapB, kt * kBKBytes, x.tn * BN + crank * kBHalfRows, x.l, lfb, polB);
            } else {
#pragma unroll
              for (int j = 0; j < Cfg::kSfbBlocks; ++j)
                ptx::tma_load_2d_pair_elect(sSFB + j * kSfSlabBytes, &p.tmSFB[x.g], 0,
                                            sfb_row + static_cast<int>(atoms_per_block / 4 * 8) * j + kt * 8,
                                            lfb, polB);
            }
          } else if (warp == 0) {
            ptx::mbar_arrive_expect_tx_elect(fb, stage_tx);
            ptx::tma_load_3d_elect(sA, mapA, kt * kBKBytes, x.tm * kBM, x.l, fb, polA);
            ptx::bulk_load_elect(sSFA, sfa + static_cast<size_t>(kt) * kSfSlabBytes, kSfSlabBytes, fb, polA);
          } else if constexpr (!kMc) {
            if (warp == 1) {
              ptx::tma_load_3d_elect(sB, mapB, kt * kBKBytes, x.tn * BN, x.l, fb, polB);
            } else {
              for (int j = 0; j < nsfb; ++j)
                ptx::bulk_load_elect(sSFB + j * kSfSlabBytes,
                                     sfb + (static_cast<size_t>(j) * atoms_per_block + kt * 4) * kSfAtomBytes,
                                     kSfSlabBytes, fb, polB);
            }
          } else if (warp == 1) {
            // this CTA's half of the B rows, for both CTAs
            ptx::tma_load_3d_mc_elect(sB + crank * kBHalfRows * kBKBytes, mapB, kt * kBKBytes,
                                      x.tn * BN + crank * kBHalfRows, x.l, fb, polB, kPeers);
          } else {
            // every CL-th B scale slab, for both CTAs
            for (int j = crank; j < nsfb; j += CL)
              ptx::bulk_load_mc_elect(sSFB + j * kSfSlabBytes,
                                      sfb + (static_cast<size_t>(j) * atoms_per_block + kt * 4) * kSfAtomBytes,
                                      kSfSlabBytes, fb, polB, kPeers);
          }
          // Record what went out (every lane stores the same values: no
          // divergent branch in the issue loop).  Bytes are counted as each
          // destination barrier sees them: a multicast copy delivers its full
          // size to every CTA of the cluster.
          uint32_t sent;
          if (warp == 0) {
            sent = Cfg::kABytes + kSfSlabBytes;
            const bool arms = !P2 || crank == 0;
            if (arms) {
              ctl.arm_use[stage] = count;
              ctl.arm_bytes[stage] = P2 ? 2u * Cfg::kStageBytes : stage_tx;
            }
          } else if (warp == 1) {
            sent = static_cast<uint32_t>(kBHalfRows) * kBKBytes;
          } else if constexpr (P2) {
            sent = Cfg::kSfbBlocks * kSfSlabBytes;
          } else if constexpr (kMc) {
            sent = static_cast<uint32_t>(nsfb > crank ? (nsfb - crank + CL - 1) / CL : 0) * kSfSlabBytes;
          } else {
            sent = static_cast<uint32_t>(nsfb) * kSfSlabBytes;
          }
          ctl.rec_use[warp][stage] = count;
          ctl.rec_bytes[warp][stage] = sent;
        }
        ++count;
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // Stream-K finisher of a cluster plan (this CTA's last item is segment 0
    // of a split tile): warp 0 waits for the other segment's ready flags and
    // copies its fp32 partial (128 x BN, the workspace layout) into the ring,
    // piece by piece into the stages as the last MMAs release them, counted
    // on part_full.  The epilogue then reads it from shared memory instead of
    // waiting for L2 after its accumulator is complete.
    if constexpr (CL == 2 && !kRed) {
      if (warp == 0 && ok && any_item && x.nseg == 2 && x.seg == 0 && p.sched.sk_fixup) {
        const long long slot = x.tile - p.sched.dp_tiles;
        const char* src = reinterpret_cast<const char*>(p.workspace + slot * (BN * kBM));
        const int* flags = p.counters + slot * kEpiWarps;
        bool ready = true;
        if (lane == 0) {
          const uint64_t t0 = ptx::globaltimer();
          for (int f = 0; f < kEpiWarps && ready; ++f) {
            for (uint32_t i = 0; ptx::ld_acquire_gpu(flags + f) == 0; ++i) {
              if ((i & 7u) != 0) continue;
              if (ctl.abort) {
                ready = false;
                break;
              }
              if (ptx::globaltimer() - t0 > p.timeout_ns) {
                ctl.abort = 1;
                atomicCAS(p.status, 0, kStatusTimeoutProducer);
                ready = false;
                break;
              }
            }
          }
        }
        if (__shfl_sync(0xffffffffu, ready ? 1 : 0, 0)) {
          ptx::fence_proxy_async_global();  // the copies read what the flags published
          constexpr uint32_t kPartBytes = BN * kBM * 4;
          const uint32_t pbar = ptx::smem_addr(&ctl.part_full);
          ctl.part_armed = kPartBytes;
          ptx::mbar_arrive_expect_tx_elect(pbar, kPartBytes);
          for (uint32_t off = 0; off < kPartBytes;) {
            if (!warp_wait(W, empty_bar(stage), phase ^ 1u, kStatusTimeoutProducer)) break;
            const uint32_t n = kPartBytes - off < static_cast<uint32_t>(Cfg::kStageBytes) ? kPartBytes - off
                                                                                         : Cfg::kStageBytes;
            ptx::bulk_load_elect(smem_base + stage * Cfg::kStageBytes, src + off, n, pbar, pol_stream);
            ctl.part_issued = off + n;
            off += n;
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
    }
    // After an abort the copies still in flight are waited for at the end
    // of the kernel, from the records above (drain_after_abort).
  } else if (warp == kMmaWarp && (!P2 || crank == 0)) {
    // ------------------------------------------------------------ MMA issuer
    // Whole warp in the loop, one elected lane issues every tcgen05 operation
    // (always the same lane, so its commits track all of them).  In a 2-SM
    // pair only the even CTA's MMA warp runs; its MMAs, scale copies and
    // commits act on both CTAs.
    constexpr uint32_t idesc = make_idesc_nvf4(P2 ? 2 * kBM : kBM, BN);
    // Descriptors of stage 0.  Another stage, MMA k-block or scale atom
    // differs only in the start-address field (bits 0-13, address >> 4; every
    // address here is below 256 KB, so the field never carries), so the loop
    // adds constants instead of rebuilding 20 descriptors per k-tile: the
    // tensor pipe's queue is shallow, and the issue gap between two k-tiles'
    // MMAs is time the pipe sits idle.
    const uint64_t dA0 = operand_desc(smem_base);
    const uint64_t dB0 = operand_desc(smem_base + Cfg::kABytes);
    const uint64_t dSFA0 = scale_desc(smem_base + Cfg::kABytes + Cfg::kBBytes);
    const uint64_t dSFB0 = dSFA0 + (kSfSlabBytes >> 4);
    constexpr uint64_t kStageStep = Cfg::kStageBytes >> 4;
    constexpr uint64_t kAtomStep = kSfAtomBytes >> 4;
    constexpr uint64_t kSlabStep = kSfSlabBytes >> 4;
    constexpr uint64_t kKbStep = 32 >> 4;  // 64 E2M1 codes = 32 bytes per row per MMA
    static_assert(Cfg::kDynSmem + 2048 < (1 << 18), "shared addresses fit the 14-bit descriptor field");
    const uint32_t sf_tmem0 = tmem + Cfg::kSfBaseCol;
    const uint32_t mfull0 = full_bar(0), mempty0 = empty_bar(0);
    int stage = 0;
    uint32_t phase = 0;
    int ab = 0;
    uint32_t aphase = 0;
    bool ok = true;
    WorkCursor cur;
    work_begin(p.sched, unit, units, cur, wrank);
    Work x;
    while (ok && work_next(p.sched, unit, units, cur, x)) {
      if (!warp_wait(W, acc_empty_bar(ab), aphase ^ 1u, kStatusTimeoutMma)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after_sync();
      const uint32_t d_tmem = tmem + ab * BN;
      // A 64-wide tile uses the upper half of its 128-row B scale atom when
      // it starts at row 64 of the atom: column j holds rows 32j..32j+31
      // ("nvfp4 group gemm, submission 407526": sfb_lane).
      const uint32_t sfb_col0 = BN < 128 ? static_cast<uint32_t>((x.tn * BN) % 128 / 32) : 0u;
      for (int kt = x.kt0; kt < x.kt1; ++kt) {
        if (!warp_wait(W, mfull0 + 8u * stage, phase, kStatusTimeoutMma)) {
          ok = false;
          break;
        }
        // Scale slot = smem stage: the stage was refilled only after the MMAs
        // that last read this slot completed (they released the stage), so a
        // completed "full" phase also means the slot is free to overwrite.
        // No tcgen05 fence here: the copies and MMAs only read shared memory
        // that the completed phase made visible, and a fence per k-tile
        // would hold back the tensor pipe.
        const uint64_t so = static_cast<uint64_t>(stage) * kStageStep;
        const uint64_t dA = dA0 + so, dB = dB0 + so, dSFA = dSFA0 + so, dSFB = dSFB0 + so;
        const uint32_t sfa_t = sf_tmem0 + stage * Cfg::kSfSlotCols;
        const uint32_t sfb_t = sfa_t + Cfg::kSfaCols;
        // Per MMA k-block: its scale atoms -> tensor memory, then the MMA, so
        // the copies of k-block kb+1 can proceed while the MMA of kb runs.
        // Atom kb of a 128-row block holds the 4 scales of MMA k-block kb;
        // column j of it holds rows 32j..32j+31.
#pragma unroll
        for (int kb = 0; kb < kBK / kMmaK; ++kb) {
          // 64 E2M1 codes = 32 bytes per row per MMA: advance inside the swizzle row.
          const uint32_t acc = (kt > x.kt0 || kb > 0) ? 1u : 0u;
          ptx::tc_kblock_elect<P2 ? 2 : 1, Cfg::kSfbBlocks>(
              sfa_t + 4 * kb, dSFA + kb * kAtomStep, sfb_t + kb * Cfg::kSfbKbCols, dSFB + kb * kAtomStep,
              sfb_t + kb * Cfg::kSfbKbCols + 4, dSFB + kSlabStep + kb * kAtomStep, d_tmem, dA + kb * kKbStep,
              dB + kb * kKbStep, idesc, sfa_t + 4 * kb, sfb_t + kb * Cfg::kSfbKbCols + sfb_col0, acc);
        }
        if constexpr (P2)
          ptx::tc_commit2_mc_elect(mempty0 + 8u * stage, kPeers);  // the stage is free in both CTAs
        else if constexpr (!kMc)
          ptx::tc_commit_elect(mempty0 + 8u * stage);
        else
          ptx::tc_commit_mc_elect(mempty0 + 8u * stage, kPeers);  // the stage is free once both CTAs read it
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if constexpr (P2)
        ptx::tc_commit2_mc_elect(acc_full_bar(ab), kPeers);  // each CTA's epilogue drains its own rows
      else
        ptx::tc_commit_elect(acc_full_bar(ab));
      if (++ab == Cfg::kAccBufs) {
        ab = 0;
        aphase ^= 1u;
      }
    }
    if (!ok) {
      const uint32_t drain_bar = ptx::smem_addr(&ctl.mma_drain);
      if constexpr (P2)
        ptx::tc_commit2_mc_elect(drain_bar, 1);
      else
        ptx::tc_commit_elect(drain_bar);
      if (lane == 0) W.drain(drain_bar, 0);
      __syncwarp();
    }
  } else if (warp >= kFirstEpiWarp) {
    // ------------------------------------------------------------ epilogue
    ptx::griddep_wait();  // before any store or workspace access
    const int ew = warp - kFirstEpiWarp;  // epilogue warp 0..3
    const int sub = warp & 3;          // tensor-memory sub-partition this warp may read
    const int row = sub * 32 + lane;   // tile row owned by this thread
    const uint32_t gather_bar = ptx::smem_addr(&ctl.epi_gather);
    const uint32_t bcast_bar = ptx::smem_addr(&ctl.epi_bcast);
    int ab = 0;
    uint32_t aphase = 0;
    uint32_t gphase = 0;
    [[maybe_unused]] int red_items = 0;
    // Store 32 columns of this warp's 32 rows, packed as 16 half2 words per
    // thread: 64-byte-swizzled staging (16-byte chunk j of row r at chunk
    // j ^ ((r >> 1) & 3), conflict-free) and one TMA store of the 32 x 32 box.
    auto stage_and_store = [&](const Work& x, int col, const uint32_t* h, uint32_t sbuf) {
      const uint32_t row_addr = sbuf + lane * 64;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        st_shared_v4(row_addr + ((j ^ ((lane >> 1) & 3)) << 4), h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]);
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        ptx::tma_store_3d(&p.tmC[x.g], sbuf, x.tn * BN + col, x.tm * kBM + sub * 32, x.l);
        ptx::bulk_commit();
      }
    };
    // Through this warp's staging buffer: the store that last read it must
    // have read it before it is rewritten.
    auto store_box = [&](const Work& x, int col, const uint32_t* h) {
      const uint32_t sbuf = epi_base + ew * Cfg::kEpiBufBytes;
      if (lane == 0) ptx::bulk_wait_read<0>();
      __syncwarp();
      stage_and_store(x, col, h, sbuf);
    };
    auto store_chunk = [&](const Work& x, int q, const float* v) {
      uint32_t h[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) h[i] = pack_half2(v[2 * i], v[2 * i + 1]);
      store_box(x, 64 * q, h);
      store_box(x, 64 * q + 32, h + 16);
    };
    // Tensor memory -> registers, 64 columns of this thread's row.
    auto load_chunk = [&](uint32_t t_addr, float* v) {
      uint32_t r[64];
      ptx::tmem_load_32cols(t_addr, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
      ptx::tmem_load_32cols(t_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
      ptx::tmem_load_wait();
      ptx::reg_fence32(&r[0]);
      ptx::reg_fence32(&r[32]);
#pragma unroll
      for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
    };

    WorkCursor cur;
    work_begin(p.sched, unit, units, cur, wrank);
    Work x;
    [[maybe_unused]] uint32_t kt_seen = 0;  // k-tiles of this CTA's work list so far (current item included)
    while (work_next(p.sched, unit, units, cur, x)) {
      kt_seen += static_cast<uint32_t>(x.kt1 - x.kt0);
      // This CTA's last work item?  Once its accumulator is complete every
      // MMA of the CTA (and of its cluster peer's shared tiles) has read its
      // stage, and no copy will land in the ring again.
      WorkCursor peek = cur;
      Work next_x;
      const bool last_item = !work_next(p.sched, unit, units, peek, next_x);
      if (!warp_wait(W, acc_full_bar(ab), aphase, kStatusTimeoutEpilogue)) break;
      ptx::tc_fence_after_sync();
      const uint32_t t_row = tmem + (static_cast<uint32_t>(sub * 32) << 16) + ab * BN;
      const bool rows_live = x.tm * kBM + sub * 32 < p.M[x.g];  // else the whole box is past M
      const int my_ab = ab;
      if (++ab == Cfg::kAccBufs) {
        ab = 0;
        aphase ^= 1u;
      }
      auto release_acc = [&]() {
        ptx::tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          // A pair's accumulator barrier lives in the even CTA, whose MMAs
          // overwrite both CTAs' accumulators.  The arrival publishes only
          // that this warp's tensor-memory reads are complete, so the odd
          // CTA's remote arrival needs no cluster-scope release.
          if (P2 && crank != 0)
            ptx::mbar_arrive_remote(ptx::mapa_shared(acc_empty_bar(my_ab), 0));
          else
            ptx::mbar_arrive(acc_empty_bar(my_ab));
        }
      };

      if (x.nseg == 1) {
        // Drain the whole accumulator row into registers as fp16 first and
        // release it, so the next tile's MMAs start while this one is stored.
        // 128 columns per tensor-memory wait (four loads in flight), so a
        // 256-wide accumulator is drained in two round trips, not four.
        uint32_t h[BN / 2];
        constexpr int kDrainCols = BN < 128 ? BN : 128;
#pragma unroll
        for (int q = 0; q < BN / kDrainCols; ++q) {
          uint32_t r[kDrainCols];
#pragma unroll
          for (int c = 0; c < kDrainCols / 32; ++c)
            ptx::tmem_load_32cols(t_row + kDrainCols * q + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&r[32 * c]));
          ptx::tmem_load_wait();
#pragma unroll
          for (int c = 0; c < kDrainCols / 32; ++c) ptx::reg_fence32(&r[32 * c]);
#pragma unroll
          for (int i = 0; i < kDrainCols / 2; ++i)
            h[kDrainCols / 2 * q + i] = pack_half2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
        }
        release_acc();
        if (rows_live) {
          if (last_item) {
            // The ring is idle: every box gets its own staging buffer there, so
            // the warp's stores go out back to back instead of each waiting for
            // the previous one to leave the warp's single buffer (the last
            // tile's epilogue is the kernel's tail).
            static_assert(kEpiWarps * (BN / 32) * Cfg::kEpiBufBytes <= kStages * Cfg::kStageBytes,
                          "final staging exceeds the ring");
#pragma unroll
            for (int c = 0; c < BN / 32; ++c)
              stage_and_store(x, 32 * c, &h[16 * c], smem_base + (ew * (BN / 32) + c) * Cfg::kEpiBufBytes);
          } else {
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) store_box(x, 32 * c, &h[16 * c]);
          }
        }
        continue;
      }

      if constexpr (CL == 2 && !kRed) {
        // Stream-K tile of a CTA pair (the schedule's sk_fixup): exactly two
        // segments, each CTA handling its own 128 rows.  Segment 1 -- the
        // tile's last k-tiles, its cluster's first stream-K item -- stores its
        // fp32 partial ([BN/4][128 rows][4], 16 bytes of a row per thread) and
        // sets one ready flag per epilogue warp.  Segment 0 -- the first
        // k-tiles, its cluster's last item -- waits for the flag of its warp's
        // rows, adds the partial to its accumulator (two addends, so the sum
        // does not depend on which segment finished first) and stores the
        // tile, staged in the idle ring.
        if (x.nseg != 2 || !p.sched.sk_fixup) {
          if (lane == 0) {
            ctl.abort = 1;
            atomicCAS(p.status, 0, kStatusBadClusterPlan);
          }
          release_acc();
          break;
        }
        const long long slot = x.tile - p.sched.dp_tiles;
        float4* ws = reinterpret_cast<float4*>(p.workspace) + slot * (BN / 4 * kBM) + row;
        int* flag = p.counters + slot * kEpiWarps + ew;
        if (x.seg != 0) {
#pragma unroll 1
          for (int q = 0; q < BN / 64; ++q) {
            float v[64];
            load_chunk(t_row + 64 * q, v);
#pragma unroll
            for (int c4 = 0; c4 < 16; ++c4)
              __stcg(ws + (16 * q + c4) * kBM, make_float4(v[4 * c4], v[4 * c4 + 1], v[4 * c4 + 2], v[4 * c4 + 3]));
          }
          release_acc();
          __threadfence();
          __syncwarp();
          if (lane == 0) ptx::st_release_gpu(flag, 1);
          continue;
        }
        // Segment 0: the producer copied the partial into the ring, piece j
        // into the stage after this CTA's last k-tile plus j (kt_seen counts
        // every k-tile of this CTA's work list).  Each 32-column box is summed,
        // staged in ring space the partial does not use (the stages after the
        // pieces, then the tail of the last piece's stage; the warp's own
        // buffer if neither has room) and stored at once.
        if (!warp_wait(W, ptx::smem_addr(&ctl.part_full), 0, kStatusTimeoutEpilogue)) {
          release_acc();
          break;
        }
        {
          constexpr uint32_t kPartBytes = BN * kBM * 4;
          constexpr uint32_t kPieces = (kPartBytes + Cfg::kStageBytes - 1) / Cfg::kStageBytes;
          static_assert(kPieces <= static_cast<uint32_t>(kStages), "partial larger than the ring");
          constexpr uint32_t kLastPiece = kPartBytes - (kPieces - 1) * Cfg::kStageBytes;
          constexpr uint32_t kBoxesPerStage = Cfg::kStageBytes / Cfg::kEpiBufBytes;
          constexpr uint32_t kFreeBoxes = (kStages - kPieces) * kBoxesPerStage;
          constexpr uint32_t kTailOff = (kLastPiece + Cfg::kEpiBufBytes - 1) / Cfg::kEpiBufBytes * Cfg::kEpiBufBytes;
          constexpr uint32_t kTailBoxes = (Cfg::kStageBytes - kTailOff) / Cfg::kEpiBufBytes;
#pragma unroll 1
          for (int q = 0; q < BN / 32; ++q) {
            uint32_t r[32];
            ptx::tmem_load_32cols(t_row + 32 * q, r);
            ptx::tmem_load_wait();
            ptx::reg_fence32(r);
            uint32_t hq[16];
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
              const uint32_t o = ((8 * q + c4) * kBM + row) * 16;
              const float4 t = ld_shared_v4(smem_base + ((kt_seen + o / Cfg::kStageBytes) % kStages) * Cfg::kStageBytes +
                                            o % Cfg::kStageBytes);
              hq[2 * c4] = pack_half2(__uint_as_float(r[4 * c4]) + t.x, __uint_as_float(r[4 * c4 + 1]) + t.y);
              hq[2 * c4 + 1] = pack_half2(__uint_as_float(r[4 * c4 + 2]) + t.z, __uint_as_float(r[4 * c4 + 3]) + t.w);
            }
            if (!rows_live) continue;
            const uint32_t b = ew * (BN / 32) + q;  // box index in the CTA
            if (b < kFreeBoxes) {
              stage_and_store(x, 32 * q, hq,
                              smem_base + ((kt_seen + kPieces + b / kBoxesPerStage) % kStages) * Cfg::kStageBytes +
                                  (b % kBoxesPerStage) * Cfg::kEpiBufBytes);
            } else if (b - kFreeBoxes < kTailBoxes) {
              stage_and_store(x, 32 * q, hq,
                              smem_base + ((kt_seen + kPieces - 1) % kStages) * Cfg::kStageBytes + kTailOff +
                                  (b - kFreeBoxes) * Cfg::kEpiBufBytes);
            } else {
              store_box(x, 32 * q, hq);
            }
          }
        }
        release_acc();
        // partial consumed: ready for the next launch; drop its L2 lines
        if (lane == 0) *flag = 0;
        const char* base = reinterpret_cast<const char*>(reinterpret_cast<const float4*>(p.workspace) +
                                                         slot * (BN / 4 * kBM) + sub * 32);
        for (int line = lane; line < (BN / 4) * 4; line += 32)
          ptx::discard_l2(base + static_cast<size_t>(line >> 2) * (kBM * 16) + (line & 3) * 128);
        continue;
      }

      if constexpr (kRed) {
        // The CL segments of this tile are the CL CTAs of this cluster (rank
        // = segment) and each CTA reduces and stores BN/CL of the columns.
        // The operand ring, idle once a CTA's only work item is done, holds
        // CL receive slots (slot j: segment j's fp32 partial of this CTA's
        // columns) and then CL staging slots (staging slot r: this CTA's
        // partial of rank r's columns).  A slot is laid out by epilogue warp:
        // [warp][column / 4][row % 32][4 floats], so each warp's 32 rows are
        // one contiguous part of kSlotBytes / 4.  Every warp drains its rows
        // into its own receive slot and the staging slots -- the other ranks'
        // columns first -- and, once every CTA of the cluster is idle, bulk-
        // copies its part of each staging slot into the owner's receive slot,
        // where the owner's red_full barrier counts the bytes; the warps'
        // copies run side by side and overlap the draining of the CTA's own
        // columns.  The owner sums the CL slots in segment (= k) order, as
        // the workspace path does.  Each thread reads back only its own row.
        constexpr int kOwnCols = BN / CL;
        constexpr uint32_t kSlotBytes = kOwnCols * kBM * 4;
        constexpr uint32_t kWarpPart = kSlotBytes / kEpiWarps;
        static_assert(kOwnCols % 32 == 0, "whole 32-column boxes per CTA");
        static_assert(2 * CL * kSlotBytes + kEpiWarps * (kOwnCols / 32) * Cfg::kEpiBufBytes <= kStages * Cfg::kStageBytes,
                      "reduction slots and C staging exceed the ring");
        if (x.nseg != CL || x.seg != crank || red_items++ != 0) {
          if (lane == 0) {
            ctl.abort = 1;
            atomicCAS(p.status, 0, kStatusBadClusterPlan);
          }
          release_acc();
          break;
        }
        const uint32_t go_bar = ptx::smem_addr(&ctl.red_go);
        const uint32_t rfull_bar = ptx::smem_addr(&ctl.red_full);
        // This CTA's MMAs are complete (acc_full), so its ring may be
        // written: tell every CTA of the cluster.
        if (ew == 0 && lane < CL) ptx::mbar_arrive_remote(ptx::mapa_shared(go_bar, static_cast<uint32_t>(lane)));
        if (ew == 0 && lane == 0) {
          ptx::mbar_arrive_expect_tx(rfull_bar, (CL - 1) * kSlotBytes);
          ctl.red_armed = 1;
        }
        // receive slot of this CTA's columns, staging slot of rank r's
        auto slot_of = [&](int r) {
          return smem_base + static_cast<uint32_t>(r == static_cast<int>(crank) ? r : CL + r) * kSlotBytes;
        };
        const uint32_t part = static_cast<uint32_t>(sub) * kWarpPart + static_cast<uint32_t>(lane) * 16;
        bool sent_ok = true;
        auto send_parts = [&]() {
          // every lane's staging stores visible to the bulk copies, every
          // CTA of the cluster idle, then one copy per other rank
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (!warp_wait<true>(W, go_bar, 0, kStatusTimeoutEpilogue)) {
            sent_ok = false;
            return;
          }
          if (lane == 0) {
#pragma unroll
            for (int r = 0; r < CL; ++r)
              if (r != static_cast<int>(crank)) {
                ptx::bulk_copy_to_cluster(
                    ptx::mapa_shared(smem_base + crank * kSlotBytes + sub * kWarpPart, static_cast<uint32_t>(r)),
                    smem_base + static_cast<uint32_t>(CL + r) * kSlotBytes + sub * kWarpPart, kWarpPart,
                    ptx::mapa_shared(rfull_bar, static_cast<uint32_t>(r)));
                ctl.red_sent[sub] |= 1u << r;
              }
          }
          __syncwarp();
        };
        // 64-column chunks, the other ranks' first: with two ranks, the
        // peer's half is sent while this CTA's own half is drained
        constexpr int kChunks = BN / 64;
#pragma unroll
        for (int qi = 0; qi < kChunks; ++qi) {
          const int q = CL == 2 ? (qi + (crank == 0 ? 1 : 0)) % kChunks : qi;
          float v[64];
          load_chunk(t_row + 64 * q, v);
#pragma unroll
          for (int c4 = 0; c4 < 16; ++c4) {
            const int col = 64 * q + 4 * c4;
            st_shared_v4(slot_of(col / kOwnCols) + part + (col % kOwnCols) / 4 * 512, __float_as_uint(v[4 * c4]),
                         __float_as_uint(v[4 * c4 + 1]), __float_as_uint(v[4 * c4 + 2]),
                         __float_as_uint(v[4 * c4 + 3]));
          }
          if (CL == 2 && qi == 0) send_parts();
        }
        release_acc();
        if (CL != 2) send_parts();
        if (!sent_ok) break;
        if (!warp_wait(W, rfull_bar, 0, kStatusTimeoutEpilogue)) break;
#pragma unroll
        for (int cg = 0; cg < kOwnCols / 32; ++cg) {
          float4 acc[8];
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) acc[c4] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int j = 0; j < CL; ++j)
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
              const float4 t = ld_shared_v4(smem_base + j * kSlotBytes + part + (cg * 8 + c4) * 512);
              acc[c4].x += t.x;
              acc[c4].y += t.y;
              acc[c4].z += t.z;
              acc[c4].w += t.w;
            }
          uint32_t hs[16];
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            hs[2 * c4] = pack_half2(acc[c4].x, acc[c4].y);
            hs[2 * c4 + 1] = pack_half2(acc[c4].z, acc[c4].w);
          }
          // every box its own staging buffer in the idle ring, past the slots
          if (rows_live)
            stage_and_store(x, crank * kOwnCols + 32 * cg, hs,
                            smem_base + 2 * CL * kSlotBytes + (ew * (kOwnCols / 32) + cg) * Cfg::kEpiBufBytes);
        }
        continue;
      }

      // Stream-K segment: publish this partial tile as [BN/4][128 rows][4]
      // fp32, so each thread stores (and later loads) 16 bytes of its row and
      // a warp touches 512 contiguous bytes per column group.
      float4* ws = reinterpret_cast<float4*>(p.workspace) + sk_slot(p.sched, x, x.seg) * (BN / 4 * kBM) + row;
#pragma unroll 1
      for (int q = 0; q < BN / 64; ++q) {
        float v[64];
        load_chunk(t_row + 64 * q, v);
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4)
          __stcg(ws + (16 * q + c4) * kBM, make_float4(v[4 * c4], v[4 * c4 + 1], v[4 * c4 + 2], v[4 * c4 + 3]));
      }
      release_acc();
      __threadfence();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(gather_bar);
      bool ok = true;
      const int ctr = sk_counter(p.sched, x);
      if (ew == 0) {
        ok = warp_wait(W, gather_bar, gphase, kStatusTimeoutEpilogue);
        if (ok && lane == 0) {
          __threadfence();
          const int old = atomicAdd(&p.counters[ctr], 1);
          const int last = (old == x.nseg - 1) ? 1 : 0;
          if (last) __threadfence();
          ctl.last_flag = last;
          ptx::mbar_arrive(bcast_bar);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (!warp_wait(W, bcast_bar, gphase, kStatusTimeoutEpilogue)) break;
      gphase ^= 1u;
      if (!ctl.last_flag) continue;
      __threadfence();
      // Last segment to finish: sum the segments' partials in k order (0, 1,
      // ...), so the result does not depend on which segment finished last.
      const float4* ws0 = reinterpret_cast<const float4*>(p.workspace) + sk_slot(p.sched, x, 0) * (BN / 4 * kBM) + row;
      constexpr int kMaxSeg = 4;  // loads of up to 4 segments in flight at once
      // Sum 128 columns at a time into packed fp16 registers before storing
      // them, so the loads of all four 32-column groups are in flight together.
      constexpr int kPassCols = BN < 128 ? BN : 128;
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += kPassCols) {
        uint32_t hs[kPassCols / 2];
#pragma unroll
        for (int c = 0; c < kPassCols / 32; ++c) {  // 32-column groups
          float4 acc[8];
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) acc[c4] = make_float4(0.f, 0.f, 0.f, 0.f);
          const int cg = c0 / 4 + 8 * c;  // first 4-column group of this 32-column group
          for (int j0 = 0; j0 < x.nseg; j0 += kMaxSeg) {
            float4 part[kMaxSeg][8];
#pragma unroll
            for (int j = 0; j < kMaxSeg; ++j)
#pragma unroll
              for (int c4 = 0; c4 < 8; ++c4)
                part[j][c4] = (j0 + j < x.nseg)
                    ? __ldcg(ws0 + static_cast<size_t>(j0 + j) * (BN / 4 * kBM) + (cg + c4) * kBM)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int j = 0; j < kMaxSeg; ++j)
              if (j0 + j < x.nseg)
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4) {
                  acc[c4].x += part[j][c4].x;
                  acc[c4].y += part[j][c4].y;
                  acc[c4].z += part[j][c4].z;
                  acc[c4].w += part[j][c4].w;
                }
          }
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            hs[16 * c + 2 * c4] = pack_half2(acc[c4].x, acc[c4].y);
            hs[16 * c + 2 * c4 + 1] = pack_half2(acc[c4].z, acc[c4].w);
          }
        }
        if (rows_live) {
#pragma unroll
          for (int c = 0; c < kPassCols / 32; ++c) store_box(x, c0 + 32 * c, &hs[16 * c]);
        }
      }
      // The partials are consumed: drop their L2 lines without writing them
      // back.  This warp read exactly the lines of its own 32 rows.
      __syncwarp();
      for (int j = 0; j < x.nseg; ++j) {
        const char* base = reinterpret_cast<const char*>(
            reinterpret_cast<const float4*>(p.workspace) + sk_slot(p.sched, x, j) * (BN / 4 * kBM) + sub * 32);
        for (int line = lane; line < (BN / 4) * 4; line += 32)  // (BN/4) column groups x 4 lines of 128 B
          ptx::discard_l2(base + static_cast<size_t>(line >> 2) * (kBM * 16) + (line & 3) * 128);
      }
      if (ew == 0 && lane == 0) p.counters[ctr] = 0;  // ready for the next launch
    }
    if (lane == 0) ptx::bulk_wait<0>();
    __syncwarp();
  }

  ptx::tc_fence_before_sync();
  __syncthreads();
  // No CTA leaves while a peer may still multicast into its shared memory or
  // signal its barriers.  Every CTA publishes its abort flag to all CTAs of
  // the cluster before the barrier, so the decision to drain below is the
  // same in every CTA.
  bool drain = ctl.abort != 0;
  if constexpr (CL > 1) {
    if (threadIdx.x < CL)
      ptx::st_shared_cluster(ptx::mapa_shared(ptx::smem_addr(&ctl.peer_abort[crank]), threadIdx.x),
                             static_cast<uint32_t>(ctl.abort));
    ptx::cluster_sync();
#pragma unroll
    for (int r = 0; r < CL; ++r) drain = drain || ctl.peer_abort[r] != 0;
  }
  if (drain) {
    // After an abort, copies may still be in flight into this CTA's shared
    // memory: wait for them, counted, before it is released.
    if (threadIdx.x == 0) drain_after_abort();
    __syncthreads();
    if constexpr (CL > 1) ptx::cluster_sync();
  }
  ptx::tc_fence_after_sync();
  if (warp == kMmaWarp) {
    if constexpr (P2)
      ptx::tmem_dealloc2(tmem, Cfg::kTmemCols);
    else
      ptx::tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

// ---------------------------------------------------------------- launcher
template <int BN, int CL, int MODE>
static cudaError_t launch_bn(const GemmParams& p, int grid, cudaStream_t stream, bool pdl) {
  using Cfg = TileCfg<BN, MODE == kModePair>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kNumThreads, 1, 1);
  cfg.dynamicSmemBytes = Cfg::kDynSmem;
  cfg.stream = stream;
  // Programmatic dependent launch: this grid may start while the previous
  // kernel on the stream finishes; the kernel waits for it (griddepcontrol)
  // before its first global-memory access.
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (CL > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = CL;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, nvfp4_gemm_kernel<BN, CL, MODE>, p);
}

template <int BN, int CL, int MODE>
static cudaError_t prepare_bn() {
  return cudaFuncSetAttribute(nvfp4_gemm_kernel<BN, CL, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              TileCfg<BN, MODE == kModePair>::kDynSmem);
}

// Largest number of co-resident clusters of CL CTAs (0 on error).
template <int BN, int CL, int MODE>
static int max_clusters_bn() {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CL * 1024, 1, 1);
  cfg.blockDim = dim3(kNumThreads, 1, 1);
  cfg.dynamicSmemBytes = TileCfg<BN, MODE == kModePair>::kDynSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, nvfp4_gemm_kernel<BN, CL, MODE>, &cfg) != cudaSuccess) return 0;
  return n;
}

cudaError_t gemm_prepare_device(int bn) {
  cudaError_t e;
  switch (bn) {
    case 64: return prepare_bn<64, 1, kModeSingle>();
    case 128:
      if ((e = prepare_bn<128, 1, kModeSingle>()) != cudaSuccess) return e;
      if ((e = prepare_bn<128, 2, kModeMulticast>()) != cudaSuccess) return e;
      if ((e = prepare_bn<128, 2, kModeReduce>()) != cudaSuccess) return e;
      return prepare_bn<128, 4, kModeReduce>();
    case 256:
      if ((e = prepare_bn<256, 1, kModeSingle>()) != cudaSuccess) return e;
      if ((e = prepare_bn<256, 2, kModeMulticast>()) != cudaSuccess) return e;
      return prepare_bn<256, 2, kModePair>();
    default: return cudaErrorInvalidValue;
  }
}

// Launch of the variant for (BN, mode, cluster size); cudaErrorInvalidValue for
// combinations that are not instantiated.
cudaError_t gemm_launch(int bn, int cluster, int mode, const GemmParams& p, int grid, cudaStream_t stream,
                        bool pdl) {
  switch (mode) {
    case kModeSingle:
      if (cluster != 1) break;
      switch (bn) {
        case 64: return launch_bn<64, 1, kModeSingle>(p, grid, stream, pdl);
        case 128: return launch_bn<128, 1, kModeSingle>(p, grid, stream, pdl);
        case 256: return launch_bn<256, 1, kModeSingle>(p, grid, stream, pdl);
        default: break;
      }
      break;
    case kModeMulticast:
      if (cluster != 2) break;
      if (bn == 128) return launch_bn<128, 2, kModeMulticast>(p, grid, stream, pdl);
      if (bn == 256) return launch_bn<256, 2, kModeMulticast>(p, grid, stream, pdl);
      break;
    case kModePair:
      if (cluster == 2 && bn == 256) return launch_bn<256, 2, kModePair>(p, grid, stream, pdl);
      break;
    case kModeReduce:
      if (bn != 128) break;
      if (cluster == 2) return launch_bn<128, 2, kModeReduce>(p, grid, stream, pdl);
      if (cluster == 4) return launch_bn<128, 4, kModeReduce>(p, grid, stream, pdl);
      break;
    default: break;
  }
  return cudaErrorInvalidValue;
}

int gemm_max_clusters(int bn, int cluster, int mode) {
  switch (mode) {
    case kModeMulticast:
      if (cluster != 2) return 0;
      return bn == 256 ? max_clusters_bn<256, 2, kModeMulticast>() : bn == 128 ? max_clusters_bn<128, 2, kModeMulticast>() : 0;
    case kModePair:
      return (cluster == 2 && bn == 256) ? max_clusters_bn<256, 2, kModePair>() : 0;
    case kModeReduce:
      if (bn != 128) return 0;
      return cluster == 2 ? max_clusters_bn<128, 2, kModeReduce>() : cluster == 4 ? max_clusters_bn<128, 4, kModeReduce>() : 0;
    default: return 0;
  }
}

int gemm_stages(int bn, bool pair) {
  if (pair) return bn == 256 ? TileCfg<256, true>::kStages : 0;
  switch (bn) {
    case 64: return TileCfg<64>::kStages;
    case 128: return TileCfg<128>::kStages;
    case 256: return TileCfg<256>::kStages;
    default: return 0;
  }
}

}  // namespace nvfp4
