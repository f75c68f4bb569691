// Kernel parameter block and compile-time tiling shared by the host launcher
// and the device kernel of libnvfp4gemm.  Internal: not part of the C ABI.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "schedule.h"

namespace nvfp4 {

constexpr int kMaxGroups = 8;

// One CTA tile: 128 rows of A (the tcgen05 M=128 shape), BN rows of B, and
// 256 K-elements per pipeline stage (128 bytes of packed E2M1 per row, i.e. one
// 128-byte swizzle row).  "nvfp4 gemm, submission 125598" and
// "nvfp4_group_gemm, submission 498453" use a 128x128x256 MMA tiler; that is
// kept as the base tile here.
constexpr int kBM = 128;
constexpr int kBK = 256;
constexpr int kBKBytes = kBK / 2;          // 128 B per row per k-tile
constexpr int kMmaK = 64;                  // K of one kind::mxf4nvf4 MMA
constexpr int kSfAtomBytes = 512;          // 128 rows x 4 scales
constexpr int kSfSlabBytes = 4 * kSfAtomBytes;  // one 128-row block, one k-tile

// Warp roles: kProducerWarps TMA producers, one MMA warp, four epilogue warps
// (one per 32-lane tensor-memory sub-partition): 8 warps, two warpgroups.
constexpr int kProducerWarps = 3;  // warp 0: A + SFA, warp 1: B, warp 2: SFB
constexpr int kMmaWarp = kProducerWarps;
constexpr int kFirstEpiWarp = kProducerWarps + 1;
constexpr int kEpiWarps = 4;
constexpr int kNumThreads = 32 * (kProducerWarps + 1 + kEpiWarps);

// Status codes a kernel may leave in the device status word.
constexpr int kStatusTimeoutProducer = 1;
constexpr int kStatusTimeoutMma = 2;
constexpr int kStatusTimeoutEpilogue = 3;
constexpr int kStatusBadClusterPlan = 4;  // cluster reduction launched on a plan it does not fit

// Kernel variants (template MODE; CL = CTAs per cluster):
//   kModeSingle     CL = 1, one CTA per tile
//   kModeMulticast  CL = 2, tiles 2q, 2q+1 of the same B columns share B by TMA multicast
//   kModePair       CL = 2, the same two tiles as one 256-row tile of 2-SM MMAs
//   kModeReduce     CL = S, the S stream-K segments of one tile, summed through
//                   distributed shared memory instead of a global workspace
constexpr int kModeSingle = 0;
constexpr int kModeMulticast = 1;
constexpr int kModePair = 2;
constexpr int kModeReduce = 3;

// Host-built parameter block, passed by value as a __grid_constant__ kernel
// parameter: the tensor maps live in the parameter space and need no device
// allocation or copy (the pages keep them in a device blob instead).
struct GemmParams {
  CUtensorMap tmA[kMaxGroups];   // uint8 {K/2, M, L}, box {128, 128, 1}, 128B swizzle
  CUtensorMap tmB[kMaxGroups];   // uint8 {K/2, N, L}, box {128, BN, 1}, 128B swizzle
  CUtensorMap tmC[kMaxGroups];   // fp16 {N, M, L}, box {32, 32, 1}, 64B swizzle
  // Repacked scales as uint8 {256, bytes/256}, box {256, 8} = one 2 KB slab.
  // Encoded only for 2-SM pair launches, whose copies must signal the pair's
  // leader CTA (only the tensor form of the bulk copy can).
  CUtensorMap tmSFA[kMaxGroups];
  CUtensorMap tmSFB[kMaxGroups];
  const uint8_t* sfa[kMaxGroups];  // repacked scales
  const uint8_t* sfb[kMaxGroups];
  int M[kMaxGroups], N[kMaxGroups];
  int sf_rows_a[kMaxGroups];     // ceil(M/128): 128-row scale blocks per batch
  int sf_rows_b[kMaxGroups];     // ceil(N/128)
  int a_streams[kMaxGroups];     // 1: A is the streamed operand (evict-first), B kept
  Schedule sched;                // data-parallel + stream-K work decomposition
  float* workspace;              // stream-K partials, [slot][BN/4][128][4] fp32
  int* counters;                 // per stream-K tile arrival counters (zero between launches)
  int* status;                   // device status word
  unsigned long long timeout_ns; // limit of every bounded wait
  int debug_skip_ktile;          // test-only fault injection (-1 = off)
  int prefetch_ktiles;           // k-tiles per CTA prefetched into L2 before the launch dependency wait
};

// Per-BN compile-time configuration.  P2: 2-SM pair tiles (tcgen05
// cta_group::2, M = 256 across the two CTAs of a cluster): each CTA holds its
// 128 rows of A, half of the BN rows of B and the B scales of all BN rows.
template <int BN, bool P2 = false>
struct TileCfg {
  static constexpr int kBN = BN;
  static constexpr int kABytes = kBM * kBKBytes;               // 16 KB
  static constexpr int kBBytes = (P2 ? BN / 2 : BN) * kBKBytes; // B rows held by this CTA x 128 B
  static constexpr int kSfbBlocks = (BN + 127) / 128;          // 128-row scale blocks
  static constexpr int kStageBytes = kABytes + kBBytes + kSfSlabBytes + kSfbBlocks * kSfSlabBytes;
  // Epilogue staging: one 32 rows x 32 fp16 box (64-byte swizzle) per
  // epilogue warp, so that shared memory goes to the operand ring instead
  // (4 stages at BN = 256, 6 at BN = 128, 5 for 2-SM pairs at BN = 256).
  static constexpr int kEpiBoxCols = 32;
  static constexpr int kEpiBufBytes = 32 * kEpiBoxCols * 2;     // 2 KB
  static constexpr int kEpiBytes = kEpiWarps * kEpiBufBytes;
  static constexpr int kSmemBudget = 227 * 1024 - 1024;          // minus static shared memory
  static constexpr int kStages = (kSmemBudget - kEpiBytes - 1024) / kStageBytes;
  static constexpr int kDynSmem = kStages * kStageBytes + kEpiBytes + 1024;  // +1024 alignment slack
  // Tensor memory: accumulators first, then a ring of scale slots.
  static constexpr int kAccBufs = (BN <= 128) ? 2 : 1;
  static_assert(BN == 64 || BN % 128 == 0, "tile widths: 64, 128, 256");
  static_assert(!P2 || BN == 256, "2-SM pair tiles are 256 x 256");
  static constexpr int kSfaCols = 4 * (kBK / kMmaK);               // 16 per k-tile
  // B scale columns per MMA k-block: BN/32, but a whole 4-column atom is
  // copied even when the tile is narrower than the 128-row atom (BN = 64: the
  // MMA reads the half of the atom that holds its rows).
  static constexpr int kSfbKbCols = BN / 32 > 4 ? BN / 32 : 4;
  static constexpr int kSfbCols = kSfbKbCols * (kBK / kMmaK);
  static constexpr int kSfSlots = kStages;  // one tensor-memory scale slot per smem stage
  static constexpr int kSfSlotCols = kSfaCols + kSfbCols;
  static constexpr int kSfBaseCol = kAccBufs * BN;
  static constexpr int kTmemCols = 512;
  static_assert(kSfBaseCol + kSfSlots * kSfSlotCols <= kTmemCols, "tensor memory overflow");
  static_assert(kStages >= 2, "not enough shared memory for two stages");
};

}  // namespace nvfp4
