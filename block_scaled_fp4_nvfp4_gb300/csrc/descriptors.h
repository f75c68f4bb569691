// Bit-field encoders for the two tcgen05 descriptors the GEMM builds: the
// shared-memory matrix descriptor and the block-scaled MMA instruction
// descriptor.  Field positions follow the PTX ISA tables for tcgen05 (sm_100
// family).  "nvfp4 group gemm, submission 407526" builds the same two words
// for M=128, N=64 (grouped_kernel, MMA warp: make_desc_AB / make_desc_SF and
// i_desc); its values are the host-side check of these encoders.
#pragma once

#include <stdint.h>

namespace nvfp4 {

// Shared-memory matrix descriptor.
//   bits  0-13  start address >> 4
//   bits 16-29  leading-dimension byte offset >> 4 (not used by the layouts
//               here: K-major 128B-swizzled tiles and 16-byte-row scale atoms)
//   bits 32-45  stride-dimension byte offset >> 4: distance between
//               consecutive 8-row core-matrix groups
//   bits 46-48  fixed value 0b001
//   bits 49-51  base offset (0: every tile starts 1024-byte aligned)
//   bits 61-63  layout: 0 = no swizzle, 2 = 128-byte swizzle
enum SmemLayout : uint32_t { kNoSwizzle = 0, kSwizzle128B = 2 };

__host__ __device__ constexpr uint64_t make_smem_desc(uint32_t smem_addr, uint32_t sbo_bytes,
                                                      uint32_t layout) {
  return (static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4)) |
         (static_cast<uint64_t>((sbo_bytes & 0x3FFFFu) >> 4) << 32) | (1ull << 46) |
         (static_cast<uint64_t>(layout & 7u) << 61);
}

// K-major operand tile, 128 bytes (256 E2M1 codes) per row, 128-byte swizzle:
// 8-row groups are 1024 bytes apart.
__host__ __device__ constexpr uint64_t operand_desc(uint32_t smem_addr) {
  return make_smem_desc(smem_addr, 1024, kSwizzle128B);
}

// Scale atom: 32 rows x 16 bytes, unswizzled, 8-row groups 128 bytes apart.
__host__ __device__ constexpr uint64_t scale_desc(uint32_t smem_addr) {
  return make_smem_desc(smem_addr, 128, kNoSwizzle);
}

// Instruction descriptor for tcgen05.mma .kind::mxf4nvf4 (block-scaled).
//   bits  4-5   B scale-factor id (0)
//   bits  7-9   A format: 1 = E2M1
//   bits 10-12  B format: 1 = E2M1
//   bits 13,14  negate A / B (0)
//   bits 15,16  A / B major-ness (0 = K-major)
//   bits 17-22  N >> 3
//   bit  23     scale format: 0 = UE4M3 (block of 16), 1 = UE8M0
//   bits 27-28  M >> 7
//   bits 29-30  A scale-factor id (0)
__host__ __device__ constexpr uint32_t make_idesc_nvf4(int M, int N) {
  return (1u << 7) | (1u << 10) | ((static_cast<uint32_t>(N) >> 3) << 17) | (0u << 23) |
         ((static_cast<uint32_t>(M) >> 7) << 27);
}

}  // namespace nvfp4
