// Fused NVFP4 quantization: bf16 / fp16 values -> packed E2M1 codes plus E4M3
// block scales written directly in the repacked (tensor-core atom) layout that
// the GEMM reads, so no row-major scale array and no separate repack pass.
//
// The pages take A, B and their scales already quantized and print no
// quantizer; the recipe is the plainest reading of the formats they name (E2M1
// codes, one E4M3 scale per 16 consecutive values along K), in IEEE fp32:
//   amax = max |x_i| over a block of 16;  sf = E4M3(amax / 6), round to nearest
//   even, finite values above 448 give 448;  d = value of sf;
//   code_i = E2M1(x_i / d), round to nearest even on {0, .5, 1, 1.5, 2, 3, 4, 6},
//   magnitudes above 6 give 6, sign of x_i / d kept;  d = 0 gives code 0.
//
// Work split: one warp per (batch, 128-row block, 64-value chunk of K), i.e. per
// 512-byte scale atom.  Eight lanes read one row's 128 bytes together (one full
// line per 8 lanes, 512 contiguous bytes per warp load, 32 contiguous bytes of
// codes per row per store); lanes 2b and 2b+1 hold 16-value block b and
// combine their maxima with one shuffle.  The atom is assembled in shared
// memory (byte (r % 32) * 16 + ((r % 128) / 32) * 4 + block % 4) and stored
// with one 16-byte store per lane.  Atoms of the padding (rows past the last
// row, k past K up to the 256-wide k-tile) come out zero.  The grid is one
// wave of resident blocks walking the atoms.
//
// x / d without a full division per value: r = 1/d correctly rounded once per
// block, q0 = RN(x r) (within one ulp of x / d), and Markstein's correction
// step (P. Markstein, IBM J. Res. Develop. 34(1), 1990; Handbook of
// Floating-Point Arithmetic, theorem on division with a correctly rounded
// reciprocal) q = RN(q0 - RN(q0 d - x) r), the residual exact by FMA, is the
// correctly rounded quotient when nothing underflows (bf16 / fp16 values
// divided by an E4M3 scale stay far above the fp32 underflow threshold).  The
// residual is formed as q0 d + (-x) and subtracted, so a signed zero x gives
// q = x: -0.0 keeps its sign bit.  Both steps run on packed fp32 pairs
// (fma.rn.f32x2), and block maxima on packed bf16 / fp16 pairs.  The same
// step with the correctly rounded constant 1/6 gives amax / 6, and a table in
// shared memory holds d and 1/d for the 128 non-negative E4M3 codes.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ptx.cuh"

namespace nvfp4 {

namespace {

// Two E2M1 codes in one byte, `lo` in bits 0-3 (the even k), `hi` in bits 4-7:
// the hardware conversion rounds to nearest even and saturates at +-6.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// Two packed fp32 values in one 64-bit register, for the f32x2 instructions.
__device__ __forceinline__ uint64_t pack_f2(float lo, float hi) {
  return static_cast<uint64_t>(__float_as_uint(lo)) | (static_cast<uint64_t>(__float_as_uint(hi)) << 32);
}
__device__ __forceinline__ uint64_t mul_f2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fma_f2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// Eight 16-bit values (one uint4) -> four packed fp32 pairs, and the same
// pairs negated; plus the largest magnitude of the eight (exact).
template <bool kF16>
__device__ __forceinline__ float unpack8(const uint4 v, uint64_t* x2, uint64_t* nx2) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float amax = 0.0f;
  if constexpr (kF16) {
    __half2 m = __habs2(*reinterpret_cast<const __half2*>(&w[0]));
#pragma unroll
    for (int i = 1; i < 4; ++i) m = __hmax2(m, __habs2(*reinterpret_cast<const __half2*>(&w[i])));
    amax = fmaxf(__low2float(m), __high2float(m));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      x2[i] = pack_f2(t.x, t.y);
      nx2[i] = pack_f2(-t.x, -t.y);
    }
  } else {
    __nv_bfloat162 m = __habs2(*reinterpret_cast<const __nv_bfloat162*>(&w[0]));
#pragma unroll
    for (int i = 1; i < 4; ++i) m = __hmax2(m, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&w[i])));
    amax = fmaxf(__low2float(m), __high2float(m));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      // bf16 -> fp32 is the bit pattern shifted into the upper half
      const uint64_t lo = static_cast<uint64_t>(w[i] << 16), hi = static_cast<uint64_t>(w[i] & 0xFFFF0000u);
      x2[i] = lo | (hi << 32);
      nx2[i] = x2[i] ^ 0x8000000080000000ull;
    }
  }
  return amax;
}

// Groups of 4 rows loaded before any is processed: 128 bytes per lane in
// flight.  With 3 blocks per SM (registers capped at 80, a few bytes of
// spill) this beats 4 groups (GB300, 7168 x 16384 bf16: 63.9 vs 65.7 us);
// 16 groups at 2 or 3 blocks per SM are slower (72 / 80 us).
constexpr int kRowGroupsPerBatch = 8;
constexpr int kThreads = 256;

template <bool kF16>
__global__ void __launch_bounds__(kThreads, 3) quantize_kernel(const uint16_t* __restrict__ x,
                                                            uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                                                            int rows, int K, int L, int row_blocks,
                                                            int atoms_per_block) {
  __shared__ __align__(16) uint8_t atoms[kThreads / 32][512];  // one scale atom per warp
  __shared__ float2 scale_tab[128];                             // {d, 1/d} per E4M3 code 0..127
  for (int c = threadIdx.x; c < 128; c += blockDim.x) {
    const float dv = __half2float(__half(__nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(c), __NV_E4M3)));
    scale_tab[c] = make_float2(dv, c != 0 ? __frcp_rn(dv) : 0.0f);
  }
  // Programmatic dependent launch: the table above overlaps the previous
  // kernel on the stream; global memory waits for it (it may produce x or
  // still read the codes and scales about to be overwritten).
  ptx::griddep_launch_dependents();
  ptx::griddep_wait();
  __syncthreads();
  const int lane = threadIdx.x & 31;
  uint8_t* atom = atoms[threadIdx.x >> 5];
  const int sub = lane >> 3;  // row of a group of 4 rows
  const int j = lane & 7;     // 16-byte chunk (8 values) of the row's 64 values
  const int b = j >> 1;       // 16-value block of the chunk
  const long long tasks = static_cast<long long>(L) * row_blocks * atoms_per_block;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const int kblocks = K / 16;
  for (long long t = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; t < tasks;
       t += nwarps) {
    const int kc = static_cast<int>(t % atoms_per_block);  // 64-value chunk = scale atom
    const long long lrb = t / atoms_per_block;              // batch * row_blocks + row block
    const int rb = static_cast<int>(lrb % row_blocks);
    const int l = static_cast<int>(lrb / row_blocks);
    const bool kvalid = kc * 4 + b < kblocks;
#pragma unroll 1
    for (int g0 = 0; g0 < 32; g0 += kRowGroupsPerBatch) {
      uint4 v[kRowGroupsPerBatch];
#pragma unroll
      for (int u = 0; u < kRowGroupsPerBatch; ++u) {
        const int row = rb * 128 + (g0 + u) * 4 + sub;
        v[u] = make_uint4(0u, 0u, 0u, 0u);
        if (row < rows && kvalid)
          v[u] = __ldcs(reinterpret_cast<const uint4*>(x + (static_cast<long long>(l) * rows + row) * K +
                                                       kc * 64 + j * 8));
      }
#pragma unroll
      for (int u = 0; u < kRowGroupsPerBatch; ++u) {
        const int rin = (g0 + u) * 4 + sub;  // row inside the 128-row block
        const int row = rb * 128 + rin;
        uint64_t x2[4], nx2[4];
        float amax = unpack8<kF16>(v[u], x2, nx2);
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        constexpr float kSixth = 1.0f / 6.0f;  // correctly rounded reciprocal of 6
        const float a0 = __fmul_rn(amax, kSixth);
        const float a6 = __fmaf_rn(__fmaf_rn(-a0, 6.0f, amax), kSixth, a0);  // amax / 6, correctly rounded
        const __nv_fp8_storage_t sc = __nv_cvt_float_to_fp8(a6, __NV_SATFINITE, __NV_E4M3);
        const float2 dr = scale_tab[sc & 0x7F];
        const float d = dr.x;
        uint32_t word = 0;
        if (d != 0.0f) {
          const float r = dr.y;
          const uint64_t r2 = pack_f2(r, r), nr2 = pack_f2(-r, -r), d2 = pack_f2(d, d);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint64_t q0 = mul_f2(x2[i], r2);
            const uint64_t q = fma_f2(fma_f2(q0, d2, nx2[i]), nr2, q0);
            word |= e2m1x2(__uint_as_float(static_cast<uint32_t>(q)), __uint_as_float(static_cast<uint32_t>(q >> 32)))
                    << (8 * i);
          }
        }
        if (row < rows && kvalid)
          *reinterpret_cast<uint32_t*>(codes + (static_cast<long long>(l) * rows + row) * (K / 2) + kc * 32 + j * 4) =
              word;
        if ((j & 1) == 0) atom[(rin & 31) * 16 + (rin >> 5) * 4 + b] = static_cast<uint8_t>(sc);
      }
    }
    __syncwarp();
    *reinterpret_cast<uint4*>(sf + (lrb * atoms_per_block + kc) * 512 + lane * 16) =
        *reinterpret_cast<const uint4*>(atom + lane * 16);
    __syncwarp();
  }
}

}  // namespace

// Blocks of the quantize kernel resident per SM (0 on error).
int quantize_blocks_per_sm(int is_f16) {
  int n = 0;
  cudaError_t e = is_f16 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, quantize_kernel<true>, kThreads, 0)
                         : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, quantize_kernel<false>, kThreads, 0);
  return e == cudaSuccess ? n : 0;
}

// `max_blocks`: blocks resident at once on the device (one wave).
cudaError_t quantize_launch(const void* x, int is_f16, void* codes, void* sf, int rows, int K, int L,
                            int max_blocks, cudaStream_t stream) {
  const int row_blocks = (rows + 127) / 128;
  const int atoms_per_block = (K + 255) / 256 * 4;
  const long long tasks = static_cast<long long>(L) * row_blocks * atoms_per_block;
  long long blocks = (tasks + kThreads / 32 - 1) / (kThreads / 32);
  if (blocks > max_blocks) blocks = max_blocks;
  if (blocks < 1) blocks = 1;
  const uint16_t* xs = static_cast<const uint16_t*>(x);
  uint8_t* c = static_cast<uint8_t*>(codes);
  uint8_t* s = static_cast<uint8_t*>(sf);
  // a programmatic dependent of the previous kernel on the stream, like the GEMM
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (is_f16) return cudaLaunchKernelEx(&cfg, quantize_kernel<true>, xs, c, s, rows, K, L, row_blocks, atoms_per_block);
  return cudaLaunchKernelEx(&cfg, quantize_kernel<false>, xs, c, s, rows, K, L, row_blocks, atoms_per_block);
}

}  // namespace nvfp4
