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
// codes take the step negated, so that x itself is the FMA's addend and no
// negated copy of the inputs is needed: nq0 = RN(x (-r)) = -q0,
// t = RN(nq0 d + x) = x - q0 d (exact), nq = RN(nq0 + t (-r)) = -q, round to
// nearest being symmetric; E2M1 is sign-magnitude, so one xor of the packed
// codes (every nibble's bit 3) turns the codes of nq into those of q, and a
// signed zero x gives the code of x: +0 -> 0x0, -0 -> 0x8 (GB300, 7168 x
// 16384 bf16: 58.7 -> 56.3 us).  Both steps run on packed fp32 pairs
// (fma.rn.f32x2), and block maxima on packed bf16 / fp16 pairs.  The same
// step, unnegated, with the correctly rounded constant 1/6 gives amax / 6, and
// a table in shared memory holds d and 1/d for the 128 non-negative E4M3
// codes.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ptx.cuh"

namespace nvfp4 {

namespace {

// Eight E2M1 codes from four packed fp32 pairs: byte i holds pair i, its low
// half (the even k) in bits 0-3 and its high half in bits 4-7.  The hardware
// conversion rounds to nearest even and saturates at +-6; the four bytes are
// packed by one vector move instead of widening, shifting and or-ing each.
// (GB300, 7168 x 16384 bf16: 61.6 -> 60.0 us.)
__device__ __forceinline__ uint32_t e2m1x8(const uint64_t* q) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(__uint_as_float(static_cast<uint32_t>(q[0]))), "f"(__uint_as_float(static_cast<uint32_t>(q[0] >> 32))),
        "f"(__uint_as_float(static_cast<uint32_t>(q[1]))), "f"(__uint_as_float(static_cast<uint32_t>(q[1] >> 32))),
        "f"(__uint_as_float(static_cast<uint32_t>(q[2]))), "f"(__uint_as_float(static_cast<uint32_t>(q[2] >> 32))),
        "f"(__uint_as_float(static_cast<uint32_t>(q[3]))), "f"(__uint_as_float(static_cast<uint32_t>(q[3] >> 32))));
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

// Eight 16-bit values (one uint4) -> four packed fp32 pairs, plus the
// largest magnitude of the eight (exact).  The maximum runs on packed pairs
// with max.xorsign.abs (max(|a|, |b|), the sign bit the xor of the two: only
// the magnitude is used), three instructions for the eight values (GB300,
// 7168 x 16384 bf16: 61.6 -> 60.2 us).
template <bool kF16>
__device__ __forceinline__ float unpack8(const uint4 v, uint64_t* x2) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float amax = 0.0f;
  if constexpr (kF16) {
    uint32_t m;
    asm("max.xorsign.abs.f16x2 %0, %1, %2;" : "=r"(m) : "r"(w[0]), "r"(w[1]));
    asm("max.xorsign.abs.f16x2 %0, %1, %2;" : "=r"(m) : "r"(m), "r"(w[2]));
    asm("max.xorsign.abs.f16x2 %0, %1, %2;" : "=r"(m) : "r"(m), "r"(w[3]));
    const __half2 mh = *reinterpret_cast<const __half2*>(&m);
    amax = fmaxf(fabsf(__low2float(mh)), fabsf(__high2float(mh)));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      x2[i] = pack_f2(t.x, t.y);
    }
  } else {
    uint32_t m;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(w[0]), "r"(w[1]));
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(m), "r"(w[2]));
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(m), "r"(w[3]));
    // bf16 -> fp32 is the bit pattern in the upper half
    amax = fmaxf(fabsf(__uint_as_float(m << 16)), fabsf(__uint_as_float(m & 0xFFFF0000u)));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      // bf16 -> fp32 is the bit pattern shifted into the upper half
      const uint64_t lo = static_cast<uint64_t>(w[i] << 16), hi = static_cast<uint64_t>(w[i] & 0xFFFF0000u);
      x2[i] = lo | (hi << 32);
    }
  }
  return amax;
}

// Groups of 4 rows loaded before any is processed: 128 bytes per lane in
// flight, at 3 blocks per SM (74 registers, no spills).  GB300, 7168 x 16384
// bf16: 51.6 us; 4 groups at 4 blocks per SM 51.9, 8 at 4 blocks 51.2 (a few
// bytes of spill), 16 at 3 blocks 62.0.
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
  const bool small_tasks = tasks <= 0xFFFFFFFFll;
  for (long long t = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; t < tasks;
       t += nwarps) {
    int kc, rb, l;  // 64-value chunk (= scale atom), 128-row block, batch
    long long lrb;  // batch * row_blocks + row block
    if (small_tasks) {  // 32-bit divisions, same quotients (GB300, 7168 x 16384 bf16: 51.6 -> 51.2 us)
      const uint32_t tt = static_cast<uint32_t>(t);
      const uint32_t q = tt / static_cast<uint32_t>(atoms_per_block);
      kc = static_cast<int>(tt - q * static_cast<uint32_t>(atoms_per_block));
      const uint32_t q2 = q / static_cast<uint32_t>(row_blocks);
      rb = static_cast<int>(q - q2 * static_cast<uint32_t>(row_blocks));
      l = static_cast<int>(q2);
      lrb = q;
    } else {
      kc = static_cast<int>(t % atoms_per_block);
      lrb = t / atoms_per_block;
      rb = static_cast<int>(lrb % row_blocks);
      l = static_cast<int>(lrb / row_blocks);
    }
    const bool kvalid = kc * 4 + b < kblocks;
    // this lane's first row of the block and the 4-row stride, computed once
    // per task instead of a 64-bit row offset per load and store (GB300,
    // 7168 x 16384 bf16: 56.4 -> 51.6 us, and no register spills)
    const long long row0 = static_cast<long long>(l) * rows + rb * 128 + sub;
    const uint16_t* xp = x + row0 * K + kc * 64 + j * 8;
    uint8_t* cp = codes + row0 * (K / 2) + kc * 32 + j * 4;
    const long long xstep = 4LL * K, cstep = 2LL * K;
    const int lim = kvalid ? rows - (rb * 128 + sub) : 0;  // row groups g with 4 g < lim are in range
#pragma unroll 1
    for (int g0 = 0; g0 < 32; g0 += kRowGroupsPerBatch, xp += kRowGroupsPerBatch * xstep,
             cp += kRowGroupsPerBatch * cstep) {
      uint4 v[kRowGroupsPerBatch];
#pragma unroll
      for (int u = 0; u < kRowGroupsPerBatch; ++u) {
        v[u] = make_uint4(0u, 0u, 0u, 0u);
        if ((g0 + u) * 4 < lim) v[u] = __ldcs(reinterpret_cast<const uint4*>(xp + u * xstep));
      }
#pragma unroll
      for (int u = 0; u < kRowGroupsPerBatch; ++u) {
        const int rin = (g0 + u) * 4 + sub;  // row inside the 128-row block
        uint64_t x2[4];
        float amax = unpack8<kF16>(v[u], x2);
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
          const uint64_t nr2 = pack_f2(-r, -r), d2 = pack_f2(d, d);
          uint64_t nq[4];  // -(x / d), correctly rounded (see the top of the file)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint64_t nq0 = mul_f2(x2[i], nr2);
            nq[i] = fma_f2(fma_f2(nq0, d2, x2[i]), nr2, nq0);
          }
          word = e2m1x8(nq) ^ 0x88888888u;  // the codes of -nq: every sign bit flipped
        }
        if ((g0 + u) * 4 < lim) *reinterpret_cast<uint32_t*>(cp + u * cstep) = word;
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
