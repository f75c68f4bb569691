// Scale-factor repack: row-major E4M3 scales [L][rows][K/16] -> the 512-byte
// atom layout the tensor cores read.
//
// out[l][rm][ck][r0][r1][c0] = sf[l][128*rm + 32*r1 + r0][4*ck + c0]
// ("nvfp4 gemm, submission 125598", custom_kernel docstring: permuted scales
// of logical shape [32, 4, rest_m, 4, rest_k, l]; the atom order and the
// 2048-byte k-tile slabs follow "nvfp4 group gemm, submission 407526",
// grouped_kernel TMA producer).  rest_k is padded to whole 256-wide k-tiles;
// padding is zero.
//
// One CTA transposes a 128-row x 128-column tile of scales (the 32 atoms of
// one 128-row block and eight k-tiles) through shared memory: it reads the
// tile row by row (each warp four 128-byte row segments per instruction) and
// writes the 32 atoms as 16 KB of contiguous output (each warp one 512-byte
// atom per instruction).  The shared tile has a 33-word row pitch, so both
// the row-wise stores and the atom-wise reads hit 32 different banks.
#include <cuda_runtime.h>
#include <stdint.h>

#include "ptx.cuh"

namespace nvfp4 {

constexpr int kTileRows = 128;   // one 128-row scale block
constexpr int kTileCols = 128;   // scale bytes per row: 32 atoms, eight 256-wide k-tiles
constexpr int kPitchWords = kTileCols / 4 + 1;
constexpr int kRepackThreads = 256;

__global__ void __launch_bounds__(kRepackThreads) repack_scales_kernel(const uint8_t* __restrict__ sf,
                                                                       uint8_t* __restrict__ out, int rows,
                                                                       int cols, int rest_m, int rest_k,
                                                                       int ctiles) {
  __shared__ uint32_t tile[kTileRows * kPitchWords];
  // Programmatic dependent launch: the next kernel on the stream may be
  // scheduled now, and this grid may have started before the previous kernel
  // finished, so it waits for it before touching global memory (the previous
  // kernel may produce `sf` or still read `out`).
  ptx::griddep_launch_dependents();
  ptx::griddep_wait();
  // block = (l * rest_m + rm) * ctiles + ct
  const int ct = static_cast<int>(blockIdx.x % static_cast<unsigned>(ctiles));  // atoms 32*ct .. 32*ct+31
  const long long lm = blockIdx.x / static_cast<unsigned>(ctiles);
  const int rm = static_cast<int>(lm % rest_m);                                  // 128-row block
  const long long l = lm / rest_m;
  const int t = threadIdx.x;
  const int c_base = ct * kTileCols;
  const bool vec = (cols & 15) == 0;         // every row starts 16-byte aligned
  const bool words = (cols & 3) == 0;        // every row starts 4-byte aligned
  // load: element i of the 128 x 8 grid of 16-byte chunks, zero past the edges
#pragma unroll
  for (int i = 0; i < kTileRows * kTileCols / 16 / kRepackThreads; ++i) {
    const int idx = t + i * kRepackThreads;
    const int row = idx >> 3, chunk = idx & 7;
    const int r = rm * kTileRows + row;
    const int c = c_base + chunk * 16;
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    if (r < rows && c < cols) {
      const uint8_t* src = sf + (l * rows + r) * static_cast<long long>(cols) + c;
      if (vec) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(src));
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
      } else if (words) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (c + 4 * e < cols) w[e] = __ldg(reinterpret_cast<const uint32_t*>(src) + e);
      } else {
        for (int b = 0; b < 16 && c + b < cols; ++b) w[b >> 2] |= static_cast<uint32_t>(src[b]) << (8 * (b & 3));
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) tile[row * kPitchWords + chunk * 4 + e] = w[e];
  }
  __syncthreads();
  // store: warp w writes atoms w, w + 8, w + 16, w + 24 of the tile; lane r0
  // writes the atom's row r0 = the four scales of rows r0, r0+32, r0+64, r0+96
  const int warp = t >> 5, r0 = t & 31;
  uint4* dst = reinterpret_cast<uint4*>(out) + ((l * rest_m + rm) * rest_k) * 32 + r0;
#pragma unroll
  for (int i = 0; i < kTileCols / 4 / (kRepackThreads / 32); ++i) {
    const int a = warp + i * (kRepackThreads / 32);
    const int ck = ct * (kTileCols / 4) + a;
    if (ck >= rest_k) break;
    const uint4 v = make_uint4(tile[r0 * kPitchWords + a], tile[(r0 + 32) * kPitchWords + a],
                               tile[(r0 + 64) * kPitchWords + a], tile[(r0 + 96) * kPitchWords + a]);
    dst[static_cast<long long>(ck) * 32] = v;
  }
}

cudaError_t repack_launch(const void* sf, void* out, int rows, int K, int L, cudaStream_t stream) {
  const int cols = K / 16;
  const int rest_m = (rows + 127) / 128;
  const int rest_k = ((K + 255) / 256) * 4;
  const int ctiles = (rest_k + kTileCols / 4 - 1) / (kTileCols / 4);
  const long long blocks = static_cast<long long>(L) * rest_m * ctiles;
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  // launched like the GEMM, as a programmatic dependent of the previous kernel
  // on the stream: back-to-back launches overlap one's start with the other's end
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(kRepackThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, repack_scales_kernel, static_cast<const uint8_t*>(sf), static_cast<uint8_t*>(out),
                            rows, cols, rest_m, rest_k, ctiles);
}

}  // namespace nvfp4
