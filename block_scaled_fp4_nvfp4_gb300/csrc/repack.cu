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
// One thread writes eight 16-byte atom rows: row r0 of the eight consecutive
// atoms ck = 8*j8 .. 8*j8+7 of one 128-row block.  It reads 32 contiguous
// bytes (eight groups of four scales) from each of rows r0, r0+32, r0+64 and
// r0+96 -- whole 32-byte sectors when the row pitch K/16 is a multiple of 16
// -- and for each atom the 32 threads of a warp store 512 contiguous bytes.
#include <cuda_runtime.h>
#include <stdint.h>

namespace nvfp4 {

constexpr int kAtomsPerThread = 8;

__global__ void __launch_bounds__(256) repack_scales_kernel(const uint8_t* __restrict__ sf,
                                                            uint8_t* __restrict__ out, int rows,
                                                            int cols, int rest_m, int rest_k,
                                                            long long work) {
  const long long q = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (q >= work) return;
  // q = (((l * rest_m + rm) * groups + j8) * 32 + r0), groups = ceil(rest_k / 8)
  const int groups = (rest_k + kAtomsPerThread - 1) / kAtomsPerThread;
  const int r0 = static_cast<int>(q & 31);
  long long t = q >> 5;
  const int j8 = static_cast<int>(t % groups);
  t /= groups;
  const int rm = static_cast<int>(t % rest_m);
  const long long l = t / rest_m;
  const int c0 = j8 * kAtomsPerThread * 4;  // first scale column of atom 8*j8
  uint32_t w[4][kAtomsPerThread];
  const bool wide = (cols & 15) == 0 && c0 + kAtomsPerThread * 4 <= cols;
  const bool aligned_cols = (cols & 3) == 0;
#pragma unroll
  for (int r1 = 0; r1 < 4; ++r1) {
    const int r = rm * 128 + r1 * 32 + r0;
#pragma unroll
    for (int j = 0; j < kAtomsPerThread; ++j) w[r1][j] = 0u;
    if (r >= rows) continue;
    const uint8_t* src = sf + (l * rows + r) * static_cast<long long>(cols) + c0;
    if (wide) {
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(src));
      const uint4 b = __ldg(reinterpret_cast<const uint4*>(src) + 1);
      w[r1][0] = a.x; w[r1][1] = a.y; w[r1][2] = a.z; w[r1][3] = a.w;
      w[r1][4] = b.x; w[r1][5] = b.y; w[r1][6] = b.z; w[r1][7] = b.w;
    } else {
#pragma unroll
      for (int j = 0; j < kAtomsPerThread; ++j) {
        const int c = c0 + 4 * j;
        if (c >= cols) break;
        if (aligned_cols) {
          w[r1][j] = __ldg(reinterpret_cast<const uint32_t*>(src + 4 * j));
        } else {
          uint32_t v = 0;
          for (int cc = 0; cc < 4 && c + cc < cols; ++cc) v |= static_cast<uint32_t>(src[4 * j + cc]) << (8 * cc);
          w[r1][j] = v;
        }
      }
    }
  }
  uint4* dst = reinterpret_cast<uint4*>(out) + ((l * rest_m + rm) * rest_k) * 32 + r0;
#pragma unroll
  for (int j = 0; j < kAtomsPerThread; ++j) {
    const int ck = j8 * kAtomsPerThread + j;
    if (ck < rest_k) dst[static_cast<long long>(ck) * 32] = make_uint4(w[0][j], w[1][j], w[2][j], w[3][j]);
  }
}

cudaError_t repack_launch(const void* sf, void* out, int rows, int K, int L, cudaStream_t stream) {
  const int cols = K / 16;
  const int rest_m = (rows + 127) / 128;
  const int rest_k = ((K + 255) / 256) * 4;
  const int groups = (rest_k + kAtomsPerThread - 1) / kAtomsPerThread;
  const long long work = static_cast<long long>(L) * rest_m * groups * 32;
  if (work == 0) return cudaSuccess;
  const int threads = 256;
  const long long blocks = (work + threads - 1) / threads;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  repack_scales_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      static_cast<const uint8_t*>(sf), static_cast<uint8_t*>(out), rows, cols, rest_m, rest_k,
      work);
  return cudaGetLastError();
}

}  // namespace nvfp4
