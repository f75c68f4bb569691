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
// One thread writes one 16-byte atom row (r0): the four 4-byte groups of rows
// r0, r0+32, r0+64, r0+96.  Consecutive threads write consecutive 16-byte
// chunks, so the stores are fully coalesced; the loads are 4-byte gathers.
#include <cuda_runtime.h>
#include <stdint.h>

namespace nvfp4 {

__global__ void __launch_bounds__(256) repack_scales_kernel(const uint8_t* __restrict__ sf,
                                                            uint8_t* __restrict__ out, int rows,
                                                            int cols, int rest_m, int rest_k,
                                                            long long chunks) {
  const long long q = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (q >= chunks) return;
  // q = (((l * rest_m + rm) * rest_k + ck) * 32 + r0)
  const int r0 = static_cast<int>(q & 31);
  long long t = q >> 5;
  const int ck = static_cast<int>(t % rest_k);
  t /= rest_k;
  const int rm = static_cast<int>(t % rest_m);
  const long long l = t / rest_m;
  const int c = ck * 4;
  uint32_t w[4];
  const bool aligned_cols = (cols & 3) == 0;
#pragma unroll
  for (int r1 = 0; r1 < 4; ++r1) {
    const int r = rm * 128 + r1 * 32 + r0;
    uint32_t v = 0;
    if (r < rows && c < cols) {
      const uint8_t* src = sf + (l * rows + r) * static_cast<long long>(cols) + c;
      if (aligned_cols && c + 4 <= cols) {
        v = __ldg(reinterpret_cast<const uint32_t*>(src));
      } else {
        for (int c0 = 0; c0 < 4 && c + c0 < cols; ++c0) v |= static_cast<uint32_t>(src[c0]) << (8 * c0);
      }
    }
    w[r1] = v;
  }
  reinterpret_cast<uint4*>(out)[q] = make_uint4(w[0], w[1], w[2], w[3]);
}

cudaError_t repack_launch(const void* sf, void* out, int rows, int K, int L, cudaStream_t stream) {
  const int cols = K / 16;
  const int rest_m = (rows + 127) / 128;
  const int rest_k = ((K + 255) / 256) * 4;
  const long long chunks = static_cast<long long>(L) * rest_m * rest_k * 32;
  if (chunks == 0) return cudaSuccess;
  const int threads = 256;
  const long long blocks = (chunks + threads - 1) / threads;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  repack_scales_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      static_cast<const uint8_t*>(sf), static_cast<uint8_t*>(out), rows, cols, rest_m, rest_k,
      chunks);
  return cudaGetLastError();
}

}  // namespace nvfp4
