// Group sums of the activations for the affine weight form w = scale * q + bias
// (the MLX affine 4-bit checkpoints of TensorFold PR #859):
//
//   y[m][n] = sum_g scale[n][g] * sum_{k in g} q[n][k] x[m][k] + sum_g bias[n][g] * X[g][m],
//   X[g][m] = sum_{k in g} x[m][k]
//
// X depends on x alone, so one table serves every weight that reads the same
// x with the same group size. Layout: float32 [K/G][ld], ld = M rounded up to a
// multiple of 256 (the tcgen05 GEMM loads boxes of up to 256 x rows by four
// groups); entries m >= M are zero.
#include "w4a16_internal.h"

namespace w4a16 {
namespace {

constexpr int kXsThreads = 256;

// One warp per x row: each lane sums 8 consecutive k of a 256-wide slab, then
// the G/8 lanes of a group meet by shuffles and one of them writes X[g][m].
__global__ void __launch_bounds__(kXsThreads) xsum_kernel(const uint16_t *x, int M, int K, int group, int ld,
                                                          float *xs) {
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (kXsThreads / 32);
  const int lpg = group / 8;  // lanes per group: 8 or 16
  for (int m = blockIdx.x * (kXsThreads / 32) + (threadIdx.x >> 5); m < ld; m += warps) {
    if (m >= M) {  // padding columns: zero (warp-uniform branch)
      for (int g = lane; g < K / group; g += 32) xs[(size_t)g * ld + m] = 0.f;
      continue;
    }
    const uint16_t *row = x + (size_t)m * K;
    for (int k0 = 0; k0 < K; k0 += 256) {
      const int k = k0 + 8 * lane;
      float v = 0.f;
      if (k < K) {
        const uint4 w = *reinterpret_cast<const uint4 *>(row + k);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) v += bf16lo_to_f32(ws[i]) + bf16hi_to_f32(ws[i]);
      }
      for (int o = 1; o < lpg; o <<= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
      if (k < K && (lane & (lpg - 1)) == 0) xs[(size_t)(k / group) * ld + m] = v;
    }
  }
}

}  // namespace

int xsum_ld(int M) { return (M + 255) / 256 * 256; }

cudaError_t launch_xsum(const uint16_t *x, int M, int K, int group, float *xs, cudaStream_t stream) {
  const int ld = xsum_ld(M);
  int blocks = (ld + kXsThreads / 32 - 1) / (kXsThreads / 32);
  if (blocks > 4096) blocks = 4096;
  xsum_kernel<<<blocks, kXsThreads, 0, stream>>>(x, M, K, group, ld, xs);
  return cudaGetLastError();
}

}  // namespace w4a16
