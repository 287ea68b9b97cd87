// Group sums of the activations for the affine weight form w = scale * q + bias
// (the MLX affine 4-bit checkpoints of TensorFold PR #859):
//
//   y[m][n] = sum_g scale[n][g] * sum_{k in g} q[n][k] x[m][k] + sum_g bias[n][g] * X[m][g],
//   X[m][g] = sum_{k in g} x[m][k]
//
// X depends on x alone, so one table serves every weight that reads the same
// x with the same group size. Each X (a float32 sum) is stored as three bf16
// parts hi + mid + lo that add up to it exactly (hi = bf16(X), mid =
// bf16(X - hi), lo = X - hi - mid; every residual is exact in float32 and the
// last fits in bf16), so that the tcgen05 GEMM forms sum_g bias * X[m][g] with
// exact bf16 products against the bias operand of the packed weight.
// Layout: bf16 [M][kb3], kb3 = 3 * K/G rounded up to 64, X[m][g]'s parts at
// columns 3g, 3g+1, 3g+2, zeros beyond 3 * K/G.
#include "w4a16_internal.h"

namespace w4a16 {
namespace {

constexpr int kXsThreads = 256;

__device__ __forceinline__ uint16_t bf16_rn(float v) {
  __nv_bfloat16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<uint16_t *>(&b);
}

// One warp per x row: each lane sums 8 consecutive k of a 256-wide slab, then
// the G/8 lanes of a group meet by shuffles and one of them writes the parts.
__global__ void __launch_bounds__(kXsThreads) xsum_kernel(const uint16_t *x, int M, int K, int group, int kb3,
                                                          uint16_t *xs) {
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (kXsThreads / 32);
  const int lpg = group / 8;  // lanes per group: 8 or 16
  const int groups = K / group;
  for (int m = blockIdx.x * (kXsThreads / 32) + (threadIdx.x >> 5); m < M; m += warps) {
    const uint16_t *row = x + (size_t)m * K;
    uint16_t *out = xs + (size_t)m * kb3;
    for (int j = 3 * groups + lane; j < kb3; j += 32) out[j] = 0;
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
      if (k < K && (lane & (lpg - 1)) == 0) {
        const int gi = k / group;
        const uint16_t hi = bf16_rn(v);
        const float r1 = v - __uint_as_float((uint32_t)hi << 16);
        const uint16_t mid = bf16_rn(r1);
        const float r2 = r1 - __uint_as_float((uint32_t)mid << 16);
        out[3 * gi] = hi;
        out[3 * gi + 1] = mid;
        out[3 * gi + 2] = bf16_rn(r2);
      }
    }
  }
}

// x [M][K] -> xw [M][2K]: group g of row m written at columns 2gG .. 2gG+G-1
// and again at 2gG+G .. 2gG+2G-1, 16 bytes per thread and step.
__global__ void widen_groups_kernel(const uint4 *x, int M, int K, int group, uint4 *xw) {
  const size_t kv = K / 8, total = (size_t)M * kv;
  const int gv = group / 8;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const size_t m = i / kv;
    const int v = (int)(i % kv), g = v / gv, j = v % gv;
    const uint4 val = x[i];
    uint4 *out = xw + m * 2 * kv + (size_t)2 * g * gv + j;
    out[0] = val;
    out[gv] = val;
  }
}

}  // namespace

cudaError_t launch_widen_groups(const uint16_t *x, int M, int K, int group, uint16_t *xw, cudaStream_t stream) {
  const size_t work = (size_t)M * (K / 8);
  size_t blocks = (work + kXsThreads - 1) / kXsThreads;
  if (blocks > 65535u * 8u) blocks = 65535u * 8u;
  widen_groups_kernel<<<(unsigned)(blocks < 1 ? 1 : blocks), kXsThreads, 0, stream>>>(
      reinterpret_cast<const uint4 *>(x), M, K, group, reinterpret_cast<uint4 *>(xw));
  return cudaGetLastError();
}

cudaError_t launch_xsum(const uint16_t *x, int M, int K, int group, uint16_t *xs, cudaStream_t stream) {
  int blocks = (M + kXsThreads / 32 - 1) / (kXsThreads / 32);
  if (blocks > 4096) blocks = 4096;
  xsum_kernel<<<blocks, kXsThreads, 0, stream>>>(x, M, K, group, affine_kb3(K / group), xs);
  return cudaGetLastError();
}

}  // namespace w4a16
