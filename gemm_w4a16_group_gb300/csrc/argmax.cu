// Argmax over the bf16 outputs of the output-vocabulary head, on the device,
// so that greedy decoding reads back one index per row instead of the logits
// (the GPU argmax that lucebox PR #823 runs after its tall head).
//
// Keys (w4a16_common.cuh, argmax_key) order the bf16 values and break ties
// toward the lower index; every producer folds its keys into keys[m] with
// 64-bit atomicMax on a buffer zeroed before, and the finalize step rewrites
// each key as its index in place. The M <= 32 decode kernels produce keys in
// its epilogue (fused); for y already in memory, row_argmax_kernel does.
#include "w4a16_internal.h"

namespace w4a16 {
namespace {

constexpr int kRowThreads = 256;
constexpr int kRowChunk = 8192;  // columns per CTA

// keys[m] := 0, below every key. A kernel rather than a memset so that a chain
// of calls stays a chain of kernels with programmatic overlap: the GEMM that
// follows may start streaming its weights while this runs.
__global__ void argmax_init_kernel(int64_t *amax, int M) {
  grid_launch_dependents();
  grid_dependency_wait();  // the buffer may still be read by the kernel before
  for (int m = blockIdx.x * blockDim.x + threadIdx.x; m < M; m += gridDim.x * blockDim.x) amax[m] = 0;
}

// keys[m] := the index it encodes (first maximum of row m)
__global__ void argmax_finalize_kernel(int64_t *amax, int M) {
  grid_launch_dependents();
  grid_dependency_wait();  // the keys are complete once the producing kernel has finished
  for (int m = blockIdx.x * blockDim.x + threadIdx.x; m < M; m += gridDim.x * blockDim.x) {
    const unsigned long long key = static_cast<unsigned long long>(amax[m]);
    amax[m] = (int64_t)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
  }
}

// keys of y[m][n0 .. n0 + kRowChunk) for row m = blockIdx.y
__global__ void __launch_bounds__(kRowThreads) row_argmax_kernel(const uint16_t *y, int N, int64_t *amax) {
  __shared__ unsigned long long best;
  if (threadIdx.x == 0) best = 0;
  __syncthreads();
  const int m = blockIdx.y;
  const int n0 = blockIdx.x * kRowChunk, n1 = min(n0 + kRowChunk, N);
  const uint16_t *row = y + (size_t)m * N;
  unsigned long long k = 0;
  for (int n = n0 + threadIdx.x; n < n1; n += kRowThreads) {
    const unsigned long long c = argmax_key(row[n], n);
    k = c > k ? c : k;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long c = __shfl_xor_sync(0xFFFFFFFFu, k, o);
    k = c > k ? c : k;
  }
  if ((threadIdx.x & 31) == 0) atomicMax(&best, k);
  __syncthreads();
  if (threadIdx.x == 0 && best != 0) atomicMax(reinterpret_cast<unsigned long long *>(amax + m), best);
}

}  // namespace

namespace {
template <typename... Args>
cudaError_t launch_small(void (*kern)(Args...), int M, bool overlap, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((M + 255) / 256 < 1024 ? (M + 255) / 256 : 1024, 1, 1);
  lc.blockDim = dim3(256, 1, 1);
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = overlap ? 1 : 0;
  return cudaLaunchKernelEx(&lc, kern, args...);
}
}  // namespace

cudaError_t launch_argmax_init(int64_t *amax, int M, bool overlap, cudaStream_t stream) {
  return launch_small(argmax_init_kernel, M, overlap, stream, amax, M);
}

cudaError_t launch_argmax_finalize(int64_t *amax, int M, bool overlap, cudaStream_t stream) {
  return launch_small(argmax_finalize_kernel, M, overlap, stream, amax, M);
}

cudaError_t launch_row_argmax(const uint16_t *y, int M, int N, int64_t *amax, cudaStream_t stream) {
  for (int m0 = 0; m0 < M; m0 += 65535) {  // grid y limit
    const dim3 grid((N + kRowChunk - 1) / kRowChunk, min(M - m0, 65535), 1);
    row_argmax_kernel<<<grid, kRowThreads, 0, stream>>>(y + (size_t)m0 * N, N, amax + m0);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace w4a16
