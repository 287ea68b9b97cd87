// Internal launcher interface between the C-ABI layer and the kernels.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "w4a16_common.cuh"

namespace w4a16 {

constexpr int kMaxDevices = 64;

// A per-device fact about one kernel that is found once and then reused on
// every call (the dynamic shared-memory opt-in is a per-device function
// attribute; the occupancy query is slow next to a decode launch). 0 = not
// found yet on that device; racing first calls store the same value.
struct PerDevice {
  std::atomic<int> v[kMaxDevices];
};

// One matmul call as the kernels see it. For the fused gate/up form,
// N is the rows of ONE of the two weights (N_each), `packed` the interleaved
// buffer, and the output has N columns.
struct GemmCall {
  const uint16_t *x;
  const uint8_t *packed;
  uint16_t *y;
  int M, N, K, group, sym;  // sym: the form (kFormZero, kFormSym, kFormAffine)
  bool gateup;
  cudaStream_t stream;
  int *err;    // device error word (bounded waits that gave up)
  int device;  // current device ordinal, < kMaxDevices
  bool overlap;  // programmatic overlap with the previous kernel (M <= 32 kernels)
  int64_t *amax = nullptr;  // argmax keys per x row (M <= 32 plain GEMM), or null
  const uint16_t *xsum = nullptr;  // affine form, tcgen05 GEMM: x group sums, bf16 parts [M][kb3]
  int xs_mode = 1;  // M <= 16, the kernel that stages x once per CTA: 0 never, 1 where measured faster, 2 always
};

// Rows covered by the packed buffer of a call (padded; interleaved for gate/up).
inline int packed_rows(const GemmCall &c) {
  return c.gateup ? 2 * ((c.N + 127) / 128 * 128) : c.N;
}

// canonical weight(s) -> tiled layout; z* for the zero-point form, b* (biases)
// for the affine form, each null otherwise; the second set for gate/up only
cudaError_t launch_repack(const int32_t *qw0, const uint16_t *sc0, const int32_t *z0, const uint16_t *b0,
                          const int32_t *qw1, const uint16_t *sc1, const int32_t *z1, const uint16_t *b1,
                          int n_src, bool gateup, const Layout &L, uint8_t *packed,
                          cudaStream_t stream);
cudaError_t launch_dequantize(const uint8_t *packed, const Layout &L, int N, float *w,
                              cudaStream_t stream);
// b-bit affine codes (canonical: one little-endian bit stream per row of K
// codes) -> the affine tiled layout L, widened to nibbles (bits <= 4, L.K = K)
// or split into two nibble planes (bits 5-8, L.K = 2K); and the read-back
cudaError_t launch_repack_affine_bits(const uint32_t *qw, const uint16_t *sc, const uint16_t *b, int N, int K,
                                      int bits, const Layout &L, uint8_t *packed, cudaStream_t stream);
cudaError_t launch_dequantize_affine_bits(const uint8_t *packed, const Layout &L, int N, int K, int bits, float *w,
                                          cudaStream_t stream);
// x [M][K] -> xw [M][2K] with each group of x written twice in a row (the
// x of the two nibble planes of a 5-8-bit affine weight)
cudaError_t launch_widen_groups(const uint16_t *x, int M, int K, int group, uint16_t *xw, cudaStream_t stream);

cudaError_t launch_smallm_mma(const GemmCall &c, int sm_count);  // 1 <= M <= 32
cudaError_t launch_gemv_m1(const GemmCall &c, int sm_count);     // M == 1, not gate/up
cudaError_t launch_prompt_tc(const GemmCall &c, int sm_count);   // any M
// 2-D tiled tensor map (driver entry point found once); false if unavailable
// or rejected
bool encode_2d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw);
// tcgen05 decode kernel: 1 <= M <= 32, plain zero-point or symmetric GEMM
bool smallm_tc_supports(const GemmCall &c);
cudaError_t launch_smallm_tc(const GemmCall &c, int sm_count);
// argmax of bf16 y rows: keys (zeroed before) -> indices in place; and, for
// y already written, the keys of every row
cudaError_t launch_argmax_init(int64_t *amax, int M, bool overlap, cudaStream_t stream);
cudaError_t launch_argmax_finalize(int64_t *amax, int M, bool overlap, cudaStream_t stream);
// affine form: X[m][g] = sum of x[m][k] over group g, as three bf16 parts per
// group, bf16 [M][affine_kb3(K / group)]
cudaError_t launch_xsum(const uint16_t *x, int M, int K, int group, uint16_t *xs, cudaStream_t stream);
cudaError_t launch_row_argmax(const uint16_t *y, int M, int N, int64_t *amax, cudaStream_t stream);
// the k largest entries of every bf16 row of y [M][N], largest first
constexpr int kTopkMaxK = 1024;
cudaError_t launch_topk(const uint16_t *y, int M, int N, int k, int64_t *idx, uint16_t *vals, bool overlap,
                        int device, cudaStream_t stream);

}  // namespace w4a16
