// Offline repack (canonical -> tiled layout) and the dequantisation read-back
// used by the tests.
//
// The canonical packing (nibble j of word c holds k = 8c + j) and the exact
// w = (q - z) * scale follow the INT4 kernels of the GRIMOIRE v1.7 release
// notes ("What changed"); the affine form w = scale * q + bias is that of the
// MLX affine 4-bit checkpoints in TensorFold PR #859 ("What this changes":
// every code keeps its value, scale and bias). The tiled order is this
// library's own, described in w4a16_common.cuh.
#include "w4a16_internal.h"

namespace w4a16 {
namespace {

struct RepackSrc {
  const uint32_t *qw[2];
  const uint16_t *sc[2];
  const uint32_t *z[2];
  const uint16_t *b[2];  // biases (affine form)
  int n_src;     // rows of each source weight
  int gateup;    // 0: one weight, tile T = rows 16T..; 1: tiles alternate gate, up
  // b-bit affine codes (bits != 0): qw is one little-endian bit stream per
  // row of k_src codes; bits <= 4 are widened into the nibbles (layout K =
  // k_src), bits 5-8 are split into two 4-bit planes (below; layout K =
  // 2 k_src)
  int bits;
  int k_src;
};

// Two planes of a b-bit code q = 16 qh + ql (bits 5-8): packed group 2g holds
// qh with scale 16 s and the bias, packed group 2g + 1 holds ql with scale s
// and bias 0, both against the same x values (the x of group g, repeated).
// 16 s is exact in bf16 (scales below 2^123 do not overflow).
__device__ __forceinline__ bool two_planes(const RepackSrc &s) { return s.bits > 4; }

// code k of a row of the b-bit stream
__device__ __forceinline__ uint32_t stream_code(const uint32_t *row_words, int words, int bits, int k) {
  const long long bit = (long long)k * bits;
  const int w = (int)(bit >> 5);
  uint64_t v = row_words[w];
  if (w + 1 < words) v |= (uint64_t)row_words[w + 1] << 32;
  return (uint32_t)((v >> (bit & 31)) & ((1u << bits) - 1u));
}

// the 4-bit code at packed column k of a source row (b-bit forms)
__device__ __forceinline__ uint32_t bits_code(const RepackSrc &s, int which, int row, int k, int group) {
  const int words = (int)(((long long)s.k_src * s.bits + 31) / 32);
  const uint32_t *rw = s.qw[which] + (size_t)row * words;
  if (!two_planes(s)) return stream_code(rw, words, s.bits, k);
  const int gp = k / group, g = gp >> 1;
  const uint32_t q = stream_code(rw, words, s.bits, g * group + k % group);
  return (gp & 1) ? (q & 0xFu) : (q >> 4);
}

// scale (or bias) of packed group gi of a source row
__device__ __forceinline__ uint16_t group_value(const RepackSrc &s, int which, int row, int gi, int groups,
                                                bool bias) {
  const uint16_t *src = bias ? s.b[which] : s.sc[which];
  if (!s.bits || !two_planes(s)) return src[(size_t)row * groups + gi];
  const int g = gi >> 1, src_groups = groups / 2;
  const uint16_t v = src[(size_t)row * src_groups + g];
  if (gi & 1) return bias ? (uint16_t)0 : v;  // low plane: s, bias 0
  if (bias) return v;                          // high plane: the bias
  const float f = __uint_as_float((uint32_t)v << 16) * 16.0f;  // 16 s, exact
  return (uint16_t)(__float_as_uint(f) >> 16);
}

// (source, row) of row r (0..15) of tile T; row < 0 for padding
__device__ __forceinline__ int src_row(const RepackSrc &s, int T, int r, int &which) {
  int row;
  if (s.gateup) {
    which = T & 1;
    row = 16 * (T >> 1) + r;
  } else {
    which = 0;
    row = 16 * T + r;
  }
  return row < s.n_src ? row : -1;
}

__device__ __forceinline__ uint32_t zero_code(const RepackSrc &s, int which, int row, int gi,
                                              int groups) {
  int zw = (groups + 7) / 8;
  uint32_t word = s.z[which][(size_t)row * zw + gi / 8];
  return (word >> (4 * (gi % 8))) & 0xFu;
}

__global__ void repack_codes_kernel(RepackSrc s, Layout L, uint32_t *out) {
  const size_t total = (size_t)L.tiles * L.chunks * 128;
  const int kw = L.K / 8;
  for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total;
       idx += (size_t)gridDim.x * blockDim.x) {
    const int sidx = (int)(idx & 3);
    const int lane = (int)((idx >> 2) & 31);
    const size_t tc = idx >> 7;
    const int c = (int)(tc % L.chunks);
    const int T = (int)(tc / L.chunks);
    const int g = lane >> 2, t = lane & 3;
    const int k0 = 64 * c + 16 * t + 4 * sidx;  // k0 % 8 is 0 or 4
    uint32_t src[2];
    for (int h = 0; h < 2; ++h) {
      int which;
      int row = src_row(s, T, g + 8 * h, which);
      if (row < 0) {
        src[h] = 0u;
      } else if (s.bits) {  // four codes k0 .. k0 + 3 as nibbles
        src[h] = 0u;
        for (int q = 0; q < 4; ++q) src[h] |= bits_code(s, which, row, k0 + q, L.group) << (4 * q);
      } else {
        src[h] = s.qw[which][(size_t)row * kw + k0 / 8] >> (4 * (k0 % 8));
      }
    }
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int kofs = 2 * ((j >> 1) & 1) + (j >> 2);
      const uint32_t code = (src[j & 1] >> (4 * kofs)) & 0xFu;
      word |= code << (4 * j);
    }
    out[idx] = word;
  }
}

// scale blocks, or with `bias` the bias blocks of the same layout
__global__ void repack_scales_kernel(RepackSrc s, Layout L, bool bias, uint16_t *out) {
  const size_t total = (size_t)L.tiles * L.gblocks * 64;
  for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total;
       idx += (size_t)gridDim.x * blockDim.x) {
    const int h = (int)(idx & 1);
    const int j = (int)((idx >> 1) & 3);
    const int g = (int)((idx >> 3) & 7);
    const size_t tb = idx >> 6;
    const int blk = (int)(tb % L.gblocks);
    const int T = (int)(tb / L.gblocks);
    const int gi = 4 * blk + j;
    int which;
    const int row = src_row(s, T, g + 8 * h, which);
    out[idx] = (row < 0 || gi >= L.groups) ? (uint16_t)0 : group_value(s, which, row, gi, L.groups, bias);
  }
}

__global__ void repack_zeros_kernel(RepackSrc s, Layout L, uint8_t *out) {
  const size_t total = (size_t)L.tiles * L.gblocks * 32;
  for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total;
       idx += (size_t)gridDim.x * blockDim.x) {
    const int j = (int)(idx & 3);
    const int g = (int)((idx >> 2) & 7);
    const size_t tb = idx >> 5;
    const int blk = (int)(tb % L.gblocks);
    const int T = (int)(tb / L.gblocks);
    const int gi = 4 * blk + j;
    uint32_t v = 0;
    if (gi < L.groups) {
      for (int h = 0; h < 2; ++h) {
        int which;
        const int row = src_row(s, T, g + 8 * h, which);
        if (row >= 0) v |= zero_code(s, which, row, gi, L.groups) << (4 * h);
      }
    }
    out[idx] = (uint8_t)v;
  }
}

// affine bias operand: row r (packed order), column j = bias(r, j / 3) for
// j < 3 * groups, else 0
__global__ void repack_bias_operand_kernel(RepackSrc s, Layout L, uint16_t *out) {
  const size_t total = (size_t)L.tiles * 16 * L.kb3;
  for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total;
       idx += (size_t)gridDim.x * blockDim.x) {
    const int j = (int)(idx % L.kb3);
    const size_t r = idx / L.kb3;
    const int T = (int)(r / 16), rr = (int)(r % 16);
    const int gi = j / 3;
    int which;
    const int row = src_row(s, T, rr, which);
    out[idx] = (row < 0 || gi >= L.groups) ? (uint16_t)0 : group_value(s, which, row, gi, L.groups, true);
  }
}

// w[n][k] = (q - z) * scale (exact), or scale * q + bias rounded once to
// float32 (affine), through the same unpack as the GEMM kernels
__global__ void dequantize_kernel(const uint8_t *packed, Layout L, int N, float *w, UnpackConsts uc) {
  const size_t total = (size_t)L.tiles * L.chunks * 32;
  const uint4 *codes = reinterpret_cast<const uint4 *>(packed + L.codes_off);
  const uint32_t *scales = reinterpret_cast<const uint32_t *>(packed + L.scales_off);
  const uint8_t *zeros = packed + L.zeros_off;
  const uint32_t *biases = reinterpret_cast<const uint32_t *>(packed + L.biases_off);
  const bool affine = L.sym == kFormAffine;
  for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total;
       idx += (size_t)gridDim.x * blockDim.x) {
    const int lane = (int)(idx & 31);
    const size_t tc = idx >> 5;
    const int c = (int)(tc % L.chunks);
    const int T = (int)(tc / L.chunks);
    const int g = lane >> 2, t = lane & 3;
    const int gi = (64 * c) / L.group;
    const size_t bi = ((size_t)T * L.gblocks + gi / 4) * 8 + g;
    const uint32_t sw = scales[bi * 4 + (gi & 3)];
    const float s_g = bf16lo_to_f32(sw), s_g8 = bf16hi_to_f32(sw);
    uint32_t zg, zg8;
    float b_g = 0.f, b_g8 = 0.f;
    if (affine) {
      zg = zg8 = zero_pair(0);
      const uint32_t bw = biases[bi * 4 + (gi & 3)];
      b_g = bf16lo_to_f32(bw);
      b_g8 = bf16hi_to_f32(bw);
    } else if (L.sym == kFormSym) {
      zg = zg8 = zero_pair(8);
    } else {
      const uint32_t zb = zeros[bi * 4 + (gi & 3)];
      zg = zero_pair(zb & 0xF);
      zg8 = zero_pair(zb >> 4);
    }
    const uint4 q = codes[idx];
    const uint32_t words[4] = {q.x, q.y, q.z, q.w};
    const int n0 = 16 * T + g, n1 = n0 + 8;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      uint32_t u[4];
      unpack_word(words[s], zg, zg8, uc, u);
      const int k = 64 * c + 16 * t + 4 * s;
      // u[0]: row g, k+0 / k+1; u[1]: row g+8, k+0 / k+1; u[2]: row g, k+2 / k+3; u[3]: row g+8
      // (q - z) * scale + 0 is the exact product; scale * q + bias one rounding
      if (n0 < N) {
        float *r = w + (size_t)n0 * L.K + k;
        r[0] = fmaf(bf16lo_to_f32(u[0]), s_g, b_g);
        r[1] = fmaf(bf16hi_to_f32(u[0]), s_g, b_g);
        r[2] = fmaf(bf16lo_to_f32(u[2]), s_g, b_g);
        r[3] = fmaf(bf16hi_to_f32(u[2]), s_g, b_g);
      }
      if (n1 < N) {
        float *r = w + (size_t)n1 * L.K + k;
        r[0] = fmaf(bf16lo_to_f32(u[1]), s_g8, b_g8);
        r[1] = fmaf(bf16hi_to_f32(u[1]), s_g8, b_g8);
        r[2] = fmaf(bf16lo_to_f32(u[3]), s_g8, b_g8);
        r[3] = fmaf(bf16hi_to_f32(u[3]), s_g8, b_g8);
      }
    }
  }
}

// the 4-bit code at (row n, packed column k) of the tiled layout
__device__ __forceinline__ uint32_t tiled_code(const uint8_t *packed, const Layout &L, int n, int k) {
  const int T = n / 16, r = n % 16, gg = r % 8, h = r / 8;
  const int c = k / 64, kk = k % 64, t = kk / 16, sidx = (kk % 16) / 4, koff = kk % 4;
  const int j = (koff == 0 ? 0 : koff == 1 ? 4 : koff == 2 ? 2 : 6) + h;  // kofs(j) = koff, row half h
  const uint32_t *codes = reinterpret_cast<const uint32_t *>(packed + L.codes_off);
  const uint32_t word = codes[(((size_t)T * L.chunks + c) * 32 + (4 * gg + t)) * 4 + sidx];
  return (word >> (4 * j)) & 0xFu;
}

// the bf16 scale (or bias, from `section`) of (row n, packed group gi)
__device__ __forceinline__ float tiled_group_value(const uint8_t *packed, size_t section, const Layout &L, int n,
                                                   int gi) {
  const int T = n / 16, r = n % 16, gg = r % 8, h = r / 8;
  const uint16_t *v = reinterpret_cast<const uint16_t *>(packed + section);
  const uint16_t b = v[(((size_t)T * L.gblocks + gi / 4) * 8 + gg) * 8 + (gi & 3) * 2 + h];
  return __uint_as_float((uint32_t)b << 16);
}

// w[n][k] = scale * q + bias of a b-bit affine weight, rounded once to
// float32, read back from its tiled planes: q = 16 qh + ql with qh, ql and
// their scales 16 s and s in packed groups 2g and 2g + 1 (bits 5-8), or the
// widened code itself (bits 2-4)
__global__ void dequantize_bits_kernel(const uint8_t *packed, Layout L, int N, int K, int bits, float *w) {
  const size_t total = (size_t)N * K;
  const int G = L.group;
  for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total;
       idx += (size_t)gridDim.x * blockDim.x) {
    const int n = (int)(idx / K), k = (int)(idx % K);
    const int g = k / G;
    float q, sc, bi;
    if (bits > 4) {
      const int khi = 2 * g * G + k % G;
      q = (float)(16 * tiled_code(packed, L, n, khi) + tiled_code(packed, L, n, khi + G));
      sc = tiled_group_value(packed, L.scales_off, L, n, 2 * g + 1);
      bi = tiled_group_value(packed, L.biases_off, L, n, 2 * g);
    } else {
      q = (float)tiled_code(packed, L, n, k);
      sc = tiled_group_value(packed, L.scales_off, L, n, g);
      bi = tiled_group_value(packed, L.biases_off, L, n, g);
    }
    w[idx] = fmaf(sc, q, bi);
  }
}

int grid_for(size_t work, int threads) {
  size_t b = (work + threads - 1) / threads;
  if (b > 65535u * 16u) b = 65535u * 16u;
  return (int)(b < 1 ? 1 : b);
}

}  // namespace

namespace {
cudaError_t launch_repack_src(RepackSrc &s, const Layout &L, uint8_t *packed, cudaStream_t stream);
}

cudaError_t launch_repack_affine_bits(const uint32_t *qw, const uint16_t *sc, const uint16_t *b, int N, int K,
                                      int bits, const Layout &L, uint8_t *packed, cudaStream_t stream) {
  RepackSrc s;
  s.qw[0] = s.qw[1] = qw;
  s.sc[0] = s.sc[1] = sc;
  s.z[0] = s.z[1] = nullptr;
  s.b[0] = s.b[1] = b;
  s.n_src = N;
  s.gateup = 0;
  s.bits = bits;
  s.k_src = K;
  return launch_repack_src(s, L, packed, stream);
}

cudaError_t launch_dequantize_affine_bits(const uint8_t *packed, const Layout &L, int N, int K, int bits, float *w,
                                          cudaStream_t stream) {
  const int th = 256;
  dequantize_bits_kernel<<<grid_for((size_t)N * K, th), th, 0, stream>>>(packed, L, N, K, bits, w);
  return cudaGetLastError();
}

cudaError_t launch_repack(const int32_t *qw0, const uint16_t *sc0, const int32_t *z0, const uint16_t *b0,
                          const int32_t *qw1, const uint16_t *sc1, const int32_t *z1, const uint16_t *b1,
                          int n_src, bool gateup, const Layout &L, uint8_t *packed,
                          cudaStream_t stream) {
  RepackSrc s;
  s.qw[0] = reinterpret_cast<const uint32_t *>(qw0);
  s.qw[1] = reinterpret_cast<const uint32_t *>(qw1 ? qw1 : qw0);
  s.sc[0] = sc0;
  s.sc[1] = sc1 ? sc1 : sc0;
  s.z[0] = reinterpret_cast<const uint32_t *>(z0);
  s.z[1] = reinterpret_cast<const uint32_t *>(z1 ? z1 : z0);
  s.b[0] = b0;
  s.b[1] = b1 ? b1 : b0;
  s.n_src = n_src;
  s.gateup = gateup ? 1 : 0;
  s.bits = 0;
  s.k_src = L.K;
  return launch_repack_src(s, L, packed, stream);
}

namespace {
cudaError_t launch_repack_src(RepackSrc &s, const Layout &L, uint8_t *packed, cudaStream_t stream) {
  const int th = 256;
  size_t nc = (size_t)L.tiles * L.chunks * 128;
  repack_codes_kernel<<<grid_for(nc, th), th, 0, stream>>>(s, L,
                                                          reinterpret_cast<uint32_t *>(packed + L.codes_off));
  size_t ns = (size_t)L.tiles * L.gblocks * 64;
  repack_scales_kernel<<<grid_for(ns, th), th, 0, stream>>>(
      s, L, false, reinterpret_cast<uint16_t *>(packed + L.scales_off));
  if (L.sym == kFormAffine) {
    repack_scales_kernel<<<grid_for(ns, th), th, 0, stream>>>(
        s, L, true, reinterpret_cast<uint16_t *>(packed + L.biases_off));
    const size_t nb = (size_t)L.tiles * 16 * L.kb3;
    repack_bias_operand_kernel<<<grid_for(nb, th), th, 0, stream>>>(
        s, L, reinterpret_cast<uint16_t *>(packed + L.bops_off));
  }
  if (L.sym == kFormZero) {
    size_t nz = (size_t)L.tiles * L.gblocks * 32;
    repack_zeros_kernel<<<grid_for(nz, th), th, 0, stream>>>(s, L, packed + L.zeros_off);
  }
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_dequantize(const uint8_t *packed, const Layout &L, int N, float *w,
                              cudaStream_t stream) {
  const int th = 256;
  size_t n = (size_t)L.tiles * L.chunks * 32;
  dequantize_kernel<<<grid_for(n, th), th, 0, stream>>>(packed, L, N, w, host_unpack_consts());
  return cudaGetLastError();
}

}  // namespace w4a16
