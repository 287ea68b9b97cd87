// Decode-regime kernels, M <= 16 rows of x against the whole weight.
//
// Both kernels stream the repacked weight exactly once per call (HBM-bound),
// each lane issuing one 16-byte load per 16-row tile and 64-wide K chunk, and
// turn nibbles into exact (q - z) values in registers:
//
//  * smallm_mma_kernel (M = 1..16): the two rows x 16 k a lane holds are the
//    A fragment of mma.sync m16n8k16 (bf16 in, f32 accumulate) after the
//    bf16 rebuild; x rows are the B fragment (zero rows above M). One group's
//    products sum in a fresh accumulator, then acc += scale * partial in
//    float32. "2-16 rows ... INT4 weights and bf16 activations" is the DPAS
//    verify GEMM of the GRIMOIRE v1.7 release notes ("What changed"), and the
//    same pages' v1.8 notes ("INT4 verify faster") show it occupancy-bound:
//    here the weight tile is read once for all rows and unpacked once.
//  * gemv_m1_kernel (M = 1): CUDA-core form. Each nibble is rebuilt as a
//    float32 2^23 + q * 16^p by OR-ing the magic exponent onto it in place
//    (one LOP3, no shift for the low five nibbles), the constant 2^23 + z * 16^p
//    is subtracted exactly, the product with x accumulates in float32 (packed
//    f32x2 FMA), and the 16^-p factor is applied once per group. Lanes then
//    meet by warp shuffles (the single-user ESIMD GEMV of the same v1.7 notes).
//
// Split-K: KW warps of a CTA take disjoint K slices of the same tiles and sum
// through shared memory; for short N, KC CTAs of a cluster split K further and
// rank 0 sums the others' partials through distributed shared memory, in rank
// order (split-K by clusters on sm_90+, as in TensorFold PR #859, "What this
// changes"). Sums never use atomics, so results are bitwise reproducible.
#include "w4a16_internal.h"

namespace w4a16 {
namespace {

constexpr int kMaxWarps = 8;

struct DecodeParams {
  const uint16_t *x;
  const uint4 *codes;
  const uint32_t *scales;  // [tile][gblock][g][4 groups] words of (row g | row g+8 << 16)
  const uint32_t *zeros;   // [tile][gblock][g] words of 4 bytes (row g | row g+8 << 4)
  uint16_t *y;
  int M, N, K;             // N: output columns (N_each for gate/up)
  int tiles, chunks, groups, gblocks;
  int ld;                  // y row stride in elements
};

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 ldg_stream(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint4 ldg_keep(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ldg_u32(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  __nv_bfloat16 b = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t *>(&b);
}

__device__ __forceinline__ float silu_f32(float g) { return g / (1.0f + __expf(-g)); }

// Slice [g0, g1) of the K groups for this warp.
__device__ __forceinline__ void k_slice(int groups, int &g0, int &g1) {
  const int kw = blockDim.x >> 5;
  const int nsl = gridDim.y * kw;
  const int sidx = blockIdx.y * kw + (threadIdx.x >> 5);
  g0 = (int)((long long)groups * sidx / nsl);
  g1 = (int)((long long)groups * (sidx + 1) / nsl);
}

// Sum the per-warp partials red[w][e] (w < KW) into red[0][e]; with a cluster,
// rank 0 then adds every other rank's red[0][e] in rank order. Returns true in
// the CTA that must write the outputs.
template <int E>
__device__ __forceinline__ bool reduce_partials(float (*red)[E]) {
  const int kw = blockDim.x >> 5;
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float s = red[0][e];
    for (int w = 1; w < kw; ++w) s += red[w][e];
    red[0][e] = s;
  }
  if (gridDim.y == 1) {
    __syncthreads();
    return true;
  }
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
  uint32_t rank;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  if (rank == 0) {
    const uint32_t nranks = gridDim.y;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      float s = red[0][e];
      const uint32_t local = smem_u32(&red[0][e]);
      for (uint32_t r = 1; r < nranks; ++r) {
        uint32_t remote;
        float v;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(r));
        asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
        s += v;
      }
      red[0][e] = s;
    }
  }
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
  __syncthreads();
  return rank == 0;
}

// ---------------------------------------------------------------------------
// small-M tensor-core kernel
// ---------------------------------------------------------------------------
template <int MT, int TPW, bool SYM, int CPG, int PF, bool GATEUP>
__global__ void __launch_bounds__(256) smallm_mma_kernel(DecodeParams p) {
  constexpr int E = TPW * MT * 4 * 32;
  __shared__ float red[kMaxWarps][E];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int tile0 = blockIdx.x * TPW;
  int gb, ge;
  k_slice(p.groups, gb, ge);

  const uint4 *wp[TPW];
  const uint32_t *sp[TPW];
  const uint32_t *zp[TPW];
#pragma unroll
  for (int i = 0; i < TPW; ++i) {
    const int tile = min(tile0 + i, p.tiles - 1);
    wp[i] = p.codes + (size_t)tile * p.chunks * 32 + lane;
    sp[i] = p.scales + ((size_t)tile * p.gblocks * 8 + g) * 4;
    zp[i] = p.zeros + ((size_t)tile * p.gblocks * 8 + g);
  }
  // x rows g and g + 8 (B fragment columns); rows >= M stay zero
  const uint4 *xp[MT];
  bool xv[MT];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    const int m = g + 8 * mt;
    xv[mt] = m < p.M;
    xp[mt] = reinterpret_cast<const uint4 *>(p.x + (size_t)(xv[mt] ? m : 0) * p.K + 16 * t);
  }

  float acc[TPW][MT][4];
#pragma unroll
  for (int i = 0; i < TPW; ++i)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[i][mt][r] = 0.f;

  // prefetch ring: weights, x fragments and scale / zero words of PF groups
  uint4 rw[PF][CPG][TPW];
  uint4 rx[PF][CPG][MT][2];
  uint32_t rs[PF][TPW], rz[PF][TPW];

  auto load_group = [&](int gg, uint4 (&w)[CPG][TPW], uint4 (&xx)[CPG][MT][2], uint32_t (&s)[TPW],
                        uint32_t (&z)[TPW]) {
#pragma unroll
    for (int cc = 0; cc < CPG; ++cc) {
      const int c = gg * CPG + cc;
#pragma unroll
      for (int i = 0; i < TPW; ++i) w[cc][i] = ldg_stream(wp[i] + (size_t)c * 32);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        if (xv[mt]) {
          xx[cc][mt][0] = ldg_keep(xp[mt] + (size_t)c * 8);
          xx[cc][mt][1] = ldg_keep(xp[mt] + (size_t)c * 8 + 1);
        } else {
          xx[cc][mt][0] = make_uint4(0, 0, 0, 0);
          xx[cc][mt][1] = make_uint4(0, 0, 0, 0);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < TPW; ++i) {
      s[i] = ldg_u32(sp[i] + (size_t)(gg >> 2) * 32 + (gg & 3));
      z[i] = SYM ? 0u : ldg_u32(zp[i] + (size_t)(gg >> 2) * 8);
    }
  };

#pragma unroll
  for (int d = 0; d < PF; ++d)
    if (gb + d < ge) load_group(gb + d, rw[d], rx[d], rs[d], rz[d]);

  for (int gi = gb; gi < ge; gi += PF) {
#pragma unroll
    for (int d = 0; d < PF; ++d) {
      const int gg = gi + d;
      if (gg < ge) {
        uint4 w[CPG][TPW];
        uint4 xx[CPG][MT][2];
        uint32_t s[TPW], z[TPW];
#pragma unroll
        for (int cc = 0; cc < CPG; ++cc) {
#pragma unroll
          for (int i = 0; i < TPW; ++i) w[cc][i] = rw[d][cc][i];
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            xx[cc][mt][0] = rx[d][cc][mt][0];
            xx[cc][mt][1] = rx[d][cc][mt][1];
          }
        }
#pragma unroll
        for (int i = 0; i < TPW; ++i) {
          s[i] = rs[d][i];
          z[i] = rz[d][i];
        }
        if (gg + PF < ge) load_group(gg + PF, rw[d], rx[d], rs[d], rz[d]);

        uint32_t zg[TPW], zg8[TPW];
#pragma unroll
        for (int i = 0; i < TPW; ++i) {
          if (SYM) {
            zg[i] = zg8[i] = zero_pair(8);
          } else {
            const uint32_t zb = (z[i] >> (8 * (gg & 3))) & 0xFFu;
            zg[i] = zero_pair(zb & 0xF);
            zg8[i] = zero_pair(zb >> 4);
          }
        }
        float part[TPW][MT][4];
#pragma unroll
        for (int i = 0; i < TPW; ++i)
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int r = 0; r < 4; ++r) part[i][mt][r] = 0.f;
#pragma unroll
        for (int cc = 0; cc < CPG; ++cc) {
#pragma unroll
          for (int st = 0; st < 4; ++st) {
            // B fragment: x words 2st (k+0, k+1) and 2st+1 (k+2, k+3) of this lane's 16 k
            uint32_t b0[MT], b1[MT];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              const uint4 &xh = xx[cc][mt][st >> 1];
              b0[mt] = word_of(xh, 2 * (st & 1));
              b1[mt] = word_of(xh, 2 * (st & 1) + 1);
            }
#pragma unroll
            for (int i = 0; i < TPW; ++i) {
              uint32_t a[4];
              unpack_word(word_of(w[cc][i], st), zg[i], zg8[i], a);
#pragma unroll
              for (int mt = 0; mt < MT; ++mt) mma_bf16_16816(part[i][mt], a, b0[mt], b1[mt]);
            }
          }
        }
#pragma unroll
        for (int i = 0; i < TPW; ++i) {
          const float sg = bf16lo_to_f32(s[i]), sg8 = bf16hi_to_f32(s[i]);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            acc[i][mt][0] = fmaf(sg, part[i][mt][0], acc[i][mt][0]);
            acc[i][mt][1] = fmaf(sg, part[i][mt][1], acc[i][mt][1]);
            acc[i][mt][2] = fmaf(sg8, part[i][mt][2], acc[i][mt][2]);
            acc[i][mt][3] = fmaf(sg8, part[i][mt][3], acc[i][mt][3]);
          }
        }
      }
    }
  }

#pragma unroll
  for (int i = 0; i < TPW; ++i)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int r = 0; r < 4; ++r) red[warp][((i * MT + mt) * 4 + r) * 32 + lane] = acc[i][mt][r];

  if (!reduce_partials<E>(red)) return;

  // element e = ((i*MT + mt)*4 + r)*32 + lane:
  //   row n = 16*(tile0+i) + g + 8*(r>>1), column m = 8*mt + 2t + (r&1)
  constexpr int EO = GATEUP ? E / 2 : E;  // gate/up: tile 0 gate, tile 1 up
  for (int e = threadIdx.x; e < EO; e += blockDim.x) {
    const int ln = e & 31, r = (e >> 5) & 3, im = e >> 7;
    const int mt = im % MT, i = im / MT;
    const int m = 8 * mt + 2 * (ln & 3) + (r & 1);
    const int nl = (ln >> 2) + 8 * (r >> 1);
    if (m >= p.M) continue;
    if (GATEUP) {
      const int n = 16 * (tile0 >> 1) + nl;
      if (n < p.N) {
        const float gv = red[0][e], uv = red[0][e + MT * 4 * 32];
        p.y[(size_t)m * p.ld + n] = f32_to_bf16_bits(silu_f32(gv) * uv);
      }
    } else {
      const int n = 16 * (tile0 + i) + nl;
      if (n < p.N) p.y[(size_t)m * p.ld + n] = f32_to_bf16_bits(red[0][e]);
    }
  }
}

// ---------------------------------------------------------------------------
// one-row CUDA-core GEMV
// ---------------------------------------------------------------------------
template <int TPW, bool SYM, int CPG, int PF>
__global__ void __launch_bounds__(256) gemv_m1_kernel(DecodeParams p) {
  constexpr int E = TPW * 2 * 8;  // (tile, row half, g)
  __shared__ float red[kMaxWarps][E];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int tile0 = blockIdx.x * TPW;
  int gb, ge;
  k_slice(p.groups, gb, ge);

  const uint4 *wp[TPW];
  const uint32_t *sp[TPW];
  const uint32_t *zp[TPW];
#pragma unroll
  for (int i = 0; i < TPW; ++i) {
    const int tile = min(tile0 + i, p.tiles - 1);
    wp[i] = p.codes + (size_t)tile * p.chunks * 32 + lane;
    sp[i] = p.scales + ((size_t)tile * p.gblocks * 8 + g) * 4;
    zp[i] = p.zeros + ((size_t)tile * p.gblocks * 8 + g);
  }
  const uint4 *xp = reinterpret_cast<const uint4 *>(p.x + 16 * t);

  float out[TPW][2];
#pragma unroll
  for (int i = 0; i < TPW; ++i) out[i][0] = out[i][1] = 0.f;

  uint4 rw[PF][CPG][TPW];
  uint4 rx[PF][CPG][2];
  uint32_t rs[PF][TPW], rz[PF][TPW];
  auto load_group = [&](int gg, uint4 (&w)[CPG][TPW], uint4 (&xx)[CPG][2], uint32_t (&s)[TPW],
                        uint32_t (&z)[TPW]) {
#pragma unroll
    for (int cc = 0; cc < CPG; ++cc) {
      const int c = gg * CPG + cc;
#pragma unroll
      for (int i = 0; i < TPW; ++i) w[cc][i] = ldg_stream(wp[i] + (size_t)c * 32);
      xx[cc][0] = ldg_keep(xp + (size_t)c * 8);
      xx[cc][1] = ldg_keep(xp + (size_t)c * 8 + 1);
    }
#pragma unroll
    for (int i = 0; i < TPW; ++i) {
      s[i] = ldg_u32(sp[i] + (size_t)(gg >> 2) * 32 + (gg & 3));
      z[i] = SYM ? 0u : ldg_u32(zp[i] + (size_t)(gg >> 2) * 8);
    }
  };
#pragma unroll
  for (int d = 0; d < PF; ++d)
    if (gb + d < ge) load_group(gb + d, rw[d], rx[d], rs[d], rz[d]);

  constexpr uint32_t kMagic = 0x4B000000u;  // float32 2^23: mantissa step 1
  for (int gi = gb; gi < ge; gi += PF) {
#pragma unroll
    for (int d = 0; d < PF; ++d) {
      const int gg = gi + d;
      if (gg < ge) {
        uint4 w[CPG][TPW];
        uint4 xx[CPG][2];
        uint32_t s[TPW], z[TPW];
#pragma unroll
        for (int cc = 0; cc < CPG; ++cc) {
#pragma unroll
          for (int i = 0; i < TPW; ++i) w[cc][i] = rw[d][cc][i];
          xx[cc][0] = rx[d][cc][0];
          xx[cc][1] = rx[d][cc][1];
        }
#pragma unroll
        for (int i = 0; i < TPW; ++i) {
          s[i] = rs[d][i];
          z[i] = rz[d][i];
        }
        if (gg + PF < ge) load_group(gg + PF, rw[d], rx[d], rs[d], rz[d]);

        // nibble j of a word: row g + 8*(j&1), class p(j) (its place 16^p), k offset kofs(j)
        //   j : 0 1 2 3 4 5 6 7
        //   p : 0 1 2 3 4 0 1 2      (j = 5..7 are read from the word shifted right by 20)
        // -(2^23 + z * 16^p(j)) is added exactly (both operands are integers below 2^24).
        float2 cz[4];
        float2 part[TPW][4];  // pairs (j=0,1) (2,3) (4,5) (6,7)
#pragma unroll
        for (int i = 0; i < TPW; ++i)
#pragma unroll
          for (int q = 0; q < 4; ++q) part[i][q] = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < TPW; ++i) {
          uint32_t za = 8, zb = 8;
          if (!SYM) {
            const uint32_t zbyte = (z[i] >> (8 * (gg & 3))) & 0xFFu;
            za = zbyte & 0xF;
            zb = zbyte >> 4;
          }
          constexpr uint32_t kNeg = 0x80000000u;
          cz[0] = make_float2(__uint_as_float(kNeg | kMagic | za), __uint_as_float(kNeg | kMagic | (zb << 4)));
          cz[1] = make_float2(__uint_as_float(kNeg | kMagic | (za << 8)),
                              __uint_as_float(kNeg | kMagic | (zb << 12)));
          cz[2] = make_float2(__uint_as_float(kNeg | kMagic | (za << 16)), __uint_as_float(kNeg | kMagic | zb));
          cz[3] = make_float2(__uint_as_float(kNeg | kMagic | (za << 4)),
                              __uint_as_float(kNeg | kMagic | (zb << 8)));
#pragma unroll
          for (int cc = 0; cc < CPG; ++cc) {
#pragma unroll
            for (int st = 0; st < 4; ++st) {
              const uint32_t wd = word_of(w[cc][i], st);
              const uint32_t w20 = wd >> 20;
              const uint32_t xa = word_of(xx[cc][st >> 1], 2 * (st & 1));      // k+0, k+1
              const uint32_t xb = word_of(xx[cc][st >> 1], 2 * (st & 1) + 1);  // k+2, k+3
              const float x0 = bf16lo_to_f32(xa), x1 = bf16hi_to_f32(xa);
              const float x2 = bf16lo_to_f32(xb), x3 = bf16hi_to_f32(xb);
              const float2 v01 = make_float2(__uint_as_float(kMagic | (wd & 0xFu)),
                                             __uint_as_float(kMagic | (wd & 0xF0u)));
              const float2 v23 = make_float2(__uint_as_float(kMagic | (wd & 0xF00u)),
                                             __uint_as_float(kMagic | (wd & 0xF000u)));
              const float2 v45 = make_float2(__uint_as_float(kMagic | (wd & 0xF0000u)),
                                             __uint_as_float(kMagic | (w20 & 0xFu)));
              const float2 v67 = make_float2(__uint_as_float(kMagic | (w20 & 0xF0u)),
                                             __uint_as_float(kMagic | (w20 & 0xF00u)));
              // j=0,1 at k+0; j=2,3 at k+2; j=4,5 at k+1; j=6,7 at k+3
              part[i][0] = __ffma2_rn(make_float2(x0, x0), __fadd2_rn(v01, cz[0]), part[i][0]);
              part[i][1] = __ffma2_rn(make_float2(x2, x2), __fadd2_rn(v23, cz[1]), part[i][1]);
              part[i][2] = __ffma2_rn(make_float2(x1, x1), __fadd2_rn(v45, cz[2]), part[i][2]);
              part[i][3] = __ffma2_rn(make_float2(x3, x3), __fadd2_rn(v67, cz[3]), part[i][3]);
            }
          }
          // undo the 16^p places: row g gets j = 0, 2, 4, 6 (p = 0, 2, 4, 1),
          // row g + 8 gets j = 1, 3, 5, 7 (p = 1, 3, 0, 2)
          const float rg = part[i][0].x + part[i][1].x * 0x1p-8f + part[i][2].x * 0x1p-16f +
                           part[i][3].x * 0x1p-4f;
          const float rg8 = part[i][0].y * 0x1p-4f + part[i][1].y * 0x1p-12f + part[i][2].y +
                            part[i][3].y * 0x1p-8f;
          out[i][0] = fmaf(bf16lo_to_f32(s[i]), rg, out[i][0]);
          out[i][1] = fmaf(bf16hi_to_f32(s[i]), rg8, out[i][1]);
        }
      }
    }
  }

  // the four lanes t = 0..3 of each g hold disjoint k of the same two rows
#pragma unroll
  for (int i = 0; i < TPW; ++i)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float v = out[i][h];
      v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
      v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
      out[i][h] = v;
    }
  if (t == 0) {
#pragma unroll
    for (int i = 0; i < TPW; ++i)
#pragma unroll
      for (int h = 0; h < 2; ++h) red[warp][(i * 2 + h) * 8 + g] = out[i][h];
  }
  if (!reduce_partials<E>(red)) return;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int gq = e & 7, h = (e >> 3) & 1, i = e >> 4;
    const int n = 16 * (tile0 + i) + gq + 8 * h;
    if (n < p.N) p.y[n] = f32_to_bf16_bits(red[0][e]);
  }
}

// ---------------------------------------------------------------------------
// launch configuration
// ---------------------------------------------------------------------------
struct DecodeCfg {
  int tpw, kw, kc;
};

DecodeCfg pick_cfg(int tiles, int groups, int sm_count, int tpw) {
  DecodeCfg c;
  c.tpw = tpw;
  c.kw = 4;
  const int ctas = (tiles + tpw - 1) / tpw;
  // aim for about 16 resident warps per SM so enough 16-byte loads are in flight
  const long long target = (long long)sm_count * 16;
  c.kc = 1;
  while (c.kc < 8 && (long long)ctas * c.kw * c.kc < target && groups >= 4 * c.kw * c.kc) c.kc *= 2;
  return c;
}

template <typename Kern>
cudaError_t launch_decode(Kern kern, const DecodeParams &prm, const DecodeCfg &cfg,
                          cudaStream_t stream) {
  const int ctas = (prm.tiles + cfg.tpw - 1) / cfg.tpw;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(ctas, cfg.kc, 1);
  lc.blockDim = dim3(32 * cfg.kw, 1, 1);
  lc.dynamicSmemBytes = 0;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  int na = 0;
  if (cfg.kc > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = cfg.kc;
    attr[0].val.clusterDim.z = 1;
    na = 1;
  }
  lc.attrs = attr;
  lc.numAttrs = na;
  return cudaLaunchKernelEx(&lc, kern, prm);
}

DecodeParams make_params(const GemmCall &c, const Layout &L) {
  DecodeParams p;
  p.x = c.x;
  p.codes = reinterpret_cast<const uint4 *>(c.packed + L.codes_off);
  p.scales = reinterpret_cast<const uint32_t *>(c.packed + L.scales_off);
  p.zeros = reinterpret_cast<const uint32_t *>(c.packed + (c.sym ? L.scales_off : L.zeros_off));
  p.y = c.y;
  p.M = c.M;
  p.N = c.N;
  p.K = c.K;
  p.tiles = L.tiles;
  p.chunks = L.chunks;
  p.groups = L.groups;
  p.gblocks = L.gblocks;
  p.ld = c.N;
  return p;
}

template <int MT, bool SYM, int CPG, bool GATEUP>
cudaError_t run_mma(const DecodeParams &p, const DecodeCfg &cfg, cudaStream_t s) {
  constexpr int PF = (MT == 1 ? 4 : 2) / CPG;
  return launch_decode(smallm_mma_kernel<MT, 2, SYM, CPG, PF, GATEUP>, p, cfg, s);
}

template <bool SYM, int CPG, bool GATEUP>
cudaError_t run_mma_m(const DecodeParams &p, const DecodeCfg &cfg, cudaStream_t s) {
  return p.M <= 8 ? run_mma<1, SYM, CPG, GATEUP>(p, cfg, s) : run_mma<2, SYM, CPG, GATEUP>(p, cfg, s);
}

template <bool GATEUP>
cudaError_t run_mma_all(const DecodeParams &p, const DecodeCfg &cfg, int sym, int group,
                        cudaStream_t s) {
  if (sym) {
    return group == 64 ? run_mma_m<true, 1, GATEUP>(p, cfg, s) : run_mma_m<true, 2, GATEUP>(p, cfg, s);
  }
  return group == 64 ? run_mma_m<false, 1, GATEUP>(p, cfg, s) : run_mma_m<false, 2, GATEUP>(p, cfg, s);
}

}  // namespace

cudaError_t launch_smallm_mma(const GemmCall &c, int sm_count) {
  const Layout L = make_layout(packed_rows(c), c.K, c.group, c.sym);
  DecodeParams p = make_params(c, L);
  const DecodeCfg cfg = pick_cfg(L.tiles, L.groups, sm_count, 2);
  if (c.gateup) return run_mma_all<true>(p, cfg, c.sym, c.group, c.stream);
  return run_mma_all<false>(p, cfg, c.sym, c.group, c.stream);
}

cudaError_t launch_gemv_m1(const GemmCall &c, int sm_count) {
  const Layout L = make_layout(packed_rows(c), c.K, c.group, c.sym);
  DecodeParams p = make_params(c, L);
  const DecodeCfg cfg = pick_cfg(L.tiles, L.groups, sm_count, 2);
  if (c.sym) {
    return c.group == 64 ? launch_decode(gemv_m1_kernel<2, true, 1, 4>, p, cfg, c.stream)
                         : launch_decode(gemv_m1_kernel<2, true, 2, 2>, p, cfg, c.stream);
  }
  return c.group == 64 ? launch_decode(gemv_m1_kernel<2, false, 1, 4>, p, cfg, c.stream)
                       : launch_decode(gemv_m1_kernel<2, false, 2, 2>, p, cfg, c.stream);
}

}  // namespace w4a16
