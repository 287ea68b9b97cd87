// Decode GEMM on the fifth-generation tensor cores (tcgen05), 1 <= M <= 32
// rows of x, zero-point and symmetric forms. Selected by kernel override 5;
// the mma.sync decode kernels stay the automatic choice (measured faster at
// M <= 16, and within 2 % at M = 32).
//
// The mma.sync decode kernels spend one m16n8k16 per packed word for every 8
// x rows, so their cost per word grows with M. Here the weight is the MMA's A
// operand (M = 128 weight rows) and lives in tensor memory; x rows, padded to
// 16 or 32, are the B operand (N = 16 or 32) in shared memory. The per-word
// work is the exact unpack and a store into TMEM, whatever M is:
//
//  * A producer thread streams each 128-row tile's codes (one tensor copy of
//    8 KB per 128-k stage), scale blocks and zero blocks once, evict-first.
//  * A loader warp stages x with 8-byte asynchronous copies, in the k order
//    that the TMEM layout of A below implies, into 128-byte-swizzled K-major
//    tiles.
//  * Four dequantising warps (one per 32-lane quarter of TMEM) rebuild
//    (q - z) exactly in bf16, with the three shifts, four LOP3s and four bf16x2
//    subtractions of the mma.sync kernels, and write the registers straight
//    into TMEM with the 16x256b store shape, which takes them in the mma.sync
//    fragment order: word s of lane 4g + t (rows g and g + 8, k = 16t + 4s ..
//    16t + 4s + 3) goes to columns 8s + 2t and 8s + 2t + 1. So TMEM column
//    8s + 2t + e of a 64-k chunk holds k = 16t + 4s + 2e + {0, 1}, and position
//    p of the s-th K = 16 MMA step is k = 16 (p / 4) + 4s + p % 4, the order in
//    which x is staged.
//  * Two threads issue tcgen05.mma (kind::f16, A from TMEM, fp32 D in TMEM)
//    for even and odd stages, one accumulator per 64-k chunk.
//  * Four epilogue warps fold each group's accumulators into fp32 registers
//    with the group's scale (one weight row per thread) and write the bf16
//    outputs.
//
// The dequantised weight never passes through shared memory, whose bandwidth
// would otherwise bound the stream (a store and a tensor-core read of 16 bytes
// per packed word). Long weights run as persistent CTAs, two per SM; short
// ones (few 128-row tiles) split K over the CTAs of a cluster, whose rank 0
// sums the partials in rank order through distributed shared memory.
//
// What paces it (measured with per-stage %globaltimer stamps): the round trip
// of a TMEM A stage (dequantise, hand over, issue eight MMAs, completion,
// hand back) takes ~1.5 us, and the 256 TMEM columns a CTA can hold beside
// its accumulators fit two or three such stages, so a CTA moves ~8 KB of
// codes per ~0.5 us. One 128 x N x 16 MMA (N <= 64) costs ~23 ns per issuing
// thread, A from TMEM or shared memory alike, so the tensor core itself would
// allow twice the copy peak.
//
// "2-16 rows ... INT4 weights and bf16 activations" is the DPAS verify GEMM of
// the GRIMOIRE v1.7 release notes ("What changed"); the group-wise scale fold
// and the exact code rebuild are those of the other decode kernels.
#include <algorithm>

#include "w4a16_internal.h"

namespace w4a16 {
namespace {

constexpr int kTcThreads = 384;      // 12 warps
constexpr int kTcRows = 128;         // weight rows per tile: the MMA's M
constexpr int kTcT16 = kTcRows / 16; // 16-row tiles of the packed layout per tile
constexpr int kStageChunks = 2;      // 64-wide K chunks per pipeline stage
// warp roles: the MMAs of even and odd stages are issued by two threads on
// different SM sub-partitions (measured no faster than one thread, which the
// round trip of a TMEM stage paces either way; kept since a stage then never
// waits for the previous stage's issue)
constexpr int kWarpProducer = 0, kWarpMma0 = 1, kWarpX = 3, kWarpDq0 = 4, kWarpFold0 = 8;

template <int NMMA, int SPG>
struct TcGeo {
  static constexpr int SC = 4;   // codes stages in flight
  static constexpr int SX = 8;   // x stages
  static constexpr int XD = 3;   // x copy groups the loader keeps in flight behind the newest
  static constexpr int SS = 2;   // scale (and zero) blocks of four groups
  static constexpr int SA = NMMA == 16 ? 3 : 2;  // A stages in TMEM, 64 columns each
  // D: one NMMA-column accumulator per 64-k chunk, so that the two chunks of
  // a stage are independent MMA chains; a group slot holds a group's SPG of
  // them, and a stage takes 2 / SPG group slots
  static constexpr int NB = (256 - SA * 64) / (SPG * NMMA);
  static constexpr int SPS = 2 / SPG;
  static constexpr int D_COL0 = SA * 64;
  static constexpr uint32_t TMEM_COLS = 256;
  static constexpr int Q_BYTES = kTcT16 * kStageChunks * kChunkBytes;  // 8 KB
  static constexpr int X_SUB = NMMA * 128;                               // one 64-k chunk of x
  static constexpr int X_BYTES = kStageChunks * X_SUB;
  static constexpr int S_BYTES = kTcT16 * kScaleBlockBytes;
  static constexpr int Z_BYTES = kTcT16 * kZeroBlockBytes;
  static constexpr int RED_BYTES = NMMA * kTcRows * 4;  // split-K partials [m][row], fp32
  static constexpr int OFF_X = 0;
  static constexpr int OFF_Q = OFF_X + SX * X_BYTES;
  static constexpr int OFF_S = OFF_Q + SC * Q_BYTES;
  static constexpr int OFF_Z = OFF_S + SS * S_BYTES;
  static constexpr int OFF_RED = OFF_Q;  // the codes ring, idle once every stage is consumed
  static constexpr int NBARS = 2 * SC + 2 * SX + 2 * SS + 2 * SA + 2 * NB + 1;
  static constexpr int OFF_BAR = OFF_Z + SS * Z_BYTES;
  static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
  static constexpr int SMEM_USED = OFF_MISC + 16;
  // at least 80 KB, so that no more than two CTAs share an SM and their TMEM
  // allocations (256 columns each) always fit in its 512
  static constexpr int SMEM_ALLOC = SMEM_USED + 1024 > 80 * 1024 ? SMEM_USED + 1024 : 80 * 1024;
  static_assert(D_COL0 + NB * SPG * NMMA <= (int)TMEM_COLS && NB >= 2 && (NB & (NB - 1)) == 0, "TMEM budget");
  static_assert(X_SUB % 1024 == 0 && OFF_Q % 1024 == 0, "swizzled x tiles need 1024-byte alignment");
  static_assert(RED_BYTES <= SC * Q_BYTES, "partials fit in the codes ring");
  static_assert(2 * (SMEM_ALLOC + 1024) <= 228 * 1024, "two CTAs per SM");
};

template <int NMMA, int SPG>
struct TcBars {
  using G = TcGeo<NMMA, SPG>;
  uint32_t base;
  __device__ uint32_t at(int i) const { return base + 8 * i; }
  __device__ uint32_t qfull(int i) const { return at(i); }
  __device__ uint32_t qempty(int i) const { return at(G::SC + i); }
  __device__ uint32_t xfull(int i) const { return at(2 * G::SC + i); }
  __device__ uint32_t xempty(int i) const { return at(2 * G::SC + G::SX + i); }
  __device__ uint32_t sfull(int i) const { return at(2 * G::SC + 2 * G::SX + i); }
  __device__ uint32_t sempty(int i) const { return at(2 * G::SC + 2 * G::SX + G::SS + i); }
  __device__ uint32_t afull(int i) const { return at(2 * G::SC + 2 * G::SX + 2 * G::SS + i); }
  __device__ uint32_t aempty(int i) const { return at(2 * G::SC + 2 * G::SX + 2 * G::SS + G::SA + i); }
  __device__ uint32_t dfull(int i) const { return at(2 * G::SC + 2 * G::SX + 2 * G::SS + 2 * G::SA + i); }
  __device__ uint32_t dempty(int i) const {
    return at(2 * G::SC + 2 * G::SX + 2 * G::SS + 2 * G::SA + G::NB + i);
  }
  __device__ uint32_t mma_done() const { return at(2 * G::SC + 2 * G::SX + 2 * G::SS + 2 * G::SA + 2 * G::NB); }
};

struct TcDecodeParams {
  const uint16_t *x;
  uint16_t *y;
  int M, N, K, ld;
  int tiles16;  // 16-row tiles of the packed layout
  int chunks;   // K / 64
  int spg;      // chunks per group (1 or 2)
  int ntiles;   // 128-row tiles
  int kc;       // CTAs of a cluster splitting one tile's K (1: persistent CTAs walking the tiles)
  int *err;
  UnpackConsts uc;
};

__device__ __forceinline__ void cp_async8(uint32_t dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint32_t tc_word(const uint4 &v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

__device__ __forceinline__ uint16_t tc_bf16_bits(float f) {
  __nv_bfloat16 b = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t *>(&b);
}

// every lane waits (each then has the barrier's acquire); false if any gave up
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
  return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, abort_flag));
}

__device__ __forceinline__ void give_up_tc(volatile int *abort_flag, int *err) {
  *abort_flag = 1;
  atomicExch(err, kErrTimeout);
}

template <int NC>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[NC]) {
  if constexpr (NC == 8) tmem_ld8(taddr, v);
  else if constexpr (NC == 16) tmem_ld16(taddr, v);
  else tmem_ld32(taddr, v);
}

// NMMA: x rows padded for the MMA (16 or 32); NC: D columns the epilogue
// reads (>= M); SPG: 64-k chunks per quantisation group (1 or 2).
// Every role walks the same sequence of 128-k stages; a stage's ring slots
// and barrier phases follow from its running index `st`.
template <int QF, int NMMA, int NC, int SPG>
__global__ void __launch_bounds__(kTcThreads, 2)
    smallm_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_s,
                     const __grid_constant__ CUtensorMap tm_z, const TcDecodeParams p) {
  using G = TcGeo<NMMA, SPG>;
  constexpr bool ZP = QF == kFormZero;
  constexpr int CPB = 4 * SPG;  // chunks per block of four groups
  static_assert(NC <= NMMA && (NC == 8 || NC == 16 || NC == 32), "epilogue columns");
  static_assert(SPG == 1 || SPG == 2, "group 64 or 128");
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const TcBars<NMMA, SPG> bars{sbase + G::OFF_BAR};
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + G::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + G::OFF_MISC + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // Work: persistent CTAs take tiles blockIdx.x, + gridDim.x, ... over all of
  // K; with a split, cluster c owns tile c and rank r its r-th share of the
  // blocks of four groups. Stages are 128 k from a block boundary, so that a
  // 128-wide group never straddles two (K is a multiple of the group).
  const bool split = p.kc > 1;
  const int part = split ? (int)cluster_ctarank() : 0;
  const int t0 = split ? (int)blockIdx.x / p.kc : (int)blockIdx.x;
  const int tstep = split ? p.ntiles : (int)gridDim.x;
  const int nblk = (p.chunks + CPB - 1) / CPB;
  const int c0 = split ? (int)((long long)nblk * part / p.kc) * CPB : 0;
  const int c1 = split ? min((int)((long long)nblk * (part + 1) / p.kc) * CPB, p.chunks) : p.chunks;

  if (tid == 0) {
    for (int i = 0; i < G::SC; ++i) {
      mbar_init(bars.qfull(i), 1);
      mbar_init(bars.qempty(i), 4);  // the dequantising warps
    }
    for (int i = 0; i < G::SX; ++i) {
      mbar_init(bars.xfull(i), 1);   // the loader warp
      mbar_init(bars.xempty(i), 1);  // MMA commit
    }
    for (int i = 0; i < G::SS; ++i) {
      mbar_init(bars.sfull(i), 1);
      mbar_init(bars.sempty(i), ZP ? 8 : 4);  // epilogue warps (+ dequantising warps reading zeros)
    }
    for (int i = 0; i < G::SA; ++i) {
      mbar_init(bars.afull(i), 4);
      mbar_init(bars.aempty(i), 1);
    }
    for (int i = 0; i < G::NB; ++i) {
      mbar_init(bars.dfull(i), 1);
      mbar_init(bars.dempty(i), 4);
    }
    mbar_init(bars.mma_done(), 2);  // both MMA threads
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma0) {
    tmem_alloc(smem_u32(tmem_slot), G::TMEM_COLS);
    tmem_relinquish();
  }
  // x rows M .. NMMA-1 of every stage are zero (written once, before the
  // tensor cores read any stage)
  for (int e = tid; e < G::SX * 2 * (NMMA - p.M) * 8; e += kTcThreads) {
    const int piece = e & 7, rest = e >> 3;
    const int row = p.M + rest % (NMMA - p.M), sc = rest / (NMMA - p.M);  // sc: stage * 2 + chunk
    sts128(sbase + G::OFF_X + sc * G::X_SUB + row * 128 + piece * 16, make_uint4(0, 0, 0, 0));
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_launch_dependents();

  float acc[NC];
#pragma unroll
  for (int m = 0; m < NC; ++m) acc[m] = 0.f;

  if (warp == kWarpProducer) {
    // ------------------------------------------------------------ producer
    // One tensor copy per stage: the codes of the tile's eight 16-row tiles
    // over 128 k (8 KB; a box past the last tile or the end of K is
    // zero-filled and counts in full), and one per block of four groups for
    // the scales (and zeros). The weights are constant: they stream before
    // the previous kernel on the stream has finished (programmatic overlap).
    if (lane == 0) {
      uint64_t pol;
      asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_s);
      if (ZP) tma_prefetch_desc(&tm_z);
      uint32_t st = 0, bk = 0;
      bool ok = true;
      for (int tile = t0; ok && tile < p.ntiles; tile += tstep) {
        const int j0 = tile * kTcT16;
        for (int ch = c0; ch < c1; ch += kStageChunks, ++st) {
          if (ch % CPB == 0) {
            const int s = bk % G::SS;
            if (!mbar_wait(bars.sempty(s), ((bk / G::SS) & 1) ^ 1, abort_flag)) { ok = false; break; }
            mbar_arrive_expect_tx(bars.sfull(s), G::S_BYTES + (ZP ? G::Z_BYTES : 0));
            const int blk = ch / CPB;
            tma_load_2d_hint(sbase + G::OFF_S + s * G::S_BYTES, &tm_s, blk * 32, j0, bars.sfull(s), pol);
            if (ZP) tma_load_2d_hint(sbase + G::OFF_Z + s * G::Z_BYTES, &tm_z, blk * 8, j0, bars.sfull(s), pol);
            ++bk;
          }
          const uint32_t s = st % G::SC;
          if (!mbar_wait(bars.qempty(s), ((st / G::SC) & 1) ^ 1, abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(bars.qfull(s), G::Q_BYTES);
          tma_load_2d_hint(sbase + G::OFF_Q + s * G::Q_BYTES, &tm_q, ch * 128, j0, bars.qfull(s), pol);
        }
      }
      if (!ok) {
        give_up_tc(abort_flag, p.err);
        // every copy issued lands before the CTA can exit
        for (uint32_t i = 0; i < G::SC && i < st; ++i) {
          const uint32_t u = st - 1 - i;
          mbar_wait_drain(bars.qfull(u % G::SC), (u / G::SC) & 1);
        }
        for (uint32_t i = 0; i < G::SS && i < bk; ++i) {
          const uint32_t u = bk - 1 - i;
          mbar_wait_drain(bars.sfull(u % G::SS), (u / G::SS) & 1);
        }
      }
    }
  } else if (warp < kWarpX) {
    // ------------------------------------------------------------ MMA issuers
    // Thread w issues the stages of parity w: the waits, eight
    // MMAs in two independent chains (one accumulator per 64-k chunk, issued
    // alternately), the commits.
    const uint32_t w = (uint32_t)(warp - kWarpMma0);
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kTcRows, NMMA);
      const uint32_t xbase = sbase + G::OFF_X, dbase = tmem + G::D_COL0;
      uint32_t st = 0;
      bool ok = true;
      for (int tile = t0; ok && tile < p.ntiles; tile += tstep) {
        for (int ch = c0; ch < c1; ch += kStageChunks, ++st) {
          if ((st & 1) != w) continue;
          const int nch = min(kStageChunks, c1 - ch);
          const uint32_t xsl = st % G::SX, as = st % G::SA, u0 = G::SPS * st, u1 = u0 + 1;
          const uint32_t a = tmem + as * 64;
          const uint32_t b0 = u0 % G::NB, b1 = u1 % G::NB;
          bool got = mbar_wait(bars.afull(as), (st / G::SA) & 1, abort_flag) &&
                     mbar_wait(bars.xfull(xsl), (st / G::SX) & 1, abort_flag) &&
                     mbar_wait(bars.dempty(b0), ((u0 / G::NB) & 1) ^ 1, abort_flag);
          // (a one-chunk last stage still cycles its second slot, so that
          // every slot's phases stay in step with the stage count)
          if (got && SPG == 1) got = mbar_wait(bars.dempty(b1), ((u1 / G::NB) & 1) ^ 1, abort_flag);
          if (!got) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d0 = dbase + b0 * (SPG * NMMA);
          const uint32_t d1 = SPG == 2 ? d0 + NMMA : dbase + b1 * NMMA;
          const uint64_t bd0 = sw128_desc(xbase + xsl * G::X_BYTES);
          const uint64_t bd1 = sw128_desc(xbase + xsl * G::X_BYTES + G::X_SUB);
          if (nch == 2) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              tc_mma_f16_ts(d0, a + 8 * j, bd0 + 2 * j, idesc, j != 0 ? 1u : 0u);
              tc_mma_f16_ts(d1, a + 32 + 8 * j, bd1 + 2 * j, idesc, j != 0 ? 1u : 0u);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) tc_mma_f16_ts(d0, a + 8 * j, bd0 + 2 * j, idesc, j != 0 ? 1u : 0u);
          }
          tc_commit(bars.dfull(b0));
          if (SPG == 1) tc_commit(bars.dfull(b1));
          tc_commit(bars.aempty(as));
          tc_commit(bars.xempty(xsl));
        }
      }
      if (!ok) give_up_tc(abort_flag, p.err);
      // every MMA issued has completed before TMEM is freed
      tc_commit(bars.mma_done());
      mbar_wait_drain(bars.mma_done(), 0);
    }
  } else if (warp == kWarpX) {
    // ------------------------------------------------------------ x loader
    // A stage's copies retire (wait_group) once the next XD stages are
    // issued; then the warp fences them into the async proxy and marks the
    // stage full. Its slot was freed SX - XD stages earlier, so the MMAs
    // never wait on this hand-off.
    grid_dependency_wait();
    // lane constants: 8-byte block beta of the staged row holds x's k-block
    // 4 (beta % 4) + beta / 4 of the chunk
    const int beta = lane & 15;
    const int kblk = 4 * (beta & 3) + (beta >> 2);
    const uint32_t lo8 = (uint32_t)(beta & 1) << 3;
    uint32_t st = 0;
    bool ok = true;
    for (int tile = t0; ok && tile < p.ntiles; tile += tstep) {
      for (int ch = c0; ch < c1; ch += kStageChunks, ++st) {
        const int nch = min(kStageChunks, c1 - ch);
        const uint32_t s = st % G::SX;
        if (!warp_wait(bars.xempty(s), ((st / G::SX) & 1) ^ 1, abort_flag)) { ok = false; break; }
        const uint32_t dst0 = sbase + G::OFF_X + s * G::X_BYTES;
        const uint16_t *src0 = p.x + (size_t)ch * 64 + 4 * kblk;
        if (nch == 2) {
          const int cc = lane >> 4;
          const uint32_t d0 = dst0 + cc * G::X_SUB + lo8;
          const uint16_t *s0 = src0 + 64 * cc;
          for (int m = 0; m < p.M; ++m)
            cp_async8(d0 + m * 128 + ((((uint32_t)beta >> 1) ^ (uint32_t)(m & 7)) << 4), s0 + (size_t)m * p.K);
        } else {
          for (int m = lane >> 4; m < p.M; m += 2)
            cp_async8(dst0 + lo8 + m * 128 + ((((uint32_t)beta >> 1) ^ (uint32_t)(m & 7)) << 4),
                      src0 + (size_t)m * p.K);
        }
        cp_async_commit();
        if (st >= (uint32_t)G::XD) {
          cp_async_wait<G::XD>();
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bars.xfull((st - G::XD) % G::SX));
        }
      }
    }
    cp_async_wait<0>();
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0)
      for (uint32_t u = st > (uint32_t)G::XD ? st - G::XD : 0; u < st; ++u) mbar_arrive(bars.xfull(u % G::SX));
    if (!ok && lane == 0) give_up_tc(abort_flag, p.err);
  } else if (warp < kWarpFold0) {
    // ------------------------------------------------------------ dequantising warps
    const int q = warp - kWarpDq0;  // TMEM lanes 32q .. 32q + 31: 16-row tiles 2q, 2q + 1
    const int g = lane >> 2;
    const UnpackConsts uc = p.uc;
    const uint32_t zsym = zero_pair(8);
    const uint32_t qbase = sbase + G::OFF_Q + (2 * q) * (kStageChunks * kChunkBytes) + lane * 16;
    const uint32_t tbase = tmem + ((uint32_t)(32 * q) << 16);
    uint32_t st = 0, bs = 0, bph = 0;
    bool ok = true;
    for (int tile = t0; ok && tile < p.ntiles; tile += tstep) {
      for (int ch = c0; ch < c1; ch += kStageChunks, ++st) {
        const int nch = min(kStageChunks, c1 - ch);
        const uint32_t qs = st % G::SC, as = st % G::SA;
        bool got = warp_wait(bars.qfull(qs), (st / G::SC) & 1, abort_flag) &&
                   warp_wait(bars.aempty(as), ((st / G::SA) & 1) ^ 1, abort_flag);
        if (got && ZP && ch % CPB == 0) got = warp_wait(bars.sfull(bs), bph, abort_flag);
        if (!got) { ok = false; break; }
        const uint32_t qa = qbase + qs * G::Q_BYTES;
        uint4 v[kStageChunks][2];
#pragma unroll
        for (int cc = 0; cc < kStageChunks; ++cc)
#pragma unroll
          for (int tt = 0; tt < 2; ++tt)
            v[cc][tt] = cc < nch ? lds128(qa + tt * (kStageChunks * kChunkBytes) + cc * kChunkBytes)
                                 : make_uint4(0, 0, 0, 0);
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.qempty(qs));
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < kStageChunks; ++cc) {
          if (cc >= nch) break;
#pragma unroll
          for (int tt = 0; tt < 2; ++tt) {
            uint32_t zg = zsym, zg8 = zsym;
            if (ZP) {
              const int gi = (ch + cc) / SPG;
              const uint32_t zb = lds8(sbase + G::OFF_Z + bs * G::Z_BYTES + (2 * q + tt) * kZeroBlockBytes +
                                       g * 4 + (gi & 3));
              zg = zero_pair(zb & 15u);
              zg8 = zero_pair(zb >> 4);
            }
            uint32_t r[16];
#pragma unroll
            for (int s = 0; s < 4; ++s) {
              uint32_t o[4];
              unpack_word(tc_word(v[cc][tt], s), zg, zg8, uc, o);
              r[4 * s + 0] = o[0];  // row g, k 16t + 4s + {0, 1}
              r[4 * s + 1] = o[2];  // row g, k 16t + 4s + {2, 3}
              r[4 * s + 2] = o[1];  // row g + 8
              r[4 * s + 3] = o[3];
            }
            tmem_st_16x256b_x4(tbase + ((uint32_t)(16 * tt) << 16) + as * 64 + cc * 32, r);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.afull(as));
        if (ZP && ((ch + nch) % CPB == 0 || ch + nch >= c1)) {
          if (lane == 0) mbar_arrive(bars.sempty(bs));
          if (++bs == (uint32_t)G::SS) { bs = 0; bph ^= 1; }
        }
      }
    }
    if (!ok && lane == 0) give_up_tc(abort_flag, p.err);
  } else {
    // ------------------------------------------------------------ epilogue warps
    const int q = warp - kWarpFold0;
    const int r = 32 * q + lane;  // weight row in the tile = TMEM lane
    const int jt = 2 * q + (lane >> 4), gq = lane & 7, h = (lane >> 3) & 1;
    const uint32_t sa0 = sbase + G::OFF_S + jt * kScaleBlockBytes + gq * 16 + h * 2;
    const uint32_t dbase = tmem + ((uint32_t)(32 * q) << 16) + G::D_COL0;
    grid_dependency_wait();
    uint32_t st = 0, bs = 0, bph = 0;
    bool ok = true;
    for (int tile = t0; ok && tile < p.ntiles; tile += tstep) {
      for (int ch = c0; ok && ch < c1; ch += kStageChunks, ++st) {
        const int nch = min(kStageChunks, c1 - ch);
        // the stage's groups: one (128-wide) or one per chunk
        for (int sub = 0; sub < G::SPS; ++sub) {
          const int gi = ch / SPG + sub;
          const uint32_t u = G::SPS * st + sub, b = u % G::NB;
          if (SPG == 1 && sub >= nch) {
            // the unused slot of a one-chunk last stage: pass its phase on
            if (!warp_wait(bars.dfull(b), (u / G::NB) & 1, abort_flag)) { ok = false; break; }
            if (lane == 0) mbar_arrive(bars.dempty(b));
            continue;
          }
          bool got = true;
          if ((gi & 3) == 0) got = warp_wait(bars.sfull(bs), bph, abort_flag);
          got = got && warp_wait(bars.dfull(b), (u / G::NB) & 1, abort_flag);
          if (!got) { ok = false; break; }
          tc_fence_after();
          const float s = __uint_as_float(lds16(sa0 + bs * G::S_BYTES + (gi & 3) * 4) << 16);
          // the group's chunk accumulators, each folded with the group's scale
#pragma unroll
          for (int c = 0; c < SPG; ++c) {
            float d[NC];
            tmem_ld_cols<NC>(dbase + b * (SPG * NMMA) + c * NMMA, d);
#pragma unroll
            for (int m = 0; m < NC; ++m) acc[m] = fmaf(s, d[m], acc[m]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bars.dempty(b));
          if ((gi & 3) == 3 || (gi + 1) * SPG >= c1) {
            if (lane == 0) mbar_arrive(bars.sempty(bs));
            if (++bs == (uint32_t)G::SS) { bs = 0; bph ^= 1; }
          }
        }
      }
      if (!ok) break;
      if (!split) {
        const int n = tile * kTcRows + r;
#pragma unroll
        for (int m = 0; m < NC; ++m) {
          if (m < p.M && n < p.N) p.y[(size_t)m * p.ld + n] = tc_bf16_bits(acc[m]);
          acc[m] = 0.f;
        }
      } else if (part != 0) {
#pragma unroll
        for (int m = 0; m < NC; ++m)
          if (m < p.M) sts32f(sbase + G::OFF_RED + (m * kTcRows + r) * 4, acc[m]);
      }
    }
    if (!ok && lane == 0) give_up_tc(abort_flag, p.err);
  }

  // ------------------------------------------------------------ tail
  __syncthreads();
  if (split) {
    // rank 0 sums the other ranks' partials in rank order, then they exit
    cluster_sync_all();
    if (part == 0 && warp >= kWarpFold0) {
      const int r = 32 * (warp - kWarpFold0) + lane;
      const int n = t0 * kTcRows + r;
#pragma unroll
      for (int m = 0; m < NC; ++m) {
        if (m >= p.M) break;
        float v = acc[m];
        for (int rk = 1; rk < p.kc; ++rk)
          v += ld_cluster_f32(mapa_shared(sbase + G::OFF_RED + (m * kTcRows + r) * 4, (uint32_t)rk));
        if (n < p.N) p.y[(size_t)m * p.ld + n] = tc_bf16_bits(v);
      }
    }
    cluster_sync_all();
  }
  if (warp == kWarpMma0) {
    tc_fence_after();
    tmem_dealloc(tmem, G::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// launch
// ---------------------------------------------------------------------------
struct TcMaps {
  CUtensorMap q, s, z;
};

template <int QF, int NMMA, int NC, int SPG>
cudaError_t launch_tc_variant(const TcMaps &tm, const TcDecodeParams &p, const GemmCall &c, int sm_count) {
  using G = TcGeo<NMMA, SPG>;
  auto kern = smallm_tc_kernel<QF, NMMA, NC, SPG>;
  static PerDevice configured;
  if (!configured.v[c.device].load(std::memory_order_relaxed)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    configured.v[c.device].store(1, std::memory_order_relaxed);
  }
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(p.kc > 1 ? (unsigned)(p.ntiles * p.kc) : (unsigned)std::min(p.ntiles, 2 * sm_count), 1, 1);
  lc.blockDim = dim3(kTcThreads, 1, 1);
  lc.dynamicSmemBytes = G::SMEM_ALLOC;
  lc.stream = c.stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (p.kc > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = p.kc;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (c.overlap) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  lc.attrs = attr;
  lc.numAttrs = na;
  return cudaLaunchKernelEx(&lc, kern, tm.q, tm.s, tm.z, p);
}

template <int QF, int SPG>
cudaError_t launch_tc_rows(const TcMaps &tm, const TcDecodeParams &p, const GemmCall &c, int sm_count) {
  if (p.M <= 8) return launch_tc_variant<QF, 16, 8, SPG>(tm, p, c, sm_count);
  if (p.M <= 16) return launch_tc_variant<QF, 16, 16, SPG>(tm, p, c, sm_count);
  return launch_tc_variant<QF, 32, 32, SPG>(tm, p, c, sm_count);
}

template <int QF>
cudaError_t launch_tc_form(const TcMaps &tm, const TcDecodeParams &p, const GemmCall &c, int sm_count) {
  return p.spg == 1 ? launch_tc_rows<QF, 1>(tm, p, c, sm_count) : launch_tc_rows<QF, 2>(tm, p, c, sm_count);
}

}  // namespace

bool smallm_tc_supports(const GemmCall &c) {
  return c.M >= 1 && c.M <= 32 && !c.gateup && !c.amax && (c.sym == kFormZero || c.sym == kFormSym);
}

cudaError_t launch_smallm_tc(const GemmCall &c, int sm_count) {
  if (!smallm_tc_supports(c)) return cudaErrorInvalidValue;
  const Layout L = make_layout(c.N, c.K, c.group, c.sym);
  // codes: per 16-row tile a row of chunks x 128 words, 2 chunks x 8 tiles
  // per box; scale and zero blocks: 32 and 8 words per block, 8 tiles
  TcMaps tm;
  bool ok = encode_2d(&tm.q, CU_TENSOR_MAP_DATA_TYPE_UINT32, c.packed + L.codes_off, (uint64_t)L.chunks * 128,
                      (uint64_t)L.tiles, (uint64_t)L.chunks * kChunkBytes, kStageChunks * 128, kTcT16,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
  ok = ok && encode_2d(&tm.s, CU_TENSOR_MAP_DATA_TYPE_UINT32, c.packed + L.scales_off, (uint64_t)L.gblocks * 32,
                       (uint64_t)L.tiles, (uint64_t)L.gblocks * kScaleBlockBytes, 32, kTcT16,
                       CU_TENSOR_MAP_SWIZZLE_NONE);
  tm.z = tm.s;
  if (c.sym == kFormZero)
    ok = ok && encode_2d(&tm.z, CU_TENSOR_MAP_DATA_TYPE_UINT32, c.packed + L.zeros_off, (uint64_t)L.gblocks * 8,
                         (uint64_t)L.tiles, (uint64_t)L.gblocks * kZeroBlockBytes, 8, kTcT16,
                         CU_TENSOR_MAP_SWIZZLE_NONE);
  if (!ok) return cudaErrorInvalidValue;
  TcDecodeParams p;
  p.x = c.x;
  p.y = c.y;
  p.M = c.M;
  p.N = c.N;
  p.K = c.K;
  p.ld = c.N;
  p.tiles16 = L.tiles;
  p.chunks = L.chunks;
  p.spg = c.group / kChunkK;
  p.ntiles = (c.N + kTcRows - 1) / kTcRows;
  p.err = c.err;
  p.uc = host_unpack_consts();
  // Split K over a cluster when the tiles fill less than half of the two CTA
  // slots per SM: as many ranks (<= 8) as fit in one wave, each with at least
  // two blocks of four groups.
  p.kc = 1;
  const int slots = 2 * sm_count;
  const int nblk = (L.chunks + 4 * p.spg - 1) / (4 * p.spg);
  if (p.ntiles * 2 <= slots) {
    p.kc = std::min(8, slots / p.ntiles);
    while (p.kc > 1 && nblk < 2 * p.kc) --p.kc;
  }
  return c.sym == kFormSym ? launch_tc_form<kFormSym>(tm, p, c, sm_count)
                           : launch_tc_form<kFormZero>(tm, p, c, sm_count);
}

}  // namespace w4a16
