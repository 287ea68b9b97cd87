// Prompt-regime GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
//   y[m][n] = sum_g scale[n][g] * sum_{k in g} x[m][k] * (q[n][k] - z[n][g])
//
// The integer (q - z) is exact in bf16 and each product with a bf16 x is exact
// in float32, so the tensor core sums one group's products into a TMEM tile
// (fp32), and CUDA cores fold it into a register accumulator with the group's
// scale in float32. The affine form w = scale * q + bias (the MLX affine 4-bit
// checkpoints of TensorFold PR #859) runs the same MMAs on the exact codes q,
// and each tile ends with one more group whose operands TMA loads as they
// are: the weight's bias operand (each bias at three K columns) against the
// x group sums X_g = sum_{k in g} x[m][k] split into three bf16 parts
// (w4a16_xsum). Its accumulator is sum_g bias * X_g (exact products, float32
// sums) and the epilogue adds it with scale 1. Rounding a dequantised (q - z) * scale to bf16 before the
// MMA, as the TensorFold PR #859 prompt GEMM does ("each weight rounded once to
// bf16"), would cost up to 2^-9 per weight; this split keeps every weight
// exact. The feed-forward gate is fused as in the GRIMOIRE v1.8 release notes
// ("INT4 prompt processing"): each 128 weight rows of a tile are 64 gate rows
// and the 64 matching up rows (16-row tiles alternate), so h = SiLU(g) * u is
// formed from two float32 accumulators of the same thread before a single
// bf16 rounding.
//
// A tile is 256 weight rows by 256 rows of x, computed by a pair of CTAs on
// two SMs with the pair form of the MMA (cta_group::2, M = 256, N = 256,
// K = 16): each CTA dequantises its own 128 weight rows (the A operand) and
// stages its own 128 x rows (its half of the B operand). Per multiply-add
// this halves the shared-memory operand traffic of an SM and the x bytes it
// pulls from L2 against a one-SM tile of 256 x rows by 128 weight rows, with
// the same dequantisation work per SM. With the weights on the M side, a TMEM
// lane is one weight row, so an epilogue thread folds each group with a single
// scale held in a register.
//
// One persistent CTA pair per two SMs, 512 threads per CTA, warp-specialised:
//   warp 0       TMA producer: the CTA's x rows [128 x 64] (128-byte swizzle), the
//                packed codes of its 128 weight rows x 64 k, and per four groups
//                their scale (+ zero) block; affine: then the bias operand and
//                x group sums of the closing group
//   warp 1       TMEM allocation (both CTAs); in the even CTA the single thread
//                issuing D[b] (+)= W . X^T for the pair, b = group parity
//   warps 4-7    dequantisers: codes -> bf16 (q - z) written straight into the
//                128-byte-swizzled K-major W tile (warps 4-11 for tiles of
//                64 or 128 x rows)
//   warps 8-15   epilogue: per group, TMEM -> registers, acc += scale * D[b];
//                per tile, the bf16 store (or SiLU(gate) * up) (warps 12-15
//                for tiles of 64 or 128 x rows)
// The odd CTA signals the even CTA's barriers with remote arrivals (W half
// written, TMEM buffer drained); the MMA thread's commits arrive on the
// barriers of both CTAs. Every wait is bounded; a wait that gives up sets the
// device error word and both CTAs' abort flags, every role leaves its loop,
// drains what it started, and the pair meets at a cluster barrier before the
// TMEM is freed.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "w4a16_internal.h"

namespace w4a16 {
namespace {

// Output stores with an L2 evict-first hint: the output (143-285 MB at 4,096
// rows) streams through L2 once, and without the hint it displaces the x tiles
// and weight tiles that the other pairs are still reading.
#ifndef W4A16_PROMPT_Y_EVICT_FIRST
#define W4A16_PROMPT_Y_EVICT_FIRST 1
#endif
__device__ __forceinline__ uint64_t y_store_policy() {
  uint64_t pol = 0;
  if (W4A16_PROMPT_Y_EVICT_FIRST) asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void st_y(uint16_t *a, uint16_t v, uint64_t pol) {
  if (W4A16_PROMPT_Y_EVICT_FIRST)
    asm volatile("st.global.L2::cache_hint.b16 [%0], %1, %2;" ::"l"(a), "h"(v), "l"(pol) : "memory");
  else
    *a = v;
}

constexpr int BW = 256, BK = 64;  // pair tile: weight rows, k per stage
constexpr int HW = BW / 2;        // weight rows of one CTA
constexpr int NT16 = HW / 16;     // 16-row weight tiles of one CTA
#ifndef W4A16_PROMPT_SL
#define W4A16_PROMPT_SL 5
#endif
// x + codes ring and dequantised W ring, in step: stage s uses slot s % SL of
// both, and one MMA commit per stage (empty_L) releases both
constexpr int SL = W4A16_PROMPT_SL;
constexpr int SW = SL;
constexpr int SS = 2;                // scale-block ring (4 groups each)
constexpr int kThreads = 512;

constexpr int W_BYTES = HW * BK * 2;  // 16384
constexpr int Q_BYTES = HW * BK / 2;  // 4096
constexpr int RS_BYTES = NT16 * kScaleBlockBytes;  // 1024
constexpr int RZ_BYTES = NT16 * kZeroBlockBytes;   // 256
// barriers: full_L, empty_L [SL]; full_W, (unused) [SW]; full_S, empty_S [SS];
// tfull, tempty [up to 4 TMEM buffers]; mma_done [1]
constexpr int kMaxTBuf = 4;
constexpr int NBARS = 2 * SL + 2 * SW + 2 * SS + 2 * kMaxTBuf + 1;

// Everything that depends on the pair's x rows per tile, BX = 256 for long
// prompts, 128 or 64 for a few dozen rows: a short M then issues MMAs of
// N = BX instead of computing 256 columns of which most are padding; and on
// the weight form QF (a scale-block slot holds the scales, and the zeros of
// the zero-point form).
//
// Warp roles by tile width: at 256 x rows, 4 dequantising warps and 8
// epilogue warps (two per TMEM lane quarter, each on half the columns) and
// two TMEM buffers; at 64 or 128 x rows a 64-wide K stage carries a quarter
// or half of the MMAs and the dequantisers set the pace, so 8 of them, 4
// epilogue warps on all the columns of their lanes, and four TMEM buffers.
template <int BXT, int QF>
struct XGeo {
  static constexpr int BX = BXT, HX = BX / 2;  // x rows of the pair, of one CTA
  static constexpr int DQW = BX == 256 ? 4 : 8;  // dequantising warps: 4 .. 4 + DQW - 1
  static constexpr int EPW = 12 - DQW;           // epilogue warps: the rest of the 16
  static constexpr int EC = BX * 4 / EPW;        // D columns per epilogue thread
  static constexpr int NB = BX == 256 ? 2 : 4;   // TMEM accumulators (groups in flight)
  static constexpr int X_BYTES = HX * BK * 2;
  static constexpr int RZS = RZ_BYTES;  // zero block slot
  static constexpr int OFF_X = 0;
  static constexpr int OFF_W = OFF_X + SL * X_BYTES;
  static constexpr int OFF_Q = OFF_W + SW * W_BYTES;
  static constexpr int OFF_RS = OFF_Q + SL * Q_BYTES;
  static constexpr int OFF_RZ = OFF_RS + SS * RS_BYTES;
  static constexpr int OFF_BAR = OFF_RZ + SS * RZS;
  static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
  static constexpr int SMEM_USED = OFF_MISC + 16;
  static constexpr int SMEM_ALLOC = SMEM_USED + 1024;  // slack for 1024-byte alignment
  static constexpr uint32_t kIdesc = idesc_bf16_f32(BW, BX);
  static constexpr uint32_t kTmemCols = NB * BX;  // NB buffers of BX fp32 columns (a power of two)
  static_assert(NB <= kMaxTBuf && kTmemCols <= 512 && EC % 32 == 0, "TMEM budget");
  static_assert(BX == 64 || BX == 128 || BX == 256, "pair x rows");
  static_assert(OFF_W % 1024 == 0 && OFF_Q % 1024 == 0, "swizzled tiles need 1024-byte alignment");
  static_assert(OFF_RZ % 128 == 0, "TMA destinations");
  static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
};

struct PromptParams {
  uint16_t *y;
  int M, N, K;     // N: output columns (N_each for gate/up)
  int ld;          // y row stride (elements)
  int mtiles, ntiles;  // tiles of BX x rows, of 256 weight rows
  int nk;          // K / 64
  int ng;          // K / group
  int spg;         // 64-wide stages per group (1 or 2)
  int nkb;         // affine: 64-wide stages of the closing bias group (0 otherwise)
  int kc;          // pairs per cluster: 1 = persistent pairs; > 1 = split K, one tile per cluster
  int gblk;        // blocks of four groups (K split at block boundaries)
  int *err;
  UnpackConsts uc;
};

struct Bars {
  uint32_t base;
  __device__ uint32_t full_L(int i) const { return base + 8 * i; }
  __device__ uint32_t empty_L(int i) const { return base + 8 * (SL + i); }
  __device__ uint32_t full_W(int i) const { return base + 8 * (2 * SL + i); }
  __device__ uint32_t full_S(int i) const { return base + 8 * (2 * SL + 2 * SW + i); }
  __device__ uint32_t empty_S(int i) const { return base + 8 * (2 * SL + 2 * SW + SS + i); }
  __device__ uint32_t tfull(int i) const { return base + 8 * (2 * SL + 2 * SW + 2 * SS + i); }
  __device__ uint32_t tempty(int i) const { return base + 8 * (2 * SL + 2 * SW + 2 * SS + kMaxTBuf + i); }
  __device__ uint32_t mma_done() const { return base + 8 * (2 * SL + 2 * SW + 2 * SS + 2 * kMaxTBuf); }
};

// this CTA's abort flag and the peer's (remote store), then the error word
__device__ __forceinline__ void give_up(volatile int *abort_flag, uint32_t peer_abort, int *err) {
  *abort_flag = 1;
  st_cluster_u32(peer_abort, 1u);
  atomicExch(err, kErrTimeout);
}

// arrive on the even CTA's copy of a barrier: locally there, remotely from the
// odd CTA (pbase: the even CTA's rank in the cluster)
__device__ __forceinline__ void arrive_even(uint32_t bar, uint32_t rank, uint32_t pbase) {
  if (rank == 0)
    mbar_arrive(bar);
  else
    mbar_arrive_remote(mapa_shared(bar, pbase));
}

__device__ __forceinline__ uint16_t bf16_bits(float v) {
  __nv_bfloat16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<uint16_t *>(&b);
}

// tm_z: the zero blocks (zero-point form) or the bias operand (affine form);
// tm_xs: the x group sums, in bf16 parts (affine form)
// SPLIT: clusters of p.kc pairs that split one tile's K (a separate
// instantiation, so that the persistent form keeps its loop bounds and pair
// constants out of the registers of the single MMA- and TMA-issuing threads)
template <int QF, bool GATEUP, int BXT, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    prompt_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_z,
                     const __grid_constant__ CUtensorMap tm_xs, PromptParams p) {
  using G = XGeo<BXT, QF>;
  constexpr bool SYM = QF == kFormSym, AFF = QF == kFormAffine, ZP = QF == kFormZero;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  Bars bars{sbase + G::OFF_BAR};
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + G::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + G::OFF_MISC + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // A cluster holds p.kc pairs (ranks 2j, 2j+1). With kc = 1 the pairs are
  // persistent and walk the tiles; with kc > 1 a cluster owns one tile and
  // pair j takes part j of its K range (whole blocks of four groups).
  const uint32_t crank = cluster_ctarank();
  const uint32_t rank = crank & 1u;                   // 0: even CTA of the pair (issues the MMAs), 1: odd
  const uint32_t pbase = SPLIT ? crank & ~1u : 0u;    // the even CTA's rank in the cluster
  const int kpart = SPLIT ? (int)(crank >> 1) : 0;
  const uint16_t pair_mask = SPLIT ? (uint16_t)(3u << pbase) : (uint16_t)3u;
  const uint32_t peer_abort = mapa_shared(smem_u32(smem + G::OFF_MISC + 4), crank ^ 1u);
  const int pair = (int)cluster_id_x(), npairs = (int)nclusters_x();
  const int ntot = p.mtiles * p.ntiles;
  const int g0 = SPLIT ? 4 * (int)((long long)p.gblk * kpart / p.kc) : 0;
  const int g1 = SPLIT ? min(4 * (int)((long long)p.gblk * (kpart + 1) / p.kc), p.ng) : p.ng;  // groups [g0, g1)
  const int kb0 = SPLIT ? g0 * p.spg : 0, kb1 = SPLIT ? g1 * p.spg : p.nk;                       // and stages
  const bool bias_group = AFF && (!SPLIT || kpart == 0);  // affine: the closing bias group, once per tile

  if (tid == 0) {
    for (int i = 0; i < SL; ++i) {
      mbar_init(bars.full_L(i), 1);
      mbar_init(bars.empty_L(i), 1);  // the MMA commit (multicast to both CTAs)
    }
    for (int i = 0; i < SW; ++i) mbar_init(bars.full_W(i), 2 * G::DQW);  // even CTA: local + remote dequant warps
    for (int i = 0; i < SS; ++i) {
      mbar_init(bars.full_S(i), 1);
      mbar_init(bars.empty_S(i), ZP ? G::EPW + G::DQW : G::EPW);  // epilogue warps (+ dequantisers reading zeros)
    }
    for (int i = 0; i < G::NB; ++i) {
      mbar_init(bars.tfull(i), 1);
      mbar_init(bars.tempty(i), 2 * G::EPW);  // even CTA: local + remote epilogue warps
    }
    mbar_init(bars.mma_done(), 1);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc2(smem_u32(tmem_slot), G::kTmemCols);
    tmem_relinquish2();
  }
  // barriers of both CTAs initialised before any remote arrival or commit
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // Register split (launched with 128 per thread = 65536): warpgroup 0 gives
  // back to 40, the dequantising warpgroups to 96, the epilogue warpgroups
  // take 184: 128*40 + 128*96 + 256*184 = 64512 (4 dequantising warps) or
  // 128*40 + 256*96 + 128*184 = 53248 (8) <= 65536.
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 40;");
    if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      // x is re-read by every weight tile: keep it in L2; each codes tile is
      // read by the x tiles in flight at once, then not again
      uint64_t pol_keep, pol_stream;
      asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_keep));
      asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol_stream));
      tma_prefetch_desc(&tm_x);
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_s);
      if (!SYM) tma_prefetch_desc(&tm_z);
      if (AFF) tma_prefetch_desc(&tm_xs);
      uint32_t ls = 0, sc = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < ntot; tile += npairs) {
        const int mt = tile % p.mtiles, nt = tile / p.mtiles;
        const int qt = nt * (BW / 16) + (int)rank * NT16;  // first 16-row tile of this CTA's weights
        const int kbe = bias_group ? kb1 + p.nkb : kb1;  // this pair's stages of a tile
        for (int kb = kb0; kb < kbe; ++kb) {
          if (AFF && kb >= kb1) {
            // affine closing group: x group sums into the x slot, the bias
            // operand straight into the W slot
            const int slot = ls % SL;
            if (!mbar_wait(bars.empty_L(slot), ((ls / SL) & 1) ^ 1, abort_flag)) { ok = false; break; }
            mbar_arrive_expect_tx(bars.full_L(slot), G::X_BYTES + W_BYTES);
            tma_load_2d_hint(sbase + G::OFF_X + slot * G::X_BYTES, &tm_xs, (kb - kb1) * BK,
                             mt * G::BX + (int)rank * G::HX, bars.full_L(slot), pol_keep);
            tma_load_2d_hint(sbase + G::OFF_W + slot * W_BYTES, &tm_z, (kb - kb1) * BK, qt * 16, bars.full_L(slot),
                             pol_stream);
            ++ls;
            continue;
          }
          if (kb % (4 * p.spg) == 0) {
            const int slot = sc % SS;
            if (!mbar_wait(bars.empty_S(slot), ((sc / SS) & 1) ^ 1, abort_flag)) { ok = false; break; }
            mbar_arrive_expect_tx(bars.full_S(slot), RS_BYTES + (ZP ? G::RZS : 0));
            const int blk = kb / (4 * p.spg);
            tma_load_2d(sbase + G::OFF_RS + slot * RS_BYTES, &tm_s, blk * 32, qt, bars.full_S(slot));
            if (ZP) tma_load_2d(sbase + G::OFF_RZ + slot * G::RZS, &tm_z, blk * 8, qt, bars.full_S(slot));
            ++sc;
          }
          const int slot = ls % SL;
          if (!mbar_wait(bars.empty_L(slot), ((ls / SL) & 1) ^ 1, abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(bars.full_L(slot), G::X_BYTES + Q_BYTES);
          tma_load_2d_hint(sbase + G::OFF_X + slot * G::X_BYTES, &tm_x, kb * BK, mt * G::BX + (int)rank * G::HX,
                           bars.full_L(slot), pol_keep);
          tma_load_2d_hint(sbase + G::OFF_Q + slot * Q_BYTES, &tm_q, kb * 128, qt, bars.full_L(slot), pol_stream);
          ++ls;
        }
      }
      if (!ok) {
        give_up(abort_flag, peer_abort, p.err);
        // let every copy already issued land before the CTA can exit
        for (uint32_t i = 0; i < SL && i < ls; ++i) {
          const uint32_t u = ls - 1 - i;
          mbar_wait_drain(bars.full_L(u % SL), (u / SL) & 1);
        }
        for (uint32_t i = 0; i < SS && i < sc; ++i) {
          const uint32_t u = sc - 1 - i;
          mbar_wait_drain(bars.full_S(u % SS), (u / SS) & 1);
        }
      }
    }
    } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer (even CTA)
    if (lane == 0 && rank == 0) {
      uint32_t ls = 0, ws = 0, gc = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < ntot; tile += npairs) {
        const int ge = bias_group ? g1 + 1 : g1;  // this pair's groups of a tile (+ the bias group)
        for (int gi = g0; ok && gi < ge; ++gi) {
          const int nst = (AFF && gi == g1) ? p.nkb : p.spg;  // stages of this group
          const int b = gc % G::NB;
          if (!mbar_wait(bars.tempty(b), ((gc / G::NB) & 1) ^ 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + (uint32_t)(b * G::BX);
          // One wait per group, on the W barrier of the group's last stage.
          // It implies every stage of the group is ready in both CTAs: each
          // dequantising warp waits on its own CTA's full_L before it works on
          // a stage, and arrives on the group's stages in order. (Every barrier
          // operation costs this single issuing thread a few hundred cycles.)
          {
            const uint32_t wl = ws + (uint32_t)nst - 1;
            if (!mbar_wait(bars.full_W(wl % SW), (wl / SW) & 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
          }
          for (int ks = 0; ks < nst; ++ks) {
            const int sl = ls % SL, sw = ws % SW;
            const uint64_t wdesc = sw128_desc(sbase + G::OFF_W + sw * W_BYTES);
            const uint64_t xdesc = sw128_desc(sbase + G::OFF_X + sl * G::X_BYTES);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              // +32 bytes along K inside the 128-byte swizzled row = +2 in the address field
              tc_mma2_f16(d_tmem, wdesc + 2 * kk, xdesc + 2 * kk, G::kIdesc, (ks | kk) != 0);
            }
            tc_commit2_mc(bars.empty_L(sl), pair_mask);  // frees x, codes and W of the stage
            ++ls;
            ++ws;
          }
          if (!ok) break;
          tc_commit2_mc(bars.tfull(b), pair_mask);
          ++gc;
        }
      }
      if (!ok) give_up(abort_flag, peer_abort, p.err);
      // every MMA issued by this thread completes before the pair's TMEM can be freed
      tc_commit2(bars.mma_done());
      mbar_wait_drain(bars.mma_done(), 0);
    }
    }
  } else if (warp < 4 + G::DQW) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 96;");
    // ------------------------------------------------------------------ dequantisers
    const int dw = warp - 4;
    const int g = lane >> 2, t = lane & 3;
    uint32_t ls = 0, ws = 0, sc = 0;
    int cur = 0;
    bool ok = true;
    for (int tile = pair; ok && tile < ntot; tile += npairs) {
      const int kbe = bias_group ? kb1 + p.nkb : kb1;
      for (int kb = kb0; kb < kbe; ++kb) {
        if (AFF && kb >= kb1) {
          // affine closing group: TMA filled the W slot; pass it on
          const int sl = ls % SL, sw = ws % SW;
          if (!mbar_wait(bars.full_L(sl), (ls / SL) & 1, abort_flag)) { ok = false; break; }
          __syncwarp();
          if (lane == 0) arrive_even(bars.full_W(sw), rank, pbase);
          ++ls;
          ++ws;
          continue;
        }
        const int gi = kb / p.spg;
        if (ZP && kb % (4 * p.spg) == 0) {
          cur = sc % SS;
          if (!mbar_wait(bars.full_S(cur), (sc / SS) & 1, abort_flag)) { ok = false; break; }
          ++sc;
        }
        const int sl = ls % SL, sw = ws % SW;
        // full_L of the stage also means its W slot is free: the producer
        // issued the stage's loads only after the MMA commit that released
        // the slot (one ring for codes and W), so no empty_W wait is needed
        if (!mbar_wait(bars.full_L(sl), (ls / SL) & 1, abort_flag)) { ok = false; break; }
        const uint32_t qs = sbase + G::OFF_Q + sl * Q_BYTES;
        const uint32_t wt = sbase + G::OFF_W + sw * W_BYTES;
#pragma unroll
        for (int r = 0; r < NT16 / G::DQW; ++r) {
          const int i = dw + G::DQW * r;  // 16-row tile within the CTA's 128 rows
          uint32_t zg, zg8;
          if (!ZP) {
            zg = zg8 = zero_pair(SYM ? 8 : 0);  // affine: the code q itself
          } else {
            const uint32_t zb = lds8(sbase + G::OFF_RZ + cur * G::RZS + (i * 8 + g) * 4 + (gi & 3));
            zg = zero_pair(zb & 0xF);
            zg8 = zero_pair(zb >> 4);
          }
          const uint4 q = lds128(qs + (i * 32 + lane) * 16);
          uint32_t u[4][4];
          unpack_word(q.x, zg, zg8, p.uc, u[0]);
          unpack_word(q.y, zg, zg8, p.uc, u[1]);
          unpack_word(q.z, zg, zg8, p.uc, u[2]);
          unpack_word(q.w, zg, zg8, p.uc, u[3]);
          // row 16i+g holds k = 16t + 4s + {0,1} in u[s][0] and {2,3} in u[s][2];
          // row 16i+g+8 likewise in u[s][1], u[s][3]
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int n = 16 * i + g + 8 * h;
            const uint32_t row = wt + (n >> 3) * 1024 + (n & 7) * 128;
            const uint4 lo = make_uint4(u[0][h], u[0][2 + h], u[1][h], u[1][2 + h]);
            const uint4 hi = make_uint4(u[2][h], u[2][2 + h], u[3][h], u[3][2 + h]);
            sts128(row + (((2 * t) ^ (n & 7)) << 4), lo);
            sts128(row + (((2 * t + 1) ^ (n & 7)) << 4), hi);
          }
        }
        // each lane makes its stores visible to the tensor cores, then one lane
        // per warp signals the MMA thread of the pair (the codes stage is
        // released by the MMA commit, which follows this arrival)
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          arrive_even(bars.full_W(sw), rank, pbase);
          if (ZP && ((kb + 1) % (4 * p.spg) == 0 || kb + 1 == kb1)) mbar_arrive(bars.empty_S(cur));
        }
        ++ls;
        ++ws;
      }
    }
    if (!ok) give_up(abort_flag, peer_abort, p.err);
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 184;");
    // ------------------------------------------------------------------ epilogue
    constexpr int EC = G::EC;
    const int q = warp & 3;                    // TMEM lanes 32q .. 32q+31: this CTA's weight rows
    const uint64_t ypol = y_store_policy();
    const int ch2 = (warp - 4 - G::DQW) >> 2;  // D columns EC*ch2 .. +EC-1 (x rows mt*BX + EC*ch2 ..)
    const int wr = 32 * q + lane;     // weight row within the CTA's 128
    // this row's scale in a scale block: tile wr/16, g = wr%8, half (wr/8)%2
    const uint32_t soff = (uint32_t)((wr >> 4) * kScaleBlockBytes + (wr & 7) * 16 + ((wr >> 3) & 1) * 2);
    float acc[EC];
    uint32_t gc = 0, sc = 0;
    int cur = 0;
    bool ok = true;
    for (int tile = pair; ok && tile < ntot; tile += npairs) {
      const int mt = tile % p.mtiles, nt = tile / p.mtiles;
#pragma unroll
      for (int c = 0; c < EC; ++c) acc[c] = 0.f;
      for (int gi = g0; gi < (bias_group ? g1 + 1 : g1); ++gi) {
        const bool real = !AFF || gi < g1;  // not the affine closing group (scale 1)
        if (real && (gi & 3) == 0) {
          cur = sc % SS;
          if (!mbar_wait(bars.full_S(cur), (sc / SS) & 1, abort_flag)) { ok = false; break; }
          ++sc;
        }
        const float s =
            real ? __uint_as_float(lds16(sbase + G::OFF_RS + cur * RS_BYTES + soff + (gi & 3) * 4) << 16) : 1.0f;
        const int b = gc % G::NB;
        if (!mbar_wait(bars.tfull(b), (gc / G::NB) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const float2 s2 = make_float2(s, s);
#pragma unroll
        for (int ch = 0; ch < EC / 32; ++ch) {
          float d[32];
          tmem_ld32(tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * G::BX + ch2 * EC + ch * 32), d);
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            float2 a = make_float2(acc[ch * 32 + c], acc[ch * 32 + c + 1]);
            a = __ffma2_rn(s2, make_float2(d[c], d[c + 1]), a);
            acc[ch * 32 + c] = a.x;
            acc[ch * 32 + c + 1] = a.y;
          }

        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          arrive_even(bars.tempty(b), rank, pbase);
          if (real && ((gi & 3) == 3 || gi == g1 - 1)) mbar_arrive(bars.empty_S(cur));
        }
        ++gc;
      }
      if (!ok) break;
      if (SPLIT) {
        // split K: the partial sums go to the (now idle) ring, [column][row]
        // float32, for the cluster's first pair to add up
        float *part = reinterpret_cast<float *>(smem + G::OFF_X);
#pragma unroll
        for (int c = 0; c < EC; ++c) part[(ch2 * EC + c) * HW + wr] = acc[c];
        continue;
      }
      // thread = one weight row, EC x rows m0 + c
      const int m0 = mt * G::BX + ch2 * EC;
      if (GATEUP) {
        // lanes 0-15 hold gate rows, lanes 16-31 the matching up rows (16-row
        // tiles alternate); lanes 0-15 form h for x rows c < EC/2, lanes 16-31
        // for c >= EC/2, each taking the other operand from its partner lane
        constexpr int H2 = EC / 2;
        const bool gate = lane < 16;
        const int n = 16 * (nt * (BW / 32) + (int)rank * (NT16 / 2) + q) + (lane & 15);
#pragma unroll
        for (int c = 0; c < H2; ++c) {
          const float mine = gate ? acc[c] : acc[c + H2];
          const float other = __shfl_xor_sync(0xffffffffu, gate ? acc[c + H2] : acc[c], 16);
          const float gv = gate ? mine : other, uv = gate ? other : mine;
          const int m = m0 + c + (gate ? 0 : H2);
          if (n < p.N && m < p.M) st_y(p.y + (size_t)m * p.ld + n, bf16_bits(silu_f32(gv) * uv), ypol);
        }
      } else {
        const int n = nt * BW + (int)rank * HW + wr;
        if (n < p.N) {
#pragma unroll
          for (int c = 0; c < EC; ++c)
            if (m0 + c < p.M) st_y(p.y + (size_t)(m0 + c) * p.ld + n, bf16_bits(acc[c]), ypol);
        }
      }
    }
    if (!ok) give_up(abort_flag, peer_abort, p.err);
  }

  // both CTAs done with every barrier, smem operand and TMEM column of the pair
  tc_fence_before();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc2(tmem_base, G::kTmemCols);
  }
  if (SPLIT) {
    // split K: the first pair adds the other pairs' partial sums (same parity
    // CTA, ranks 2j + rank), in pair order, and stores the tile
    if (kpart == 0 && !*abort_flag) {
      const uint64_t ypol = y_store_policy();
      const float *part = reinterpret_cast<const float *>(smem + G::OFF_X);
      const uint32_t part_s = smem_u32(smem + G::OFF_X);
      const int mt = pair % p.mtiles, nt = pair / p.mtiles;
      auto sum_at = [&](int idx) {
        float v = part[idx];
        for (int j = 1; j < p.kc; ++j) v += ld_cluster_f32(mapa_shared(part_s + 4u * (uint32_t)idx, crank + 2u * j));
        return v;
      };
      if (GATEUP) {
        // gate row 32q + l and its up row 32q + 16 + l (16-row tiles alternate)
        for (int e = tid; e < G::BX * HW / 2; e += kThreads) {
          const int col = e / (HW / 2), rr = e % (HW / 2), q = rr >> 4, l = rr & 15;
          const float gv = sum_at(col * HW + 32 * q + l), uv = sum_at(col * HW + 32 * q + 16 + l);
          const int n = 16 * (nt * (BW / 32) + (int)rank * (NT16 / 2) + q) + l;
          const int m = mt * G::BX + col;
          if (n < p.N && m < p.M) st_y(p.y + (size_t)m * p.ld + n, bf16_bits(silu_f32(gv) * uv), ypol);
        }
      } else {
        for (int e = tid; e < G::BX * HW; e += kThreads) {
          const int col = e / HW, row = e % HW;
          const int n = nt * BW + (int)rank * HW + row, m = mt * G::BX + col;
          if (n < p.N && m < p.M) st_y(p.y + (size_t)m * p.ld + n, bf16_bits(sum_at(e)), ypol);
        }
      }
    }
    // the other pairs keep their partials until the first pair has read them
    cluster_sync_all();
  }
}

// ---------------------------------------------------------------------------
// host side: tensor maps and launch
// ---------------------------------------------------------------------------
// Launch as clusters of two CTAs: one pair per tile, as many pairs as fit at
// once (found once per instantiation and device), each walking the tiles with
// a stride; or, split K (p.kc > 1), one cluster of p.kc pairs per tile.
template <int QF, bool GATEUP, int BXT, bool SPLIT>
cudaError_t launch_variant(const CUtensorMap &tx, const CUtensorMap &tq, const CUtensorMap &ts,
                           const CUtensorMap &tz, const CUtensorMap &txs, const PromptParams &p, int ntot,
                           int device, cudaStream_t s) {
  using G = XGeo<BXT, QF>;
  auto kern = prompt_tc_kernel<QF, GATEUP, BXT, SPLIT>;
  cudaLaunchConfig_t lc = {};
  lc.blockDim = dim3(kThreads, 1, 1);
  lc.dynamicSmemBytes = G::SMEM_ALLOC;
  lc.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  static PerDevice max_pairs;  // clusters of this kernel that fit at once, per device
  int np = max_pairs.v[device].load(std::memory_order_relaxed);
  if (np == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    lc.gridDim = dim3(2, 1, 1);
    e = cudaOccupancyMaxActiveClusters(&np, kern, &lc);
    if (e != cudaSuccess) return e;
    if (np < 1) return cudaErrorInvalidConfiguration;
    max_pairs.v[device].store(np, std::memory_order_relaxed);
  }
  if (p.kc > 1) {
    attr[0].val.clusterDim.x = 2 * p.kc;
    lc.gridDim = dim3(2 * p.kc * ntot, 1, 1);
  } else {
    const int pairs = ntot < np ? ntot : np;
    lc.gridDim = dim3(2 * pairs, 1, 1);
  }
  return cudaLaunchKernelEx(&lc, kern, tx, tq, ts, tz, txs, p);
}

template <int QF, bool GATEUP, int BXT>
cudaError_t launch_form(const CUtensorMap &tx, const CUtensorMap &tq, const CUtensorMap &ts, const CUtensorMap &tz,
                        const CUtensorMap &txs, const PromptParams &p, int ntot, const GemmCall &c) {
  if (p.kc > 1) return launch_variant<QF, GATEUP, BXT, true>(tx, tq, ts, tz, txs, p, ntot, c.device, c.stream);
  return launch_variant<QF, GATEUP, BXT, false>(tx, tq, ts, tz, txs, p, ntot, c.device, c.stream);
}

template <int BXT>
cudaError_t launch_bx(const GemmCall &c, int sm_count) {
  using G = XGeo<BXT, kFormSym>;
  const int rows = packed_rows(c);
  const Layout L = make_layout(rows, c.K, c.group, c.sym);
  CUtensorMap tx, tq, ts, tz, txs;
  bool ok = encode_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c.x, (uint64_t)c.K, (uint64_t)c.M,
                      (uint64_t)c.K * 2, BK, G::HX, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && encode_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT32, c.packed + L.codes_off, (uint64_t)L.chunks * 128,
                       (uint64_t)L.tiles, (uint64_t)L.chunks * kChunkBytes, 128, NT16, CU_TENSOR_MAP_SWIZZLE_NONE);
  ok = ok && encode_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT32, c.packed + L.scales_off, (uint64_t)L.gblocks * 32,
                       (uint64_t)L.tiles, (uint64_t)L.gblocks * kScaleBlockBytes, 32, NT16,
                       CU_TENSOR_MAP_SWIZZLE_NONE);
  tz = txs = ts;  // unused unless set below
  if (c.sym == kFormZero) {
    ok = ok && encode_2d(&tz, CU_TENSOR_MAP_DATA_TYPE_UINT32, c.packed + L.zeros_off, (uint64_t)L.gblocks * 8,
                         (uint64_t)L.tiles, (uint64_t)L.gblocks * kZeroBlockBytes, 8, NT16,
                         CU_TENSOR_MAP_SWIZZLE_NONE);
  } else if (c.sym == kFormAffine) {
    if (!c.xsum) return cudaErrorInvalidValue;
    // the bias operand [rows][kb3] and the x group sums [M][kb3], both bf16
    // and K-major like x, in 64-wide boxes with the 128-byte swizzle
    ok = ok && encode_2d(&tz, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c.packed + L.bops_off, (uint64_t)L.kb3,
                         (uint64_t)L.tiles * 16, (uint64_t)L.kb3 * 2, BK, HW, CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && encode_2d(&txs, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c.xsum, (uint64_t)L.kb3, (uint64_t)c.M,
                         (uint64_t)L.kb3 * 2, BK, G::HX, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (!ok) return cudaErrorInvalidValue;
  PromptParams p;
  p.y = c.y;
  p.M = c.M;
  p.N = c.N;
  p.K = c.K;
  p.ld = c.N;
  p.mtiles = (c.M + G::BX - 1) / G::BX;
  p.ntiles = (rows + BW - 1) / BW;
  p.nk = c.K / BK;
  p.ng = c.K / c.group;
  p.spg = c.group / BK;
  p.nkb = c.sym == kFormAffine ? L.kb3 / BK : 0;
  p.gblk = (p.ng + 3) / 4;
  // Split K when the tiles leave most pairs idle (few weight tiles, short M):
  // up to 4 pairs per tile, each with at least two blocks of four groups.
  p.kc = 1;
  {
    const int ntiles_all = p.mtiles * p.ntiles, pairs = sm_count / 2;
    if (ntiles_all * 2 <= pairs) {
      p.kc = pairs / ntiles_all < 4 ? pairs / ntiles_all : 4;
      while (p.kc > 1 && p.gblk < 2 * p.kc) --p.kc;
    }
  }
  p.err = c.err;
  p.uc = host_unpack_consts();
  const int ntot = p.mtiles * p.ntiles;
  if (c.sym == kFormSym)
    return c.gateup ? launch_form<kFormSym, true, BXT>(tx, tq, ts, tz, txs, p, ntot, c)
                    : launch_form<kFormSym, false, BXT>(tx, tq, ts, tz, txs, p, ntot, c);
  if (c.sym == kFormAffine)
    return c.gateup ? launch_form<kFormAffine, true, BXT>(tx, tq, ts, tz, txs, p, ntot, c)
                    : launch_form<kFormAffine, false, BXT>(tx, tq, ts, tz, txs, p, ntot, c);
  return c.gateup ? launch_form<kFormZero, true, BXT>(tx, tq, ts, tz, txs, p, ntot, c)
                  : launch_form<kFormZero, false, BXT>(tx, tq, ts, tz, txs, p, ntot, c);
}

}  // namespace

// ---------------------------------------------------------------------------
// tensor maps (shared with the tcgen05 decode kernel)
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

bool encode_2d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  auto fn = get_encode();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}


cudaError_t launch_prompt_tc(const GemmCall &c, int sm_count) {
  // x-row tile: the smallest that holds M (a tile of 256 otherwise)
  if (c.M <= 64) return launch_bx<64>(c, sm_count);
  if (c.M <= 128) return launch_bx<128>(c, sm_count);
  return launch_bx<256>(c, sm_count);
}

}  // namespace w4a16
