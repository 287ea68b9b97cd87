// Decode-regime kernels, M <= 32 rows of x against the whole weight.
//
// Both kernels stream the repacked weight exactly once per call (HBM-bound)
// and are built around the integer-ALU cost of the nibble unpack, which is
// what bounds them on GB300:
//
//  * Every warp owns a ring of shared-memory slots that its lane 0 fills with
//    bulk asynchronous copies (cp.async.bulk, completion counted on one
//    mbarrier per slot). A slot is one 256-wide K unit of the warp's tiles:
//    their packed codes plus the scale (and zero) block. The bytes in flight
//    cost no registers, and the per-slot bookkeeping is spread over 32 to 64
//    packed words per lane.
//
//  * smallm_mma_kernel (M = 1..32): a lane's two rows x 16 k are the A
//    fragment of mma.sync m16n8k16 (bf16 in, f32 accumulate); x rows are the
//    B fragment. Each packed word becomes four bf16x2 registers of exact
//    q - z: three shifts and four LOP3s give 128 + q (bf16 0x4300 is 128 with
//    a mantissa step of 1, the "(0x4300 | c) - 128" rebuild of TensorFold PR
//    #859) and one bf16x2 subtraction of 128 + z per register leaves q - z.
//    One group's products sum in a fresh accumulator, then acc += scale *
//    partial in float32. Affine form (w = scale * q + bias, the MLX affine
//    4-bit checkpoints of TensorFold PR #859): the same unpack with z = 0 gives
//    q exactly, one more MMA per 16 k with an all-ones A sums the group's x
//    (X_g), and acc += scale * partial + bias * X_g. "2-16 rows ... INT4 weights and bf16 activations" is
//    the DPAS verify GEMM of the GRIMOIRE v1.7 release notes ("What changed");
//    their v1.8 notes ("INT4 verify faster") show it occupancy-bound: here each
//    weight tile is read and unpacked once for all rows and the tensor core
//    does the multiply-adds.
//  * gemv_m1_kernel (M = 1): CUDA-core form. Each nibble becomes the float32
//    2^23 + q * 16^p by OR-ing the magic exponent onto it in place (no shift
//    for the low five nibbles), 2^23 + z * 16^p is subtracted exactly, the
//    product with x accumulates in float32 (packed f32x2 FMA), and the 16^-p
//    factor is applied once per group. Lanes meet by warp shuffles (the
//    single-user ESIMD GEMV of the same v1.7 notes).
//
// Split-K: the warps of a CTA take disjoint K slices of the same tiles and sum
// through shared memory; for short N, KC CTAs of a cluster split K further and
// rank 0 sums the others' partials through distributed shared memory, in rank
// order (split-K by clusters on sm_90+, as in TensorFold PR #859, "What this
// changes"). No sum uses atomics, so results are bitwise reproducible.
#include "w4a16_internal.h"

namespace w4a16 {
namespace {

constexpr int kWarps = 4;       // warps per CTA
// ring depth (K units in flight per warp) for two tiles per warp
#ifndef W4A16_DECODE_SLOTS2
#define W4A16_DECODE_SLOTS2 2
#endif
#ifndef W4A16_UNIT_CHUNKS
#define W4A16_UNIT_CHUNKS 4
#endif
constexpr int kUnitChunks = W4A16_UNIT_CHUNKS;  // 64-wide K chunks per ring slot
static_assert(kUnitChunks == 2 || kUnitChunks == 4, "a unit is 128 or 256 k");
#ifndef W4A16_DECODE_UNIT_LOADS
#define W4A16_DECODE_UNIT_LOADS 1
#endif
constexpr bool kDecodeUnitLoads = W4A16_DECODE_UNIT_LOADS != 0;

struct DecodeParams {
  const uint16_t *x;
  const uint8_t *codes;    // [tile][chunk][lane][16 B]
  const uint8_t *scales;   // [tile][gblock][g][4 groups][2 rows] bf16
  const uint8_t *zeros;    // [tile][gblock][g][4 groups] bytes (row g | row g+8 << 4),
                           // or the biases in the scales' layout (affine form)
  uint16_t *y;
  int M, N, K;             // N: output columns (N_each for gate/up)
  int tiles, chunks, groups, gblocks, units;
  int ld;                  // y row stride in elements
  int *err;
  unsigned long long *amax;  // per x row, the running argmax key of y (or null)
  int device;              // host side only: ordinal for the per-device caches
  bool overlap;            // host side only: launch with programmatic stream serialization
  UnpackConsts uc;
};

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// same product, accumulator starting from zero
__device__ __forceinline__ void mma_bf16_16816_zero(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                                    uint32_t b1) {
  const float z = 0.f;
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%10,%10,%10};"
      : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
}

__device__ __forceinline__ uint4 ldg_keep(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  __nv_bfloat16 b = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t *>(&b);
}


// 1-D bulk copy global -> shared, completion counted on `bar`; the weights are
// read once, so they are marked first to leave L2.
__device__ __forceinline__ void bulk_copy(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// same copy without a cache hint: x is read by every CTA, so it stays in L2
__device__ __forceinline__ void bulk_copy_keep(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Slice [u0, u1) of the K units for this warp.
__device__ __forceinline__ void k_slice(int units, int &u0, int &u1) {
  const int nsl = gridDim.y * kWarps;
  const int sidx = blockIdx.y * kWarps + (threadIdx.x >> 5);
  u0 = (int)((long long)units * sidx / nsl);
  u1 = (int)((long long)units * (sidx + 1) / nsl);
}

// ---------------------------------------------------------------------------
// Per-warp ring of K-unit slots filled by bulk copies.
//   slot layout: codes [TPW][4 chunks][32 lanes][16 B], then the scale block
//   of each tile [TPW][128 B], then its zero block [TPW][32 B] (zero-point
//   form) or bias block [TPW][128 B] (affine form).
//   A unit u covers chunks 4u .. 4u+3 (fewer in a ragged last unit) and lies
//   inside scale block u (group 64) or u/2 (group 128).
// ---------------------------------------------------------------------------
template <int TPW, int QF, int SLOTS>
struct Ring {
  static constexpr int kTileCode = kUnitChunks * kChunkBytes;
  static constexpr int kScaleOff = TPW * kTileCode;
  static constexpr int kZeroOff = kScaleOff + TPW * kScaleBlockBytes;  // zero or bias blocks
  static constexpr int kThirdBytes =
      QF == kFormZero ? kZeroBlockBytes : QF == kFormAffine ? kScaleBlockBytes : 0;
  static constexpr int kSlotBytes = kZeroOff + TPW * kThirdBytes;
  static constexpr int kWarpBytes = SLOTS * kSlotBytes;
  // one bulk copy per lane: codes of each tile, then its scale block, then its
  // zero or bias block
  static constexpr int kCopies = TPW * (QF == kFormSym ? 2 : 3);

  uint32_t sbase;  // this warp's slots, shared-window address
  uint32_t bar0;   // SLOTS mbarriers, 8 bytes apart
  // this lane's copy (lanes >= kCopies issue none)
  const uint8_t *src;  // source of the copy for unit 0 / scale block 0
  uint32_t stride;     // source step per unit (codes) or per scale block
  uint32_t dst_off;    // offset inside a slot
  bool is_code;
  uint64_t policy;
  int chunks;     // chunks per tile
  int upb_shift;  // log2 of the units per scale block (1, 2 or 4 units)

  __device__ void setup(const DecodeParams &p, uint8_t *warp_base, uint64_t *warp_bars, int tile0, int cpg) {
    const int lane = threadIdx.x & 31;
    sbase = smem_u32(warp_base);
    bar0 = smem_u32(warp_bars);
    chunks = p.chunks;
    upb_shift = __ffs(4 * cpg / kUnitChunks) - 1;  // a block of four groups spans 4 * cpg chunks
    const int kind = lane / TPW, i = lane % TPW;
    const size_t tile = (size_t)min(tile0 + i, p.tiles - 1);
    is_code = kind == 0;
    if (kind == 0) {
      src = p.codes + tile * p.chunks * kChunkBytes;
      stride = kTileCode;
      dst_off = i * kTileCode;
    } else if (kind == 1) {
      src = p.scales + tile * p.gblocks * kScaleBlockBytes;
      stride = kScaleBlockBytes;
      dst_off = kScaleOff + i * kScaleBlockBytes;
    } else {
      src = p.zeros + tile * p.gblocks * kThirdBytes;
      stride = kThirdBytes;
      dst_off = kZeroOff + i * kThirdBytes;
    }
    policy = evict_first_policy();
    if (lane == 0) {
      for (int s = 0; s < SLOTS; ++s) mbar_init(bar0 + 8 * s, 1);
      fence_mbar_init();
    }
    __syncwarp();
  }

  // The whole warp: copy unit u into slot s. Lane q < kCopies issues copy q
  // and lane 0 posts the expected bytes with the slot's one arrival, so a copy
  // that lands before that arrival cannot complete the phase.
  __device__ void issue(int s, int u) {
    const int lane = threadIdx.x & 31;
    const uint32_t bar = bar0 + 8 * s;
    const int nch = min(kUnitChunks, chunks - kUnitChunks * u);
    if (lane == 0)
      mbar_arrive_expect_tx(bar, TPW * (nch * kChunkBytes + kScaleBlockBytes + kThirdBytes));
    if (lane < kCopies) {
      const uint32_t bytes = is_code ? (uint32_t)(nch * kChunkBytes) : stride;
      const size_t step = is_code ? (size_t)u : (size_t)(u >> upb_shift);
      bulk_copy(sbase + s * kSlotBytes + dst_off, src + step * stride, bytes, bar, policy);
    }
  }

  __device__ uint32_t slot(int s) const { return sbase + s * kSlotBytes; }
};

// Sum the per-warp partials red[w][e] into red[0][e]; with a cluster, rank 0
// then adds every other rank's red[0][e] in rank order. Returns true in the
// CTA that writes the outputs.
template <int E>
__device__ __forceinline__ bool reduce_partials(float (*red)[E]) {
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float s = red[0][e];
    for (int w = 1; w < kWarps; ++w) s += red[w][e];
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

// Partials red[e] of every CTA of a cluster summed into rank 0's, in rank
// order. Returns true in the CTA that writes the outputs.
template <int E>
__device__ __forceinline__ bool cluster_sum(float *red) {
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
      float s = red[e];
      const uint32_t local = smem_u32(&red[e]);
      for (uint32_t r = 1; r < nranks; ++r) {
        uint32_t remote;
        float v;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(r));
        asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
        s += v;
      }
      red[e] = s;
    }
  }
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
  __syncthreads();
  return rank == 0;
}

// Dynamic shared memory of a decode CTA: rings, their barriers, the partials
// and the abort flag.
template <int TPW, int QF, int SLOTS, int E>
struct DecodeSmem {
  using R = Ring<TPW, QF, SLOTS>;
  static constexpr int kRingOff = 0;
  static constexpr int kBarOff = kWarps * R::kWarpBytes;
  static constexpr int kRedOff = kBarOff + kWarps * SLOTS * 8;
  static constexpr int kBestOff = kRedOff + kWarps * E * 4;  // argmax keys, one per x row (<= 32)
  static constexpr int kFlagOff = kBestOff + 32 * 8;
  static constexpr int kBytes = kFlagOff + 16;
};

// Wait for the slot of the it-th unit. The outcome is made warp-uniform (a
// lane that gave up makes the whole warp give up, so no lane is left behind at
// a later __syncwarp); on giving up, raise the CTA abort flag.
template <int SLOTS>
__device__ __forceinline__ bool wait_slot(uint32_t bar0, int it, volatile int *abort_flag, int *err) {
  const int s = it % SLOTS;
  const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait<true>(bar0 + 8 * s, (it / SLOTS) & 1, abort_flag));
  if (!ok && (threadIdx.x & 31) == 0) {
    *abort_flag = 1;
    atomicExch(err, kErrTimeout);
  }
  return ok;
}

// After giving up: let the copies this warp issued land before the CTA exits.
template <int SLOTS>
__device__ __forceinline__ void drain_ring(uint32_t bar0, int first_unwaited, int issued) {
  for (int it = first_unwaited; it < issued; ++it) mbar_wait_drain(bar0 + 8 * (it % SLOTS), (it / SLOTS) & 1);
}

// ---------------------------------------------------------------------------
// small-M tensor-core kernel
// ---------------------------------------------------------------------------
template <int MT, int TPW, int QF, int CPG, int SLOTS, bool GATEUP>
__global__ void __launch_bounds__(kWarps * 32) smallm_mma_kernel(DecodeParams p) {
  constexpr int E = TPW * MT * 4 * 32;
  constexpr int GPU = kUnitChunks / CPG;  // groups per full unit
  constexpr bool AFF = QF == kFormAffine;
  using SM = DecodeSmem<TPW, QF, SLOTS, E>;
  using R = Ring<TPW, QF, SLOTS>;
  extern __shared__ __align__(128) uint8_t smem[];
  float(*red)[E] = reinterpret_cast<float(*)[E]>(smem + SM::kRedOff);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + SM::kFlagOff);

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int tile0 = blockIdx.x * TPW;
  unsigned long long *best = reinterpret_cast<unsigned long long *>(smem + SM::kBestOff);
  if (threadIdx.x == 0) *abort_flag = 0;
  if (threadIdx.x < 32) best[threadIdx.x] = 0;
  __syncthreads();
  int ub, ue;
  k_slice(p.units, ub, ue);
  const int nu = ue - ub;

  R ring;
  ring.setup(p, smem + SM::kRingOff + warp * R::kWarpBytes,
             reinterpret_cast<uint64_t *>(smem + SM::kBarOff) + warp * SLOTS, tile0, CPG);
  int issued = 0;  // warp-uniform
  for (; issued < SLOTS && issued < nu; ++issued) ring.issue(issued, ub + issued);
  // the weights are in flight; x and y belong to the previous kernel until it
  // has finished (programmatic overlap), and the next call may be scheduled
  grid_launch_dependents();
  grid_dependency_wait();

  // B fragment column g + 8 mt reads x row min(g + 8 mt, M - 1): columns past M
  // compute duplicates that are never stored
  const uint4 *xp[MT];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
    xp[mt] = reinterpret_cast<const uint4 *>(p.x + (size_t)min(g + 8 * mt, p.M - 1) * p.K + 16 * t);

  float acc[TPW][MT][4];
#pragma unroll
  for (int i = 0; i < TPW; ++i)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[i][mt][r] = 0.f;

  // One x tile (M <= 8): the unit's x (4 chunks x 2 x 16 bytes per lane) is
  // loaded before the slot wait, at immediate offsets from one address per
  // unit, and the unit's codes are read from the slot at once. More x tiles:
  // x is loaded one 64-wide chunk ahead of its use (xn), so the load latency
  // overlaps the previous chunk's unpack and MMAs.
  constexpr bool kUnitX = MT == 1 && kDecodeUnitLoads;
  uint4 xn[MT][2];
  if (!kUnitX) {
    const int c0 = min(kUnitChunks * ub, p.chunks - 1);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      xn[mt][0] = ldg_keep(xp[mt] + (size_t)c0 * 8);
      xn[mt][1] = ldg_keep(xp[mt] + (size_t)c0 * 8 + 1);
    }
  }
  int it = 0;
  for (; it < nu; ++it) {
    const int u = ub + it;
    const int nch = min(kUnitChunks, p.chunks - kUnitChunks * u);
    const int ngu = nch / CPG;  // groups in this unit
    uint4 xu[kUnitX ? kUnitChunks : 1][2];
    if (kUnitX) {
      const uint4 *xb = xp[0] + (size_t)u * (kUnitChunks * 8);
      if (nch == kUnitChunks) {
#pragma unroll
        for (int cl = 0; cl < (kUnitX ? kUnitChunks : 1); ++cl) {
          xu[cl][0] = ldg_keep(xb + cl * 8);
          xu[cl][1] = ldg_keep(xb + cl * 8 + 1);
        }
      } else {  // a ragged last unit: its chunks only
#pragma unroll
        for (int cl = 0; cl < (kUnitX ? kUnitChunks : 1); ++cl) {
          const int cc = min(cl, nch - 1);
          xu[cl][0] = ldg_keep(xb + cc * 8);
          xu[cl][1] = ldg_keep(xb + cc * 8 + 1);
        }
      }
    }
    if (!wait_slot<SLOTS>(ring.bar0, it, abort_flag, p.err)) break;
    const uint32_t sl = ring.slot(it % SLOTS);
    uint4 wu[kUnitX ? TPW : 1][kUnitX ? kUnitChunks : 1];
    if (kUnitX) {
#pragma unroll
      for (int i = 0; i < (kUnitX ? TPW : 1); ++i)
#pragma unroll
        for (int cl = 0; cl < (kUnitX ? kUnitChunks : 1); ++cl)
          wu[i][cl] = lds128(sl + i * R::kTileCode + (cl * 32 + lane) * 16);
    }
#pragma unroll
    for (int j = 0; j < GPU; ++j) {
      if (j < ngu) {
        const int gg = u * GPU + j;  // global group index
        uint32_t zg[TPW], zg8[TPW];
#pragma unroll
        for (int i = 0; i < TPW; ++i) {
          if (QF != kFormZero) {
            zg[i] = zg8[i] = zero_pair(AFF ? 0 : 8);
          } else {
            const uint32_t zb = lds8(sl + R::kZeroOff + i * kZeroBlockBytes + g * 4 + (gg & 3));
            zg[i] = zero_pair(zb & 0xF);
            zg8[i] = zero_pair(zb >> 4);
          }
        }
        float part[TPW][MT][4];
        float xs[MT][4];  // affine: the group's sum of x per column (all-ones A)
#pragma unroll
        for (int cc = 0; cc < CPG; ++cc) {
          const int cl = j * CPG + cc;  // chunk within the unit
          uint4 xx[MT][2];
          uint4 w[TPW];
          if (kUnitX) {
            xx[0][0] = xu[kUnitX ? cl : 0][0];
            xx[0][1] = xu[kUnitX ? cl : 0][1];
#pragma unroll
            for (int i = 0; i < TPW; ++i) w[i] = wu[kUnitX ? i : 0][kUnitX ? cl : 0];
          } else {
            const int c = kUnitChunks * u + cl;
            const int cn = min(c + 1, p.chunks - 1);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              xx[mt][0] = xn[mt][0];
              xx[mt][1] = xn[mt][1];
              xn[mt][0] = ldg_keep(xp[mt] + (size_t)cn * 8);
              xn[mt][1] = ldg_keep(xp[mt] + (size_t)cn * 8 + 1);
            }
#pragma unroll
            for (int i = 0; i < TPW; ++i)
              w[i] = lds128(sl + i * R::kTileCode + (cl * 32 + lane) * 16);
          }
#pragma unroll
          for (int st = 0; st < 4; ++st) {
            // B fragment: x words 2st (k+0, k+1) and 2st+1 (k+2, k+3) of this lane's 16 k
            uint32_t b0[MT], b1[MT];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              b0[mt] = word_of(xx[mt][st >> 1], 2 * (st & 1));
              b1[mt] = word_of(xx[mt][st >> 1], 2 * (st & 1) + 1);
            }
            if (AFF) {
              const uint32_t ones[4] = {0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u};
#pragma unroll
              for (int mt = 0; mt < MT; ++mt) {
                if (cc == 0 && st == 0)
                  mma_bf16_16816_zero(xs[mt], ones, b0[mt], b1[mt]);
                else
                  mma_bf16_16816(xs[mt], ones, b0[mt], b1[mt]);
              }
            }
#pragma unroll
            for (int i = 0; i < TPW; ++i) {
              uint32_t a[4];
              unpack_word(word_of(w[i], st), zg[i], zg8[i], p.uc, a);
#pragma unroll
              for (int mt = 0; mt < MT; ++mt) {
                if (cc == 0 && st == 0)
                  mma_bf16_16816_zero(part[i][mt], a, b0[mt], b1[mt]);
                else
                  mma_bf16_16816(part[i][mt], a, b0[mt], b1[mt]);
              }
            }
          }
        }
#pragma unroll
        for (int i = 0; i < TPW; ++i) {
          const uint32_t sw = lds32(sl + R::kScaleOff + i * kScaleBlockBytes + g * 16 + (gg & 3) * 4);
          const float sg = bf16lo_to_f32(sw), sg8 = bf16hi_to_f32(sw);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            acc[i][mt][0] = fmaf(sg, part[i][mt][0], acc[i][mt][0]);
            acc[i][mt][1] = fmaf(sg, part[i][mt][1], acc[i][mt][1]);
            acc[i][mt][2] = fmaf(sg8, part[i][mt][2], acc[i][mt][2]);
            acc[i][mt][3] = fmaf(sg8, part[i][mt][3], acc[i][mt][3]);
          }
          if (AFF) {
            const uint32_t bw = lds32(sl + R::kZeroOff + i * kScaleBlockBytes + g * 16 + (gg & 3) * 4);
            const float bg = bf16lo_to_f32(bw), bg8 = bf16hi_to_f32(bw);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              acc[i][mt][0] = fmaf(bg, xs[mt][0], acc[i][mt][0]);
              acc[i][mt][1] = fmaf(bg, xs[mt][1], acc[i][mt][1]);
              acc[i][mt][2] = fmaf(bg8, xs[mt][2], acc[i][mt][2]);
              acc[i][mt][3] = fmaf(bg8, xs[mt][3], acc[i][mt][3]);
            }
          }
        }
      }
    }
    // every lane has consumed the slot: refill it with the unit SLOTS ahead
    __syncwarp();
    if (issued < nu) {
      fence_proxy_async_smem();
      ring.issue(it % SLOTS, ub + issued);
      ++issued;
    }
  }
  if (it < nu && lane == 0) drain_ring<SLOTS>(ring.bar0, it, issued);

#pragma unroll
  for (int i = 0; i < TPW; ++i)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int r = 0; r < 4; ++r) red[warp][((i * MT + mt) * 4 + r) * 32 + lane] = acc[i][mt][r];

  if (!reduce_partials<E>(red)) return;

  // element e = ((i*MT + mt)*4 + r)*32 + lane:
  //   row n = 16*(tile0+i) + g + 8*(r>>1), column m = 8*mt + 2t + (r&1)
  // gate/up: tiles alternate gate, up; the pair (i, i+1) gives 16 outputs
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int ln = e & 31, r = (e >> 5) & 3, im = e >> 7;
    const int mt = im % MT, i = im / MT;
    const int m = 8 * mt + 2 * (ln & 3) + (r & 1);
    const int nl = (ln >> 2) + 8 * (r >> 1);
    if (m >= p.M) continue;
    if (GATEUP) {
      if (i & 1) continue;
      const int n = 16 * ((tile0 + i) >> 1) + nl;
      if (n < p.N) {
        const float gv = red[0][e], uv = red[0][e + MT * 4 * 32];
        p.y[(size_t)m * p.ld + n] = f32_to_bf16_bits(silu_f32(gv) * uv);
      }
    } else {
      const int n = 16 * (tile0 + i) + nl;
      if (n < p.N) {
        const uint16_t v = f32_to_bf16_bits(red[0][e]);
        if (p.y) p.y[(size_t)m * p.ld + n] = v;
        if (p.amax) atomicMax(best + m, argmax_key(v, n));
      }
    }
  }
  if (!GATEUP && p.amax) {
    // one global arrival per x row and CTA: the largest key of this CTA's outputs
    __syncthreads();
    if (threadIdx.x < p.M && best[threadIdx.x] != 0) atomicMax(p.amax + threadIdx.x, best[threadIdx.x]);
  }
}

// ---------------------------------------------------------------------------
// small-M tensor-core kernel with x staged once per CTA
//
// At M >= 2 the x rows of a call (80 KB at M = 8, 160 KB at M = 16, K = 5120)
// no longer stay in L1 beside the weight rings, and per-warp 16-byte x loads
// from L2 stall the warps. Here the four compute warps of a CTA work on
// different tiles of the same K range, so one copy of each 256-wide K unit of
// x serves all of them: a fifth warp fills a ring of slots, each holding one
// K unit of every tile's codes, scale (and zero or bias) blocks and the x rows
// (bulk asynchronous copies, one mbarrier per slot for the bytes, one per slot
// for the four warps' release). x rows sit 528 bytes apart, so the 16-byte B
// fragment loads of a warp touch 32 distinct banks. K is split only across
// the CTAs of a cluster.
// ---------------------------------------------------------------------------
#ifndef W4A16_XS_WARPS
#define W4A16_XS_WARPS 4
#endif
constexpr int kXsWarps = W4A16_XS_WARPS;  // compute warps; warp kXsWarps issues the copies
constexpr int kXsThreads = (kXsWarps + 1) * 32;
#ifndef W4A16_XS_SLOTS
#define W4A16_XS_SLOTS 2
#endif
#ifndef W4A16_XS_TPW
#define W4A16_XS_TPW 2
#endif
constexpr int kXsSlots = W4A16_XS_SLOTS;
constexpr int kXRowStride = kUnitChunks * 128 + 16;

template <int MT, int TPW, int QF>
struct XsSmem {
  static constexpr int kTiles = kXsWarps * TPW;  // 16-row tiles of a CTA
  static constexpr int kTileCode = kUnitChunks * kChunkBytes;
  static constexpr int kThird = QF == kFormZero ? kZeroBlockBytes : QF == kFormAffine ? kScaleBlockBytes : 0;
  static constexpr int kScaleOff = kTiles * kTileCode;
  static constexpr int kThirdOff = kScaleOff + kTiles * kScaleBlockBytes;
  static constexpr int kXOff = kThirdOff + kTiles * kThird;
  static constexpr int kXRows = 8 * MT;
  static constexpr int kSlotBytes = (kXOff + kXRows * kXRowStride + 127) / 128 * 128;
  static constexpr int kCopies = kTiles * (QF == kFormSym ? 2 : 3);  // weight copies per unit (+ x rows)
  static constexpr int E = kTiles * MT * 128;  // partial sums of the CTA
  static constexpr int kRingOff = 0;
  static constexpr int kRedOff = 0;  // the partials reuse the ring once every unit is consumed
  static constexpr int kBarOff = kXsSlots * kSlotBytes;  // full[s], then empty[s]
  static constexpr int kBestOff = kBarOff + 2 * kXsSlots * 8;
  static constexpr int kFlagOff = kBestOff + 16 * 8;
  static constexpr int kBytes = kFlagOff + 16;
  static_assert(E * 4 <= kXsSlots * kSlotBytes, "partials fit in the ring");
  static_assert(kXOff % 16 == 0 && kSlotBytes % 128 == 0, "bulk copy destinations");
};

template <int MT, int TPW, int QF, int CPG, bool GATEUP>
__global__ void __launch_bounds__(kXsThreads) smallm_xs_kernel(DecodeParams p) {
  using S = XsSmem<MT, TPW, QF>;
  constexpr int E = S::E;
  constexpr int GPU = kUnitChunks / CPG;  // groups per full unit
  constexpr bool AFF = QF == kFormAffine;
  extern __shared__ __align__(128) uint8_t smem[];
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + S::kFlagOff);
  unsigned long long *best = reinterpret_cast<unsigned long long *>(smem + S::kBestOff);
  const uint32_t ring = smem_u32(smem + S::kRingOff);
  const uint32_t full0 = smem_u32(smem + S::kBarOff), empty0 = full0 + 8 * kXsSlots;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int tile_base = blockIdx.x * S::kTiles;
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < kXsSlots; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kXsWarps);
    }
    fence_mbar_init();
  }
  if (threadIdx.x < 16) best[threadIdx.x] = 0;
  __syncthreads();
  // this CTA's K units: the cluster ranks split K
  const int ub = (int)((long long)p.units * blockIdx.y / gridDim.y);
  const int ue = (int)((long long)p.units * (blockIdx.y + 1) / gridDim.y);
  const int nu = ue - ub;

  float acc[TPW][MT][4];
#pragma unroll
  for (int i = 0; i < TPW; ++i)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[i][mt][r] = 0.f;

  if (warp == kXsWarps) {
    // ------------------------------------------------------------ copies
    const uint64_t policy = evict_first_policy();
    // copy q of a unit: q < kTiles codes, then scale blocks, then zero/bias
    // blocks, then (q - kCopies) an x row
    auto issue = [&](int s, int u, bool weights, bool xrows) {
      const int nch = min(kUnitChunks, p.chunks - kUnitChunks * u);
      const uint32_t slot = ring + s * S::kSlotBytes;
      const uint32_t bar = full0 + 8 * s;
      const int upb = 4 * CPG / kUnitChunks;  // units per scale block
      const int nq = S::kCopies + p.M;
      for (int q = lane; q < nq; q += 32) {
        if (q < S::kCopies) {
          if (!weights) continue;
          const int kind = q / S::kTiles, i = q % S::kTiles;
          const size_t tile = (size_t)min(tile_base + i, p.tiles - 1);
          if (kind == 0)
            bulk_copy(slot + i * S::kTileCode, p.codes + (tile * p.chunks + (size_t)kUnitChunks * u) * kChunkBytes,
                      nch * kChunkBytes, bar, policy);
          else if (kind == 1)
            bulk_copy(slot + S::kScaleOff + i * kScaleBlockBytes,
                      p.scales + (tile * p.gblocks + (size_t)(u / upb)) * kScaleBlockBytes, kScaleBlockBytes, bar,
                      policy);
          else
            bulk_copy(slot + S::kThirdOff + i * S::kThird,
                      p.zeros + (tile * p.gblocks + (size_t)(u / upb)) * S::kThird, S::kThird, bar, policy);
        } else if (xrows) {
          const int m = q - S::kCopies;
          bulk_copy_keep(slot + S::kXOff + m * kXRowStride, p.x + (size_t)m * p.K + (size_t)kUnitChunks * 64 * u,
                         nch * 128, bar);
        }
      }
    };
    auto tx_bytes = [&](int u) {
      const int nch = min(kUnitChunks, p.chunks - kUnitChunks * u);
      return (uint32_t)(S::kTiles * (nch * kChunkBytes + kScaleBlockBytes + S::kThird) + p.M * nch * 128);
    };
    // the weights of the first slots stream before the previous kernel has
    // finished (programmatic overlap); x only after it
    const int first = min(kXsSlots, nu);
    for (int it = 0; it < first; ++it) {
      if (lane == 0) mbar_arrive_expect_tx(full0 + 8 * it, tx_bytes(ub + it));
      __syncwarp();
      issue(it, ub + it, true, false);
    }
    grid_launch_dependents();
    grid_dependency_wait();
    for (int it = 0; it < first; ++it) issue(it, ub + it, false, true);
    int issued = first;
    bool ok = true;
    for (; issued < nu; ++issued) {
      const int s = issued % kXsSlots;
      // every compute warp has released the slot (its previous unit)
      bool got = true;
      if (lane == 0) got = mbar_wait<true>(empty0 + 8 * s, ((issued / kXsSlots) - 1) & 1, abort_flag);
      got = __shfl_sync(0xFFFFFFFFu, got, 0);
      if (!got) {
        ok = false;
        break;
      }
      fence_proxy_async_smem();
      if (lane == 0) mbar_arrive_expect_tx(full0 + 8 * s, tx_bytes(ub + issued));
      __syncwarp();
      issue(s, ub + issued, true, true);
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      atomicExch(p.err, kErrTimeout);
    }
    // every copy issued has landed before the slots are reused for the partials
    if (lane == 0)
      for (int it = max(0, issued - kXsSlots); it < issued; ++it)
        mbar_wait_drain(full0 + 8 * (it % kXsSlots), (it / kXsSlots) & 1);
  } else {
    // ------------------------------------------------------------ compute warps
    grid_launch_dependents();
    grid_dependency_wait();
    for (int it = 0; it < nu; ++it) {
      const int u = ub + it;
      const int ngu = min(GPU, (p.chunks - kUnitChunks * u) / CPG);
      const int s = it % kXsSlots;
      const bool got = __all_sync(0xFFFFFFFFu, mbar_wait<true>(full0 + 8 * s, (it / kXsSlots) & 1, abort_flag));
      if (!got) {
        if (lane == 0) {
          *abort_flag = 1;
          atomicExch(p.err, kErrTimeout);
        }
        break;
      }
      const uint32_t sl = ring + s * S::kSlotBytes;
      // B fragment column g + 8 mt reads x row min(g + 8 mt, M - 1)
      uint32_t xrow[MT];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
        xrow[mt] = sl + S::kXOff + min(g + 8 * mt, p.M - 1) * kXRowStride + t * 32;
#pragma unroll
      for (int j = 0; j < GPU; ++j) {
        if (j < ngu) {
          const int gg = u * GPU + j;
          uint32_t zg[TPW], zg8[TPW];
#pragma unroll
          for (int i = 0; i < TPW; ++i) {
            if (QF != kFormZero) {
              zg[i] = zg8[i] = zero_pair(AFF ? 0 : 8);
            } else {
              const uint32_t zb = lds8(sl + S::kThirdOff + (warp * TPW + i) * kZeroBlockBytes + g * 4 + (gg & 3));
              zg[i] = zero_pair(zb & 0xF);
              zg8[i] = zero_pair(zb >> 4);
            }
          }
          float part[TPW][MT][4];
          float xs[MT][4];  // affine: the group's sum of x per column (all-ones A)
#pragma unroll
          for (int cc = 0; cc < CPG; ++cc) {
            const int cl = j * CPG + cc;  // chunk within the unit
            uint4 xx[MT][2];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              xx[mt][0] = lds128(xrow[mt] + cl * 128);
              xx[mt][1] = lds128(xrow[mt] + cl * 128 + 16);
            }
            uint4 w[TPW];
#pragma unroll
            for (int i = 0; i < TPW; ++i)
              w[i] = lds128(sl + (warp * TPW + i) * S::kTileCode + (cl * 32 + lane) * 16);
#pragma unroll
            for (int st = 0; st < 4; ++st) {
              uint32_t b0[MT], b1[MT];
#pragma unroll
              for (int mt = 0; mt < MT; ++mt) {
                b0[mt] = word_of(xx[mt][st >> 1], 2 * (st & 1));
                b1[mt] = word_of(xx[mt][st >> 1], 2 * (st & 1) + 1);
              }
              if (AFF) {
                const uint32_t ones[4] = {0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u};
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                  if (cc == 0 && st == 0)
                    mma_bf16_16816_zero(xs[mt], ones, b0[mt], b1[mt]);
                  else
                    mma_bf16_16816(xs[mt], ones, b0[mt], b1[mt]);
                }
              }
#pragma unroll
              for (int i = 0; i < TPW; ++i) {
                uint32_t a[4];
                unpack_word(word_of(w[i], st), zg[i], zg8[i], p.uc, a);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                  if (cc == 0 && st == 0)
                    mma_bf16_16816_zero(part[i][mt], a, b0[mt], b1[mt]);
                  else
                    mma_bf16_16816(part[i][mt], a, b0[mt], b1[mt]);
                }
              }
            }
          }
#pragma unroll
          for (int i = 0; i < TPW; ++i) {
            const uint32_t blk = (warp * TPW + i) * kScaleBlockBytes + g * 16 + (gg & 3) * 4;
            const uint32_t sw = lds32(sl + S::kScaleOff + blk);
            const float sg = bf16lo_to_f32(sw), sg8 = bf16hi_to_f32(sw);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              acc[i][mt][0] = fmaf(sg, part[i][mt][0], acc[i][mt][0]);
              acc[i][mt][1] = fmaf(sg, part[i][mt][1], acc[i][mt][1]);
              acc[i][mt][2] = fmaf(sg8, part[i][mt][2], acc[i][mt][2]);
              acc[i][mt][3] = fmaf(sg8, part[i][mt][3], acc[i][mt][3]);
            }
            if (AFF) {
              const uint32_t bw = lds32(sl + S::kThirdOff + blk);
              const float bg = bf16lo_to_f32(bw), bg8 = bf16hi_to_f32(bw);
#pragma unroll
              for (int mt = 0; mt < MT; ++mt) {
                acc[i][mt][0] = fmaf(bg, xs[mt][0], acc[i][mt][0]);
                acc[i][mt][1] = fmaf(bg, xs[mt][1], acc[i][mt][1]);
                acc[i][mt][2] = fmaf(bg8, xs[mt][2], acc[i][mt][2]);
                acc[i][mt][3] = fmaf(bg8, xs[mt][3], acc[i][mt][3]);
              }
            }
          }
        }
      }
      // this warp is done with the slot
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * s);
    }
  }

  // partials into the (now idle) ring, then the cluster's ranks are summed
  __syncthreads();
  float *red = reinterpret_cast<float *>(smem + S::kRedOff);
  if (warp < kXsWarps) {
#pragma unroll
    for (int i = 0; i < TPW; ++i)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int r = 0; r < 4; ++r) red[(((warp * TPW + i) * MT + mt) * 4 + r) * 32 + lane] = acc[i][mt][r];
  }
  if (!cluster_sum<E>(red)) return;

  // element e = ((ti*MT + mt)*4 + r)*32 + lane, ti = the CTA's tile index:
  //   row n = 16*(tile_base+ti) + g + 8*(r>>1), column m = 8*mt + 2t + (r&1)
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int ln = e & 31, r = (e >> 5) & 3, im = e >> 7;
    const int mt = im % MT, ti = im / MT;
    const int m = 8 * mt + 2 * (ln & 3) + (r & 1);
    const int nl = (ln >> 2) + 8 * (r >> 1);
    if (m >= p.M) continue;
    if (GATEUP) {
      if (ti & 1) continue;
      const int n = 16 * ((tile_base + ti) >> 1) + nl;
      if (n < p.N) {
        const float gv = red[e], uv = red[e + MT * 4 * 32];
        p.y[(size_t)m * p.ld + n] = f32_to_bf16_bits(silu_f32(gv) * uv);
      }
    } else {
      const int n = 16 * (tile_base + ti) + nl;
      if (n < p.N) {
        const uint16_t v = f32_to_bf16_bits(red[e]);
        if (p.y) p.y[(size_t)m * p.ld + n] = v;
        if (p.amax) atomicMax(best + m, argmax_key(v, n));
      }
    }
  }
  if (!GATEUP && p.amax) {
    __syncthreads();
    if (threadIdx.x < p.M && best[threadIdx.x] != 0) atomicMax(p.amax + threadIdx.x, best[threadIdx.x]);
  }
}

// ---------------------------------------------------------------------------
// one-row CUDA-core GEMV
// ---------------------------------------------------------------------------
template <int TPW, bool SYM, int CPG, int SLOTS>
__global__ void __launch_bounds__(kWarps * 32) gemv_m1_kernel(DecodeParams p) {
  constexpr int E = TPW * 2 * 8;  // (tile, row half, g)
  constexpr int GPU = kUnitChunks / CPG;
  constexpr int QF = SYM ? kFormSym : kFormZero;  // zero-point forms only
  using SM = DecodeSmem<TPW, QF, SLOTS, E>;
  using R = Ring<TPW, QF, SLOTS>;
  extern __shared__ __align__(128) uint8_t smem[];
  float(*red)[E] = reinterpret_cast<float(*)[E]>(smem + SM::kRedOff);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + SM::kFlagOff);

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int tile0 = blockIdx.x * TPW;
  if (threadIdx.x == 0) *abort_flag = 0;
  __syncthreads();
  int ub, ue;
  k_slice(p.units, ub, ue);
  const int nu = ue - ub;

  R ring;
  ring.setup(p, smem + SM::kRingOff + warp * R::kWarpBytes,
             reinterpret_cast<uint64_t *>(smem + SM::kBarOff) + warp * SLOTS, tile0, CPG);
  int issued = 0;  // warp-uniform
  for (; issued < SLOTS && issued < nu; ++issued) ring.issue(issued, ub + issued);
  grid_launch_dependents();
  grid_dependency_wait();
  const uint4 *xp = reinterpret_cast<const uint4 *>(p.x + 16 * t);

  float out[TPW][2];
#pragma unroll
  for (int i = 0; i < TPW; ++i) out[i][0] = out[i][1] = 0.f;

  // the float32 magic 2^23 (mantissa step 1) and the nibble masks live in
  // registers so each "nibble | magic" is one LOP3
  const uint32_t magic = p.uc.magic ^ 0x43004300u ^ 0x4B000000u;
  const uint32_t m0 = p.uc.mask & 0xFu, m1 = m0 << 4, m2 = m0 << 8, m3 = m0 << 12, m4 = m0 << 16;
  constexpr uint32_t kMagic = 0x4B000000u, kNeg = 0x80000000u;
  int it = 0;
  for (; it < nu; ++it) {
    const int u = ub + it;
    const int ngu = min(GPU, (p.chunks - kUnitChunks * u) / CPG);
    if (!wait_slot<SLOTS>(ring.bar0, it, abort_flag, p.err)) break;
    const uint32_t sl = ring.slot(it % SLOTS);
#pragma unroll
    for (int j = 0; j < GPU; ++j) {
      if (j < ngu) {
        const int gg = u * GPU + j;
        uint4 xx[CPG][2];
#pragma unroll
        for (int cc = 0; cc < CPG; ++cc) {
          const int c = kUnitChunks * u + j * CPG + cc;
          xx[cc][0] = ldg_keep(xp + (size_t)c * 8);
          xx[cc][1] = ldg_keep(xp + (size_t)c * 8 + 1);
        }
#pragma unroll
        for (int i = 0; i < TPW; ++i) {
          const uint32_t sw = lds32(sl + R::kScaleOff + i * kScaleBlockBytes + g * 16 + (gg & 3) * 4);
          uint32_t za = 8, zb = 8;
          if (!SYM) {
            const uint32_t zbyte = lds8(sl + R::kZeroOff + i * kZeroBlockBytes + g * 4 + (gg & 3));
            za = zbyte & 0xF;
            zb = zbyte >> 4;
          }
          // nibble j of a word: row g + 8*(j&1), place 16^p(j), k offset kofs(j)
          //   j : 0 1 2 3 4 5 6 7
          //   p : 0 1 2 3 4 0 1 2      (j = 5..7 are read from the word shifted right by 20)
          // -(2^23 + z * 16^p(j)) is added exactly (both operands are integers below 2^24).
          const float2 cz0 = make_float2(__uint_as_float(kNeg | kMagic | za), __uint_as_float(kNeg | kMagic | (zb << 4)));
          const float2 cz1 =
              make_float2(__uint_as_float(kNeg | kMagic | (za << 8)), __uint_as_float(kNeg | kMagic | (zb << 12)));
          const float2 cz2 =
              make_float2(__uint_as_float(kNeg | kMagic | (za << 16)), __uint_as_float(kNeg | kMagic | zb));
          const float2 cz3 =
              make_float2(__uint_as_float(kNeg | kMagic | (za << 4)), __uint_as_float(kNeg | kMagic | (zb << 8)));
          float2 part[4];  // pairs (j=0,1) (2,3) (4,5) (6,7)
#pragma unroll
          for (int q = 0; q < 4; ++q) part[q] = make_float2(0.f, 0.f);
#pragma unroll
          for (int cc = 0; cc < CPG; ++cc) {
            const int cl = j * CPG + cc;
            const uint4 wv = lds128(sl + i * R::kTileCode + (cl * 32 + lane) * 16);
#pragma unroll
            for (int st = 0; st < 4; ++st) {
              const uint32_t wd = word_of(wv, st);
              const uint32_t w20 = wd >> 20;
              const uint32_t xa = word_of(xx[cc][st >> 1], 2 * (st & 1));      // k+0, k+1
              const uint32_t xb = word_of(xx[cc][st >> 1], 2 * (st & 1) + 1);  // k+2, k+3
              const float x0 = bf16lo_to_f32(xa), x1 = bf16hi_to_f32(xa);
              const float x2 = bf16lo_to_f32(xb), x3 = bf16hi_to_f32(xb);
              const float2 v01 = make_float2(__uint_as_float(lop3_and_or(wd, m0, magic)),
                                             __uint_as_float(lop3_and_or(wd, m1, magic)));
              const float2 v23 = make_float2(__uint_as_float(lop3_and_or(wd, m2, magic)),
                                             __uint_as_float(lop3_and_or(wd, m3, magic)));
              const float2 v45 = make_float2(__uint_as_float(lop3_and_or(wd, m4, magic)),
                                             __uint_as_float(lop3_and_or(w20, m0, magic)));
              const float2 v67 = make_float2(__uint_as_float(lop3_and_or(w20, m1, magic)),
                                             __uint_as_float(lop3_and_or(w20, m2, magic)));
              // j=0,1 at k+0; j=2,3 at k+2; j=4,5 at k+1; j=6,7 at k+3
              part[0] = __ffma2_rn(make_float2(x0, x0), __fadd2_rn(v01, cz0), part[0]);
              part[1] = __ffma2_rn(make_float2(x2, x2), __fadd2_rn(v23, cz1), part[1]);
              part[2] = __ffma2_rn(make_float2(x1, x1), __fadd2_rn(v45, cz2), part[2]);
              part[3] = __ffma2_rn(make_float2(x3, x3), __fadd2_rn(v67, cz3), part[3]);
            }
          }
          // undo the 16^p places: row g gets j = 0, 2, 4, 6 (p = 0, 2, 4, 1),
          // row g + 8 gets j = 1, 3, 5, 7 (p = 1, 3, 0, 2)
          const float rg = part[0].x + part[1].x * 0x1p-8f + part[2].x * 0x1p-16f + part[3].x * 0x1p-4f;
          const float rg8 = part[0].y * 0x1p-4f + part[1].y * 0x1p-12f + part[2].y + part[3].y * 0x1p-8f;
          out[i][0] = fmaf(bf16lo_to_f32(sw), rg, out[i][0]);
          out[i][1] = fmaf(bf16hi_to_f32(sw), rg8, out[i][1]);
        }
      }
    }
    __syncwarp();
    if (issued < nu) {
      fence_proxy_async_smem();
      ring.issue(it % SLOTS, ub + issued);
      ++issued;
    }
  }
  if (it < nu && lane == 0) drain_ring<SLOTS>(ring.bar0, it, issued);

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
  int tpw, kc, smem;
};

// Split-K choice: grids that already fill the GPU stay unsplit (each warp
// then streams long K slices and its ring stays full); smaller grids take the
// largest cluster split (<= 8) that keeps them within one wave, with at least
// one K unit per warp (graph-timed: 5120 x 5120 at M = 5 takes 8.7 us split
// 4 ways against 10.3 us split 2 ways). Splitting a grid of more than half a
// wave (e.g. 1.4 waves at N = 34816) was measured slower at every factor.
template <typename Kern>
cudaError_t pick_cfg(Kern kern, int smem, int tiles, int units, int sm_count, int tpw, int device,
                     PerDevice &occ_cache, DecodeCfg &c) {
  c.tpw = tpw;
  c.smem = smem;
  const long long ctas = (tiles + tpw - 1) / tpw;
  int occ = occ_cache.v[device].load(std::memory_order_relaxed);
  if (occ == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, 32 * kWarps, smem) != cudaSuccess || occ < 1)
      occ = 1;
    occ_cache.v[device].store(occ, std::memory_order_relaxed);
  }
  const long long resident = (long long)occ * sm_count;
  c.kc = 1;
  while (c.kc < 8 && ctas * c.kc * 2 <= resident && units >= kWarps * c.kc * 2) c.kc *= 2;
  return cudaSuccess;
}

template <typename Kern>
cudaError_t launch_decode(Kern kern, const DecodeParams &prm, const DecodeCfg &cfg, cudaStream_t stream) {
  const int ctas = (prm.tiles + cfg.tpw - 1) / cfg.tpw;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(ctas, cfg.kc, 1);
  lc.blockDim = dim3(32 * kWarps, 1, 1);
  lc.dynamicSmemBytes = cfg.smem;
  lc.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (cfg.kc > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 1;
    attr[na].val.clusterDim.y = cfg.kc;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (prm.overlap) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  lc.attrs = attr;
  lc.numAttrs = na;
  return cudaLaunchKernelEx(&lc, kern, prm);
}

DecodeParams make_params(const GemmCall &c, const Layout &L) {
  DecodeParams p;
  p.x = c.x;
  p.codes = c.packed + L.codes_off;
  p.scales = c.packed + L.scales_off;
  p.zeros = c.packed + (c.sym == kFormAffine ? L.biases_off : c.sym == kFormSym ? L.scales_off : L.zeros_off);
  p.y = c.y;
  p.M = c.M;
  p.N = c.N;
  p.K = c.K;
  p.tiles = L.tiles;
  p.chunks = L.chunks;
  p.groups = L.groups;
  p.gblocks = L.gblocks;
  p.units = (L.chunks + kUnitChunks - 1) / kUnitChunks;
  p.ld = c.N;
  p.err = c.err;
  p.device = c.device;
  p.overlap = c.overlap;
  p.amax = reinterpret_cast<unsigned long long *>(c.amax);
  p.uc = host_unpack_consts();
  return p;
}

constexpr int slots_for(int tpw) { return tpw >= 4 ? 2 : W4A16_DECODE_SLOTS2; }

template <int MT, int TPW, int QF, int CPG, bool GATEUP>
cudaError_t run_mma(const DecodeParams &p, int sm_count, cudaStream_t s) {
  constexpr int SLOTS = slots_for(TPW);
  auto kern = smallm_mma_kernel<MT, TPW, QF, CPG, SLOTS, GATEUP>;
  static PerDevice occ;
  DecodeCfg cfg;
  cudaError_t e = pick_cfg(kern, DecodeSmem<TPW, QF, SLOTS, TPW * MT * 4 * 32>::kBytes, p.tiles, p.units,
                           sm_count, TPW, p.device, occ, cfg);
  return e != cudaSuccess ? e : launch_decode(kern, p, cfg, s);
}

// Two 16-row tiles per warp at every N (measured faster than four at the
// 248,320-row head: more resident warps per SM).
// n8 tiles of x rows by M (up to 32 rows)
template <int QF, int CPG, bool GATEUP>
cudaError_t run_mma_m(const DecodeParams &p, int sm_count, cudaStream_t s) {
  if (p.M <= 8) return run_mma<1, 2, QF, CPG, GATEUP>(p, sm_count, s);
  if (p.M <= 16) return run_mma<2, 2, QF, CPG, GATEUP>(p, sm_count, s);
  if (p.M <= 24) return run_mma<3, 2, QF, CPG, GATEUP>(p, sm_count, s);
  return run_mma<4, 2, QF, CPG, GATEUP>(p, sm_count, s);
}

template <int QF, bool GATEUP>
cudaError_t run_mma_g(const DecodeParams &p, int sm_count, int group, cudaStream_t s) {
  return group == 64 ? run_mma_m<QF, 1, GATEUP>(p, sm_count, s) : run_mma_m<QF, 2, GATEUP>(p, sm_count, s);
}

template <bool GATEUP>
cudaError_t run_mma_all(const DecodeParams &p, int sm_count, int form, int group, cudaStream_t s) {
  if (form == kFormSym) return run_mma_g<kFormSym, GATEUP>(p, sm_count, group, s);
  if (form == kFormAffine) return run_mma_g<kFormAffine, GATEUP>(p, sm_count, group, s);
  return run_mma_g<kFormZero, GATEUP>(p, sm_count, group, s);
}

// x-staged kernel: CTAs of kXsWarps * TPW tiles; the same split-K rule over
// the cluster's CTAs (at least two K units each). With `only_full`, nothing is
// launched (and *launched stays false) unless the grid covers a whole wave:
// graph-timed, the kernel is 3-8 % faster than the per-warp-ring kernel on
// the 248,320-row head at M = 1-8 and at N = 131072, and 20-35 % slower on
// grids below a wave (N <= 65536), where four times fewer CTAs hide less
// latency.
template <int MT, int TPW, int QF, int CPG, bool GATEUP>
cudaError_t run_xs(const DecodeParams &p, int sm_count, cudaStream_t s, bool only_full, bool *launched) {
  using S = XsSmem<MT, TPW, QF>;
  auto kern = smallm_xs_kernel<MT, TPW, QF, CPG, GATEUP>;
  static PerDevice occ_cache;
  int occ = occ_cache.v[p.device].load(std::memory_order_relaxed);
  if (occ == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kBytes);
    if (e != cudaSuccess) return e;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kXsThreads, S::kBytes) != cudaSuccess || occ < 1)
      occ = 1;
    occ_cache.v[p.device].store(occ, std::memory_order_relaxed);
  }
  const long long ctas = (p.tiles + S::kTiles - 1) / S::kTiles;
  const long long resident = (long long)occ * sm_count;
  if (only_full && ctas < resident) return cudaSuccess;
  *launched = true;
  int kc = 1;
  while (kc < 8 && ctas * kc * 2 <= resident && p.units >= kc * 2 * 2) kc *= 2;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)ctas, kc, 1);
  lc.blockDim = dim3(kXsThreads, 1, 1);
  lc.dynamicSmemBytes = S::kBytes;
  lc.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (kc > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 1;
    attr[na].val.clusterDim.y = kc;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (p.overlap) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  lc.attrs = attr;
  lc.numAttrs = na;
  return cudaLaunchKernelEx(&lc, kern, p);
}

template <int QF, int CPG, bool GATEUP>
cudaError_t run_xs_m(const DecodeParams &p, int sm_count, cudaStream_t s, bool only_full, bool *launched) {
  if (p.M <= 8) return run_xs<1, W4A16_XS_TPW, QF, CPG, GATEUP>(p, sm_count, s, only_full, launched);
  return run_xs<2, W4A16_XS_TPW, QF, CPG, GATEUP>(p, sm_count, s, only_full, launched);
}

template <int QF, bool GATEUP>
cudaError_t run_xs_g(const DecodeParams &p, int sm_count, int group, cudaStream_t s, bool only_full,
                     bool *launched) {
  return group == 64 ? run_xs_m<QF, 1, GATEUP>(p, sm_count, s, only_full, launched)
                     : run_xs_m<QF, 2, GATEUP>(p, sm_count, s, only_full, launched);
}

template <bool GATEUP>
cudaError_t run_xs_all(const DecodeParams &p, int sm_count, int form, int group, cudaStream_t s, bool only_full,
                       bool *launched) {
  if (form == kFormSym) return run_xs_g<kFormSym, GATEUP>(p, sm_count, group, s, only_full, launched);
  if (form == kFormAffine) return run_xs_g<kFormAffine, GATEUP>(p, sm_count, group, s, only_full, launched);
  return run_xs_g<kFormZero, GATEUP>(p, sm_count, group, s, only_full, launched);
}

template <bool SYM, int CPG>
cudaError_t run_gemv(const DecodeParams &p, int sm_count, cudaStream_t s) {
  constexpr int TPW = 2, SLOTS = slots_for(TPW);
  auto kern = gemv_m1_kernel<TPW, SYM, CPG, SLOTS>;
  static PerDevice occ;
  DecodeCfg cfg;
  cudaError_t e = pick_cfg(kern, DecodeSmem<TPW, SYM ? kFormSym : kFormZero, SLOTS, TPW * 16>::kBytes, p.tiles, p.units, sm_count, TPW,
                           p.device, occ, cfg);
  return e != cudaSuccess ? e : launch_decode(kern, p, cfg, s);
}

}  // namespace

cudaError_t launch_smallm_mma(const GemmCall &c, int sm_count) {
  const Layout L = make_layout(packed_rows(c), c.K, c.group, c.sym);
  DecodeParams p = make_params(c, L);
  // The x-staged kernel: forced; chosen for M <= 8 when its grid fills a
  // wave; and for 9-16 rows of a zero-point weight whose grid of 8-tile CTAs
  // spans at least 1.5 CTAs per SM (graph-timed against the per-warp-ring
  // kernel: 4-7 % faster at N = 34,816 for M = 9, 13 and 16 at K = 5120 and
  // 17,408; equal at N = 65,536; slower on grids below that, on the symmetric
  // 248,320-row head (0.7 %) and on the affine form (3 %)).
  const long long xs_ctas = (L.tiles + 7) / 8;
  const bool xs_mid = c.xs_mode == 1 && c.M >= 9 && c.sym == kFormZero && !c.gateup && !c.amax &&
                      2 * xs_ctas >= 3LL * sm_count;
  if (c.M <= 16 && (c.xs_mode == 2 || xs_mid || (c.xs_mode == 1 && c.M <= 8))) {
    bool launched = false;
    const bool only_full = c.xs_mode == 1 && !xs_mid;
    const cudaError_t e = c.gateup ? run_xs_all<true>(p, sm_count, c.sym, c.group, c.stream, only_full, &launched)
                                   : run_xs_all<false>(p, sm_count, c.sym, c.group, c.stream, only_full, &launched);
    if (e != cudaSuccess || launched) return e;
  }
  if (c.gateup) return run_mma_all<true>(p, sm_count, c.sym, c.group, c.stream);
  return run_mma_all<false>(p, sm_count, c.sym, c.group, c.stream);
}

cudaError_t launch_gemv_m1(const GemmCall &c, int sm_count) {
  const Layout L = make_layout(packed_rows(c), c.K, c.group, c.sym);
  DecodeParams p = make_params(c, L);
  if (c.sym == kFormAffine) return cudaErrorInvalidValue;  // the API routes affine to the MMA kernel
  if (c.sym) return c.group == 64 ? run_gemv<true, 1>(p, sm_count, c.stream) : run_gemv<true, 2>(p, sm_count, c.stream);
  return c.group == 64 ? run_gemv<false, 1>(p, sm_count, c.stream) : run_gemv<false, 2>(p, sm_count, c.stream);
}

}  // namespace w4a16
