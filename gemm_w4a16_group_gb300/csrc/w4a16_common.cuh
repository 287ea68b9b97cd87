// Device-side helpers shared by the W4A16 kernels: the repacked layout, the
// exact nibble -> bf16 (q - z) rebuild, and thin wrappers over the sm_100-family
// PTX used by the tcgen05 GEMM (mbarrier, TMA, tcgen05.*).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace w4a16 {

// ---------------------------------------------------------------------------
// Repacked layout (see w4a16_repack in w4a16.h)
//
//  Rows are tiled 16 at a time (tile T = rows 16T .. 16T+15) and K in chunks
//  of 64. For tile T, chunk c and lane L = 4g + t (g = 0..7, t = 0..3) there is
//  one 16-byte run of four 32-bit words s = 0..3. Word s holds the codes of
//  rows 16T+g and 16T+g+8 at k = 64c + 16t + 4s + {0..3}:
//
//     nibble j of word s  ->  row 16T + g + 8*(j & 1),  k = 64c + 16t + 4s + kofs(j)
//     kofs(j) = 2*((j >> 1) & 1) + (j >> 2)        (0,0,2,2,1,1,3,3)
//
//  so that ((word >> 4p) & 0x000F000F) puts the two codes of one mma.sync A
//  register (row g or g+8, two consecutive k) into the two 16-bit halves, and
//  the 16 values of k a lane owns are contiguous in x.
//
//  Scales: per tile, per block of four groups, [g 0..7][group j 0..3][h 0..1]
//  bf16 = scale(row 16T + g + 8h, group 4*blk + j): 128 bytes per block.
//  Zeros (zero-point form only): per tile and block, [g][j] bytes holding
//  zero(row g) | zero(row g+8) << 4: 32 bytes per block.
//  Biases (affine form only): the scales' layout with bias for scale.
//  Bias operand (affine form only): bf16 [16 * tiles][kb3], kb3 = 3 * groups
//  rounded up to 64; row r holds bias(r, g) at columns 3g, 3g+1, 3g+2 and 0
//  beyond. Against the group sums of x split into three bf16 parts (hi, mid,
//  lo at the same columns), one K-major MMA operand pair gives
//  sum_g bias * X_g on the tensor cores.
// ---------------------------------------------------------------------------
constexpr int kTileRows = 16;
constexpr int kChunkK = 64;
constexpr int kChunkBytes = 512;      // 32 lanes x 16 bytes
constexpr int kScaleBlockBytes = 128; // per tile, per 4 groups
constexpr int kZeroBlockBytes = 32;

// Weight forms (the `sym` argument of the C ABI):
//   kFormZero   w = (q - z) * scale, z a packed 4-bit zero point per group
//   kFormSym    w = (q - 8) * scale
//   kFormAffine w = scale * q + bias, bias bf16 per group
constexpr int kFormZero = 0, kFormSym = 1, kFormAffine = 2;

struct Layout {
  int N, K, group, sym;  // sym: the form
  int tiles;       // ceil(N / 16)
  int chunks;      // K / 64
  int groups;      // K / group
  int gblocks;     // ceil(groups / 4)
  int kb3;         // affine: columns of the bias operand (3 * groups rounded up to 64)
  size_t codes_off, scales_off, zeros_off, biases_off, bops_off, total;
};

// columns of the affine bias operand and of the split x group sums
__host__ __device__ inline int affine_kb3(int groups) { return (3 * groups + 63) / 64 * 64; }

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

__host__ __device__ inline Layout make_layout(int N, int K, int group, int form) {
  Layout L;
  L.N = N; L.K = K; L.group = group; L.sym = form;
  L.tiles = (N + kTileRows - 1) / kTileRows;
  L.chunks = K / kChunkK;
  L.groups = K / group;
  L.gblocks = (L.groups + 3) / 4;
  L.codes_off = 0;
  L.scales_off = align_up((size_t)L.tiles * L.chunks * kChunkBytes, 256);
  L.zeros_off = align_up(L.scales_off + (size_t)L.tiles * L.gblocks * kScaleBlockBytes, 256);
  L.biases_off = align_up(L.zeros_off + (form == kFormZero ? (size_t)L.tiles * L.gblocks * kZeroBlockBytes : 0), 256);
  L.bops_off = align_up(L.biases_off + (form == kFormAffine ? (size_t)L.tiles * L.gblocks * kScaleBlockBytes : 0), 256);
  L.kb3 = affine_kb3(L.groups);
  L.total = align_up(L.bops_off + (form == kFormAffine ? (size_t)L.tiles * 16 * L.kb3 * 2 : 0), 256);
  return L;
}

// ---------------------------------------------------------------------------
// Exact unpack. bf16 0x4300 is 128.0 with a mantissa step of 1, so
// (0x4300 | c) is exactly 128 + c for a 4-bit c, and subtracting the bf16
// value 128 + z leaves the integer q - z (|q - z| <= 15) exactly. This is the
// "(0x4300 | c) - 128" code rebuild of the TensorFold PR #859 lane GEMV, with
// the zero point folded into the subtrahend.
// ---------------------------------------------------------------------------
constexpr uint32_t kNibMask = 0x000F000Fu;
constexpr uint32_t kBf16x2_128 = 0x43004300u;

// bf16x2 (128 + z) in both halves
__device__ __forceinline__ uint32_t zero_pair(uint32_t z) { return kBf16x2_128 | (z * 0x00010001u); }

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
  __nv_bfloat162 r = __hsub2(*reinterpret_cast<__nv_bfloat162 *>(&a),
                             *reinterpret_cast<__nv_bfloat162 *>(&b));
  return *reinterpret_cast<uint32_t *>(&r);
}

// (w & mask) | magic as ONE three-input LOP3. With both constants as
// immediates the compiler splits it into two logic ops, and the integer ALU
// pipe is what bounds the unpack rate, so the constants travel in registers
// (UnpackConsts comes in as a kernel argument and is not constant-folded).
struct UnpackConsts {
  uint32_t mask;   // kNibMask
  uint32_t magic;  // kBf16x2_128
};
inline UnpackConsts host_unpack_consts() { return UnpackConsts{kNibMask, kBf16x2_128}; }

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t w, uint32_t mask, uint32_t magic) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(w), "r"(mask), "r"(magic));  // (a & b) | c
  return d;
}

// Four bf16x2 registers of 128 + q from one packed word: out[p] holds nibble
// p (low half) and nibble p + 4 (high half); out[0], out[2] are row g,
// out[1], out[3] row g + 8. Three shifts and four LOP3s, all exact.
__device__ __forceinline__ void unpack_word_biased(uint32_t w, const UnpackConsts &uc, uint32_t out[4]) {
  out[0] = lop3_and_or(w, uc.mask, uc.magic);
  out[1] = lop3_and_or(w >> 4, uc.mask, uc.magic);
  out[2] = lop3_and_or(w >> 8, uc.mask, uc.magic);
  out[3] = lop3_and_or(w >> 12, uc.mask, uc.magic);
}

// Same registers holding q - z exactly: zg = zero_pair(z of row g) is
// subtracted from out[0], out[2] and zg8 (row g + 8) from out[1], out[3].
__device__ __forceinline__ void unpack_word(uint32_t w, uint32_t zg, uint32_t zg8, const UnpackConsts &uc,
                                            uint32_t out[4]) {
  unpack_word_biased(w, uc, out);
  out[0] = bf16x2_sub(out[0], zg);
  out[1] = bf16x2_sub(out[1], zg8);
  out[2] = bf16x2_sub(out[2], zg);
  out[3] = bf16x2_sub(out[3], zg8);
}

// Argmax over bf16 outputs as one unsigned 64-bit key, so that atomicMax
// finds the maximum and, among equal values, the lowest index (the first
// occurrence). High half: the bf16 bits mapped to an order-preserving
// unsigned code, -0 as +0, every NaN above +inf (a NaN is the maximum).
// Low half: 0xFFFFFFFF - n. Key 0 is below every output.
// The order-preserving 16-bit code of a bf16 value: larger code = larger
// value, -0 and +0 share 0x8000, every NaN is 0xFFFF (above +inf's 0xFF80).
__device__ __forceinline__ uint32_t order_key16(uint32_t bits) {
  bits &= 0xFFFFu;
  if (bits == 0x8000u) bits = 0;
  uint32_t o = (bits & 0x8000u) ? (~bits & 0xFFFFu) : (bits | 0x8000u);
  if ((bits & 0x7F80u) == 0x7F80u && (bits & 0x7Fu)) o = 0xFFFFu;
  return o;
}

__device__ __forceinline__ unsigned long long argmax_key(uint32_t bits, int n) {
  return ((unsigned long long)order_key16(bits) << 32) | (0xFFFFFFFFu - (uint32_t)n);
}

__device__ __forceinline__ float bf16lo_to_f32(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// ---------------------------------------------------------------------------
// Error word written by kernels (bounded waits that gave up).
// ---------------------------------------------------------------------------
constexpr int kErrTimeout = 1;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s per wait

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch. wait: block until the grids this one depends
// on (the previous kernel on the stream, when launched with programmatic
// stream serialization) have completed and their writes are visible; returns
// at once otherwise. launch_dependents: the next such kernel may be scheduled
// once every CTA of this grid has executed it (or exited).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Explicit shared-window loads and stores (32-bit shared addresses): pointers
// that pass through integer casts or structures otherwise become generic
// accesses, which cost extra address work in the hot loops.
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ float4 lds128f(uint32_t a) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
// SiLU(g) = g / (1 + e^-g) with the fast exponential and division: a few
// float32 ulps, far inside the output's bf16 rounding (the IEEE division is a
// long instruction sequence that stalled the prompt GEMM's per-tile output
// phase for ~12 us). When e^-g overflows (g < -88) the quotient is 0, the
// function's limit.
__device__ __forceinline__ float silu_f32(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

__device__ __forceinline__ uint32_t lds16(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds8(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void sts32f(uint32_t a, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// One bounded probe: the thread may sleep up to kSuspendHintNs waiting for the
// phase (it wakes when the phase completes), so waiting warps do not spin on
// issue slots that the single MMA-issuing and TMA-issuing threads need.
constexpr uint32_t kSuspendHintNs = 20000;
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Non-blocking test of the phase. On a phase already complete it costs ~17
// cycles, against ~51 for try_wait with the suspend hint (measured on GB300).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: true when the phase completed, false after kWaitLimitNs or
// when *abort became non-zero (another role gave up). TEST_FIRST: look with
// the cheap test before sleeping in try_wait (the decode kernels' slot waits
// usually find the phase complete: 0.3-0.8 % faster; the tcgen05 GEMM's
// issuing thread is 4.5 % slower with it, so it keeps the plain form).
template <bool TEST_FIRST = false>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort) {
  if (TEST_FIRST && mbar_test_wait(bar, parity)) return true;
  if (mbar_try_wait(bar, parity)) return true;
  unsigned long long t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 7u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
  }
}

// Bounded wait that ignores the abort flag: used after giving up, to let
// asynchronous work this thread started finish before the CTA exits.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
  unsigned long long t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 7u) == 7u && globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// ---------------------------------------------------------------------------
// thread-block clusters: rank, distributed shared memory, remote arrivals
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t nclusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// the same shared-memory offset in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// every thread of every CTA of the cluster
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrive on an mbarrier of another CTA (address from mapa_shared) with the
// default semantics. Used where the waiting side only hands the data to the
// tensor cores (smem operands the arriving warp wrote after a proxy fence, or
// TMEM columns it finished reading): the arrival reaches the barrier after the
// warp's shared-memory accesses. A release at cluster scope would add a full
// memory barrier (~0.8 us measured) to every arrival.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t cluster_addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t cluster_addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(cluster_addr) : "memory");
  return v;
}
__device__ __forceinline__ void st_cluster_u64(uint32_t cluster_addr, unsigned long long v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(cluster_addr), "l"(v) : "memory");
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// ---------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor) and proxy fences
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, int c0, int c1,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const void *tmap, int c0, int c1, uint32_t bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const void *tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// generic-proxy shared-memory writes -> visible to the async proxy (tensor core)
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] . B[smem]^T, kind::f16, single CTA
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] . B[smem]^T, kind::f16, single CTA. A (M = 128) sits
// in TMEM lanes 0-127, one row per lane, two consecutive k of bf16 per 32-bit
// column (the low half the smaller k): 8 columns per K = 16 instruction.
__device__ __forceinline__ void tc_mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Four repetitions of the 16-lane x 256-bit store: thread 4g + t writes, for
// repetition i, v[4i], v[4i+1] to lane g at columns 8i + 2t, 8i + 2t + 1 and
// v[4i+2], v[4i+3] to lane g + 8 at the same columns (lanes from taddr's lane
// field, which stays inside the warp's 32-lane quarter of TMEM).
__device__ __forceinline__ void tmem_st_16x256b_x4(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
// this thread's tcgen05.st operations have completed
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 8 / 16 consecutive 32-bit TMEM columns of this thread's lane (32x32b shape)
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                 "=r"(r[7])
               : "r"(taddr)
               : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// mbarrier arrives once every tcgen05 op issued so far by this thread completed
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// The CTA-pair forms (cta_group::2). A kernel uses one cta_group throughout:
// allocation, MMA, commit and deallocation. Allocation and deallocation are
// performed by one warp in each CTA of the pair; the MMA is issued by one
// thread of the pair and reads rows 0-127 of A and the first N/2 rows of B
// from the smem of the even CTA, the rest from the odd CTA at the same
// offsets, writing D lanes 0-127 to the even CTA's TMEM and 128-255 to the odd
// CTA's, at the same TMEM address.
__device__ __forceinline__ void tmem_alloc2(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish2() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_mma2_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// arrive on this CTA's mbarrier once the pair MMAs issued so far completed
__device__ __forceinline__ void tc_commit2(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
// ... on the mbarrier at this offset in every CTA of cta_mask
__device__ __forceinline__ void tc_commit2_mc(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          bar),
      "h"(cta_mask)
      : "memory");
}

// 32 consecutive 32-bit TMEM columns of this thread's lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor for a K-major operand stored with the
// 128-byte swizzle: rows of 64 bf16 (128 B), 8-row atoms of 1024 B stacked
// along M/N (stride 1024 B), descriptor version 1, swizzle mode 2 (128 B).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_addr) {
  return (uint64_t)((smem_addr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor, kind::f16: D f32, A and B bf16, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

}  // namespace w4a16
