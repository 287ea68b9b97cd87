// Top-k of bf16 rows on the device: the k largest entries of every row of
// the logits y [M][N], largest first. This widens the greedy token pick made
// on the GPU instead of copying the vocabulary's logits to the host (lucebox
// PR #823, description) from one pick to k, with the argmax conventions of
// this library: among equal values the lowest column first (-0 equals +0),
// and a NaN above +inf (NaNs among themselves by column).
//
// One cluster of S CTAs (S <= 16) per row, each CTA a contiguous slice of the
// row. Every value becomes its 16-bit order code (order_key16) and the k-th
// largest code is found by radix passes of 8 bits: each CTA counts its slice
// into a 256-bin shared histogram, the cluster's histograms are summed over
// distributed shared memory (every CTA forms the same total, so all of them
// agree on the threshold), and one warp walks the bins from the top. When the
// codes in and above the k-th code's high-byte bin number at most 2,048 (the
// usual case for logits), all of them are gathered into rank 0 and sorted.
// Otherwise a second pass finds the exact threshold code from the low bytes;
// each CTA collects the codes above it, and the codes equal to it in column
// order (in any order when every one of them is picked); the slices' counts
// give each CTA its offsets, and every pick goes into rank 0's shared memory.
// Rank 0 sorts by (code, lowest column first) with a bitonic network and
// writes the columns and their bf16 values. Nothing is allocated; no
// workspace.
#include "w4a16_internal.h"

namespace w4a16 {
namespace {

constexpr int kTkThreads = 1024;
constexpr int kTkWarps = kTkThreads / 32;
constexpr unsigned kFull = 0xFFFFFFFFu;

// A row's candidates at or above the threshold bin when there are few of
// them (the common case for logits): every one is gathered and sorted.
constexpr int kTkFewCand = 2048;

struct TopkSmem {
  uint32_t hist[2][256];   // this CTA's slice: pass 1 (high byte), pass 2 (low byte)
  uint32_t tot[2][256];    // the cluster's sums
  // few-candidates path: [0, 2048) this slice's candidates, [2048, 4096)
  // rank 0's gathered row; three-pass path: [0, 1024) rank 0's picks,
  // [1024, 2048) this slice's codes above the threshold, [2048, 3072) its
  // first codes equal to the threshold in column order
  unsigned long long buf[4096];
  uint32_t wsum[kTkWarps];
  uint32_t bin, above, ngt, neq, chunk, gbase, ebase;
};

// add `active` lanes' bins; lanes of a warp with the same bin add once
__device__ __forceinline__ void hist_add(uint32_t *hist, uint32_t bin, bool active) {
  const unsigned act = __ballot_sync(kFull, active);
  if (!active) return;
  const unsigned peers = __match_any_sync(act, bin);
  if ((int)(threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[bin], (uint32_t)__popc(peers));
}

// One warp: walking the 256 bins of `h` from the top with a count that
// starts at `base` (< k), the bin where the count reaches k and the count of
// the bins above it. h plus base hold at least k entries.
__device__ __forceinline__ void find_threshold(const uint32_t *h, uint32_t base, uint32_t k, uint32_t *bin_out,
                                               uint32_t *above_out) {
  const int lane = threadIdx.x & 31;
  uint32_t local[8], sum = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    local[i] = h[255 - 8 * lane - i];
    sum += local[i];
  }
  uint32_t inc = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(kFull, inc, o);
    if (lane >= o) inc += v;
  }
  const uint32_t exc = inc - sum;
  if (base + exc < k && base + inc >= k) {  // exactly one lane
    uint32_t cum = base + exc;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (cum + local[i] >= k) {
        *bin_out = 255 - 8 * lane - i;
        *above_out = cum;
        break;
      }
      cum += local[i];
    }
  }
}

// The cluster's histogram of pass `ps`: once every rank has counted its slice,
// every CTA sums every rank's hist[ps] into its tot[ps] (the histograms of the
// two passes are separate, so no rank overwrites one that another still reads).
__device__ __forceinline__ void cluster_total(TopkSmem &sm, int ps, uint32_t S, uint32_t rank) {
  cluster_sync_all();
  if (threadIdx.x < 256) {
    const uint32_t a = smem_u32(&sm.hist[ps][threadIdx.x]);
    uint32_t s = 0;
    for (uint32_t r = 0; r < S; ++r) s += r == rank ? sm.hist[ps][threadIdx.x] : ld_cluster_u32(mapa_shared(a, r));
    sm.tot[ps][threadIdx.x] = s;
  }
  __syncthreads();
}

// VEC values per thread and step: 8 (16-byte loads; rows 16-byte aligned, N
// a multiple of 8) or 1.
template <int VEC>
__device__ __forceinline__ void load_keys(const uint16_t *row, int v, uint32_t (&key)[VEC]) {
  if (VEC == 8) {
    const uint4 q = *reinterpret_cast<const uint4 *>(row + 8 * (size_t)v);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      key[2 * i] = order_key16(w[i] & 0xFFFFu);
      key[2 * i + 1] = order_key16(w[i] >> 16);
    }
  } else {
    key[0] = order_key16(row[v]);
  }
}

__device__ __forceinline__ unsigned long long pick_key(uint32_t code, uint32_t col) {
  return ((unsigned long long)code << 32) | (0xFFFFFFFFu - col);
}

// Block-wide bitonic sort of a[0, P) descending, P a power of two.
__device__ __forceinline__ void sort_desc(unsigned long long *a, int P) {
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      __syncthreads();
      for (int i = threadIdx.x; i < P; i += kTkThreads) {
        const int j = i ^ stride;
        if (j > i) {
          const unsigned long long x = a[i], c = a[j];
          const bool desc = (i & size) == 0;
          if (desc ? (x < c) : (x > c)) {
            a[i] = c;
            a[j] = x;
          }
        }
      }
    }
  }
  __syncthreads();
}

// Offsets of this CTA's `cnt` entries among the cluster's, in rank order
// (cluster-wide barrier first, so every rank's count is final).
__device__ __forceinline__ uint32_t rank_offset(const uint32_t *cnt, uint32_t rank) {
  uint32_t o = 0;
  for (uint32_t r = 0; r < rank; ++r) o += ld_cluster_u32(mapa_shared(smem_u32(cnt), r));
  return o;
}

template <int VEC>
__global__ void __launch_bounds__(kTkThreads, 1) topk_kernel(const uint16_t *y, int N, int k, int64_t *idx_out,
                                                             uint16_t *val_out) {
  __shared__ TopkSmem sm;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t S = cluster_nctarank(), rank = cluster_ctarank();
  const size_t row_id = cluster_id_x();
  const uint16_t *row = y + row_id * (size_t)N;
  const uint32_t K = (uint32_t)k;
  const long long nv = N / VEC;  // steps of VEC values; this CTA's slice [v0, v1)
  const int v0 = (int)(nv * rank / S), v1 = (int)(nv * (rank + 1) / S);

  // the logits are the previous kernel's output (programmatic overlap)
  grid_launch_dependents();
  grid_dependency_wait();

  for (int i = tid; i < 512; i += kTkThreads) (&sm.hist[0][0])[i] = 0;
  if (tid == 0) {
    sm.bin = 0;
    sm.above = 0;
    sm.ngt = 0;
    sm.neq = 0;
  }
  __syncthreads();

  // pass 1: the high byte of every code
  for (int b = v0; b < v1; b += kTkThreads) {
    const int v = b + tid;
    const bool ok = v < v1;
    uint32_t key[VEC];
    if (ok) load_keys<VEC>(row, v, key);
#pragma unroll
    for (int j = 0; j < VEC; ++j) hist_add(sm.hist[0], ok ? key[j] >> 8 : 0u, ok);
  }
  cluster_total(sm, 0, S, rank);
  if (warp == 0) find_threshold(sm.tot[0], 0, K, &sm.bin, &sm.above);
  __syncthreads();
  const uint32_t hb = sm.bin, above1 = sm.above;
  const uint32_t pick0 = smem_u32(&sm.buf[0]);

  if (above1 + sm.tot[0][hb] <= (uint32_t)kTkFewCand) {
    // few candidates: every code whose high byte is hb or above, gathered
    // into rank 0 (slots [2048, 4096)) and sorted there
    unsigned long long *cand = sm.buf;
    for (int b = v0; b < v1; b += kTkThreads) {
      const int v = b + tid;
      const bool ok = v < v1;
      uint32_t key[VEC];
      if (ok) load_keys<VEC>(row, v, key);
      uint32_t n = 0;
#pragma unroll
      for (int j = 0; j < VEC; ++j) n += ok && (key[j] >> 8) >= hb;
      if (n) {
        uint32_t slot = atomicAdd(&sm.ngt, n);  // the cluster holds at most kTkFewCand of them
#pragma unroll
        for (int j = 0; j < VEC; ++j)
          if (ok && (key[j] >> 8) >= hb) cand[slot++] = pick_key(key[j], (uint32_t)(VEC * v + j));
      }
    }
    cluster_sync_all();
    if (tid == 0) sm.gbase = rank_offset(&sm.ngt, rank);
    __syncthreads();
    const uint32_t rdst = mapa_shared(pick0 + 8u * kTkFewCand, 0);
    for (uint32_t i = tid; i < sm.ngt; i += kTkThreads) st_cluster_u64(rdst + 8u * (sm.gbase + i), cand[i]);
    cluster_sync_all();
    if (rank != 0) return;
    const uint32_t total = above1 + sm.tot[0][hb];
    unsigned long long *all = sm.buf + kTkFewCand;
    int P = 1;
    while ((uint32_t)P < total) P <<= 1;
    for (int i = (int)total + tid; i < P; i += kTkThreads) all[i] = 0ull;
    sort_desc(all, P);
    for (int j = tid; j < k; j += kTkThreads) {
      const uint32_t n = 0xFFFFFFFFu - (uint32_t)(all[j] & 0xFFFFFFFFull);
      idx_out[row_id * (size_t)k + j] = (int64_t)n;
      if (val_out) val_out[row_id * (size_t)k + j] = row[n];
    }
    return;
  }

  // pass 2: the low byte of the codes whose high byte is hb
  for (int b = v0; b < v1; b += kTkThreads) {
    const int v = b + tid;
    const bool ok = v < v1;
    uint32_t key[VEC];
    if (ok) load_keys<VEC>(row, v, key);
#pragma unroll
    for (int j = 0; j < VEC; ++j) hist_add(sm.hist[1], ok ? key[j] & 0xFFu : 0u, ok && (key[j] >> 8) == hb);
  }
  cluster_total(sm, 1, S, rank);
  if (warp == 0) find_threshold(sm.tot[1], above1, K, &sm.bin, &sm.above);
  __syncthreads();
  const uint32_t thr = (hb << 8) | sm.bin, above = sm.above, need = K - above;
  const bool all_eq = sm.tot[1][sm.bin] == need;  // every code equal to thr is picked: no order needed
  unsigned long long *gt = sm.buf + 1024, *eq = sm.buf + 2048;

  // pass 3: this slice's codes above thr (any order), and its codes equal to
  // thr in column order (the first `need` of them are all that can be picked)
  for (int b = v0; b < v1; b += kTkThreads) {
    const int v = b + tid;
    const bool ok = v < v1;
    uint32_t key[VEC];
    if (ok) load_keys<VEC>(row, v, key);
    uint32_t ngt = 0, neq = 0;
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
      ngt += ok && key[j] > thr;
      neq += ok && key[j] == thr;
    }
    if (ngt) {
      uint32_t slot = atomicAdd(&sm.ngt, ngt);  // below `above` <= kTopkMaxK
#pragma unroll
      for (int j = 0; j < VEC; ++j)
        if (ok && key[j] > thr) gt[slot++] = pick_key(key[j], (uint32_t)(VEC * v + j));
    }
    if (all_eq) {
      if (neq) {
        uint32_t slot = atomicAdd(&sm.neq, neq);  // below `need`
#pragma unroll
        for (int j = 0; j < VEC; ++j)
          if (ok && key[j] == thr) eq[slot++] = pick_key(key[j], (uint32_t)(VEC * v + j));
      }
      continue;
    }
    // block exclusive scan of neq (threads in column order)
    uint32_t inc = neq;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(kFull, inc, o);
      if (lane >= o) inc += t;
    }
    if (lane == 31) sm.wsum[warp] = inc;
    __syncthreads();
    if (warp == 0) {
      const uint32_t ws = sm.wsum[lane];
      uint32_t wi = ws;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(kFull, wi, o);
        if (lane >= o) wi += t;
      }
      sm.wsum[lane] = wi - ws;
      if (lane == 31) sm.chunk = wi;
    }
    __syncthreads();
    if (neq) {
      uint32_t pos = sm.neq + sm.wsum[warp] + inc - neq;
#pragma unroll
      for (int j = 0; j < VEC; ++j)
        if (ok && key[j] == thr) {
          if (pos < need) eq[pos] = pick_key(key[j], (uint32_t)(VEC * v + j));
          ++pos;
        }
    }
    __syncthreads();
    if (tid == 0) sm.neq += sm.chunk;
    __syncthreads();
  }

  // offsets from the slices before this one, then every pick into rank 0
  cluster_sync_all();
  if (tid == 0) {
    sm.gbase = rank_offset(&sm.ngt, rank);
    sm.ebase = rank_offset(&sm.neq, rank);
  }
  __syncthreads();
  const uint32_t gt_base = sm.gbase, eq_base = sm.ebase;
  const uint32_t rpick = rank == 0 ? pick0 : mapa_shared(pick0, 0);
  for (uint32_t i = tid; i < sm.ngt; i += kTkThreads) st_cluster_u64(rpick + 8 * (gt_base + i), gt[i]);
  const uint32_t neq_take = eq_base >= need ? 0u : min(sm.neq, need - eq_base);
  for (uint32_t i = tid; i < neq_take; i += kTkThreads) st_cluster_u64(rpick + 8 * (above + eq_base + i), eq[i]);
  cluster_sync_all();
  if (rank != 0) return;

  // rank 0: the k picks sorted descending (padding below every pick)
  unsigned long long *pick = sm.buf;
  int P = 1;
  while (P < k) P <<= 1;
  for (int i = k + tid; i < P; i += kTkThreads) pick[i] = 0ull;
  sort_desc(pick, P);
  for (int j = tid; j < k; j += kTkThreads) {
    const uint32_t n = 0xFFFFFFFFu - (uint32_t)(pick[j] & 0xFFFFFFFFull);
    idx_out[row_id * (size_t)k + j] = (int64_t)n;
    if (val_out) val_out[row_id * (size_t)k + j] = row[n];
  }
}

// CTAs per row: about 8K values per CTA, a power of two up to 16 (16 needs
// the non-portable cluster size; 8 is used where 16 does not fit)
template <int VEC>
cudaError_t launch_vec(const uint16_t *y, int M, int N, int k, int64_t *idx, uint16_t *vals, bool overlap,
                       int device, cudaStream_t stream) {
  auto kern = topk_kernel<VEC>;
  static PerDevice fits16;  // 1: clusters of 16 fit, -1: they do not
  int S = 1;
  while (S < 16 && (long long)N >= 2LL * 8192 * S) S *= 2;
  if (S == 16) {
    int f = fits16.v[device].load(std::memory_order_relaxed);
    if (f == 0) {
      f = -1;
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
        cudaLaunchConfig_t lc = {};
        lc.gridDim = dim3(16, 1, 1);
        lc.blockDim = dim3(kTkThreads, 1, 1);
        cudaLaunchAttribute a;
        a.id = cudaLaunchAttributeClusterDimension;
        a.val.clusterDim.x = 16;
        a.val.clusterDim.y = 1;
        a.val.clusterDim.z = 1;
        lc.attrs = &a;
        lc.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &lc) == cudaSuccess && n >= 1) f = 1;
      }
      (void)cudaGetLastError();
      fits16.v[device].store(f, std::memory_order_relaxed);
    }
    if (f < 0) S = 8;
  }
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)(M * S), 1, 1);
  lc.blockDim = dim3(kTkThreads, 1, 1);
  lc.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  int na = 1;
  if (overlap) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  lc.attrs = attr;
  lc.numAttrs = na;
  return cudaLaunchKernelEx(&lc, kern, y, N, k, idx, vals);
}

}  // namespace

cudaError_t launch_topk(const uint16_t *y, int M, int N, int k, int64_t *idx, uint16_t *vals, bool overlap,
                        int device, cudaStream_t stream) {
  // 16-byte loads when every row starts on a 16-byte boundary
  if (N % 8 == 0 && (reinterpret_cast<uintptr_t>(y) & 15) == 0)
    return launch_vec<8>(y, M, N, k, idx, vals, overlap, device, stream);
  return launch_vec<1>(y, M, N, k, idx, vals, overlap, device, stream);
}

}  // namespace w4a16
