// C ABI (include/w4a16.h): argument checks, device checks and kernel choice.
// Nothing is launched when a check fails; every check that needs no GPU runs
// before the first CUDA call.
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "w4a16.h"
#include "w4a16_internal.h"

using namespace w4a16;

namespace {

thread_local int t_last_cuda_error = 0;
std::atomic<int> g_override{0};
std::atomic<int> g_overlap{0};

// Device error word set by kernels whose bounded waits gave up.
__device__ int g_kernel_error;

// Fixed table of x group sums for w4a16_gemm_affine_noalloc (4 MiB per device,
// part of the module image: nothing is allocated at run time).
constexpr size_t kNoAllocXsumBytes = size_t(4) << 20;
static __device__ __align__(256) uint16_t g_noalloc_xsum[kNoAllocXsumBytes / sizeof(uint16_t)];

struct DeviceInfo {
  int device = 0;
  bool ready = false;
  int status = W4A16_OK;
  int sm_count = 0;
  int *err = nullptr;
  uint16_t *noalloc_xsum = nullptr;  // this device's copy of g_noalloc_xsum
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

int cuda_fail(cudaError_t e) {
  t_last_cuda_error = (int)e;
  return W4A16_ERR_CUDA;
}

// Current device's properties and error-word address (looked up once per device).
int current_device(DeviceInfo &out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return W4A16_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo &d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e);
    if (major != 10 || minor != 3) {
      d.status = W4A16_ERR_UNSUPPORTED;  // the kernels are built for sm_103a only
    } else {
      void *p = nullptr;
      if ((e = cudaGetSymbolAddress(&p, g_kernel_error)) != cudaSuccess) return cuda_fail(e);
      d.err = static_cast<int *>(p);
      if ((e = cudaGetSymbolAddress(&p, g_noalloc_xsum)) != cudaSuccess) return cuda_fail(e);
      d.noalloc_xsum = static_cast<uint16_t *>(p);
      d.sm_count = sms;
      d.status = W4A16_OK;
    }
    d.device = dev;
    d.ready = true;
  }
  out = d;
  return d.status;
}

bool sizes_ok(long long M, long long N, long long K, int group) {
  const long long lim = (1LL << 31) / 16;
  if (group != 64 && group != 128) return false;
  if (M < 1 || N < 1 || K < 64 || M >= lim || N >= lim || K >= lim) return false;
  return K % group == 0;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int finish_launch(cudaError_t e) { return e == cudaSuccess ? W4A16_OK : cuda_fail(e); }

// The kernel override is read once per call (`ov`, from g_override) and that
// value decides both the argument checks and the launch, so a concurrent
// w4a16_set_kernel_override cannot send a call the checks did not accept.

// The decode kernels (M <= 32): override 2 keeps the per-warp-ring kernel, override 4
// forces the x-staged one, otherwise the x-staged kernel takes M <= 8 calls
// whose grid fills a wave and 9-16-row zero-point calls on grids of at least
// 1.5 CTAs per SM (launch_smallm_mma)
cudaError_t launch_decode_kernel(GemmCall &c, int sm_count, int ov) {
  c.xs_mode = ov == 4 ? 2 : ov == 2 ? 0 : 1;
  return launch_smallm_mma(c, sm_count);
}

// Rows that go to a decode kernel rather than the tcgen05 GEMM: M <= 32
// (graph-timed at N = 34816, K = 5120: M = 17-24 36.5 us against 66.8 on the
// tcgen05 GEMM, M = 32 47.6 against 66.8; 3.7-4.9x at N = 5120, where the
// GEMM has few tiles), unless the tcgen05 GEMM is forced (override 3)
constexpr int kDecodeMaxM = 32;
bool use_decode(int M, int ov) { return M <= kDecodeMaxM && ov != 3; }

bool form_ok(int form) { return form == kFormZero || form == kFormSym || form == kFormAffine; }
bool zero_form(int form) { return form == kFormZero || form == kFormSym; }

// The affine calls: the decode kernel for M <= 32 (it forms the x group sums
// itself), else the tcgen05 GEMM, which reads them from `xsum`.
bool affine_uses_tc(int M, int ov) { return !use_decode(M, ov); }

int launch_affine(GemmCall &c, const uint16_t *xsum, const DeviceInfo &d, int ov) {
  if (!affine_uses_tc(c.M, ov)) return finish_launch(launch_decode_kernel(c, d.sm_count, ov));
  c.xsum = xsum;
  return finish_launch(launch_prompt_tc(c, d.sm_count));
}

// b-bit affine weights: 2-4 bits widened into nibbles, 5-8 bits in two
// nibble planes over K' = 2K (x's groups each written twice)
bool bits_ok(int bits) { return bits >= 2 && bits <= 8; }
int bits_planes(int bits) { return bits > 4 ? 2 : 1; }
size_t widened_x_bytes(int M, int K, int bits) {
  return bits > 4 ? align_up((size_t)M * 2 * (size_t)K * sizeof(uint16_t), 256) : 0;
}

// rows of a gate/up buffer (each weight padded to 128 rows), or -1 if too many
long long gateup_rows(int N_each) {
  const long long rows = 2LL * ((N_each + 127) / 128 * 128);
  return rows >= (1LL << 31) / 16 ? -1 : rows;
}


}  // namespace

extern "C" {

size_t w4a16_repacked_bytes(int N, int K, int group, int sym) {
  if (!sizes_ok(1, N, K, group) || !form_ok(sym)) return 0;
  return make_layout(N, K, group, sym).total;
}

size_t w4a16_gateup_repacked_bytes(int N_each, int K, int group, int sym) {
  if (!sizes_ok(1, N_each, K, group) || !form_ok(sym)) return 0;
  const long long rows = gateup_rows(N_each);
  if (rows < 0) return 0;
  return make_layout((int)rows, K, group, sym).total;
}

int w4a16_repack(const int32_t *qweight, const uint16_t *scales, const int32_t *zeros, int N, int K,
                 int group, int sym, void *packed, w4a16_stream_t stream) {
  if (sym != kFormZero && sym != kFormSym) return W4A16_ERR_INVALID_ARG;
  if (!qweight || !scales || !packed || (!sym && !zeros)) return W4A16_ERR_INVALID_ARG;
  if (!sizes_ok(1, N, K, group)) return W4A16_ERR_INVALID_ARG;
  if (!aligned(packed, 256) || !aligned(qweight, 4) || !aligned(scales, 2) || (zeros && !aligned(zeros, 4)))
    return W4A16_ERR_MISALIGNED;
  DeviceInfo d;
  int st = current_device(d);
  if (st != W4A16_OK) return st;
  const Layout L = make_layout(N, K, group, sym);
  return finish_launch(launch_repack(qweight, scales, sym ? nullptr : zeros, nullptr, nullptr, nullptr, nullptr,
                                     nullptr, N, false, L, static_cast<uint8_t *>(packed),
                                     reinterpret_cast<cudaStream_t>(stream)));
}

int w4a16_repack_affine(const int32_t *qweight, const uint16_t *scales, const uint16_t *biases, int N, int K,
                        int group, void *packed, w4a16_stream_t stream) {
  if (!qweight || !scales || !biases || !packed) return W4A16_ERR_INVALID_ARG;
  if (!sizes_ok(1, N, K, group)) return W4A16_ERR_INVALID_ARG;
  if (!aligned(packed, 256) || !aligned(qweight, 4) || !aligned(scales, 2) || !aligned(biases, 2))
    return W4A16_ERR_MISALIGNED;
  DeviceInfo d;
  int st = current_device(d);
  if (st != W4A16_OK) return st;
  const Layout L = make_layout(N, K, group, kFormAffine);
  return finish_launch(launch_repack(qweight, scales, nullptr, biases, nullptr, nullptr, nullptr, nullptr, N,
                                     false, L, static_cast<uint8_t *>(packed),
                                     reinterpret_cast<cudaStream_t>(stream)));
}

int w4a16_repack_affine_gateup(const int32_t *qw_gate, const uint16_t *sc_gate, const uint16_t *b_gate,
                               const int32_t *qw_up, const uint16_t *sc_up, const uint16_t *b_up, int N_each,
                               int K, int group, void *packed, w4a16_stream_t stream) {
  if (!qw_gate || !sc_gate || !b_gate || !qw_up || !sc_up || !b_up || !packed) return W4A16_ERR_INVALID_ARG;
  if (w4a16_gateup_repacked_bytes(N_each, K, group, kFormAffine) == 0) return W4A16_ERR_INVALID_ARG;
  if (!aligned(packed, 256) || !aligned(qw_gate, 4) || !aligned(qw_up, 4) || !aligned(sc_gate, 2) ||
      !aligned(sc_up, 2) || !aligned(b_gate, 2) || !aligned(b_up, 2))
    return W4A16_ERR_MISALIGNED;
  DeviceInfo d;
  int st = current_device(d);
  if (st != W4A16_OK) return st;
  const Layout L = make_layout((int)gateup_rows(N_each), K, group, kFormAffine);
  return finish_launch(launch_repack(qw_gate, sc_gate, nullptr, b_gate, qw_up, sc_up, nullptr, b_up, N_each, true,
                                     L, static_cast<uint8_t *>(packed), reinterpret_cast<cudaStream_t>(stream)));
}

int w4a16_repack_gateup(const int32_t *qw_gate, const uint16_t *sc_gate, const int32_t *z_gate,
                        const int32_t *qw_up, const uint16_t *sc_up, const int32_t *z_up, int N_each, int K,
                        int group, int sym, void *packed, w4a16_stream_t stream) {
  if (sym != kFormZero && sym != kFormSym) return W4A16_ERR_INVALID_ARG;
  if (!qw_gate || !sc_gate || !qw_up || !sc_up || !packed) return W4A16_ERR_INVALID_ARG;
  if (!sym && (!z_gate || !z_up)) return W4A16_ERR_INVALID_ARG;
  if (w4a16_gateup_repacked_bytes(N_each, K, group, sym) == 0) return W4A16_ERR_INVALID_ARG;
  if (!aligned(packed, 256) || !aligned(qw_gate, 4) || !aligned(qw_up, 4) || !aligned(sc_gate, 2) ||
      !aligned(sc_up, 2) || (z_gate && !aligned(z_gate, 4)) || (z_up && !aligned(z_up, 4)))
    return W4A16_ERR_MISALIGNED;
  DeviceInfo d;
  int st = current_device(d);
  if (st != W4A16_OK) return st;
  const Layout L = make_layout((int)gateup_rows(N_each), K, group, sym);
  return finish_launch(launch_repack(qw_gate, sc_gate, sym ? nullptr : z_gate, nullptr, qw_up, sc_up,
                                     sym ? nullptr : z_up, nullptr, N_each, true, L,
                                     static_cast<uint8_t *>(packed), reinterpret_cast<cudaStream_t>(stream)));
}

int w4a16_gemm(const uint16_t *x, const void *packed, const uint16_t *scales, const int32_t *zeros, int M,
               int N, int K, int group, int sym, uint16_t *y, w4a16_stream_t stream) {
  const int ov = g_override.load();
  if (!x || !packed || !y) return W4A16_ERR_INVALID_ARG;
  if (scales || zeros) return W4A16_ERR_INVALID_ARG;  // reserved: they travel inside `packed`
  if (!sizes_ok(M, N, K, group) || !zero_form(sym)) return W4A16_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 16) || !aligned(packed, 256)) return W4A16_ERR_MISALIGNED;
  DeviceInfo d;
  int st = current_device(d);
  if (st != W4A16_OK) return st;
  GemmCall c{x, static_cast<const uint8_t *>(packed), y, M, N, K, group, sym, false,
             reinterpret_cast<cudaStream_t>(stream), d.err, d.device, g_overlap.load() != 0};
  // M <= 32: a tensor-core decode kernel (measured faster than the CUDA-core
  // GEMV at M = 1 on every decode shape); the GEMV stays selectable.
  if (M == 1 && ov == 1) return finish_launch(launch_gemv_m1(c, d.sm_count));
  if (ov == 5 && smallm_tc_supports(c)) return finish_launch(launch_smallm_tc(c, d.sm_count));
  if (use_decode(M, ov)) return finish_launch(launch_decode_kernel(c, d.sm_count, ov));
  return finish_launch(launch_prompt_tc(c, d.sm_count));
}

int w4a16_gateup_silu(const uint16_t *x, const void *packed_gateup, int M, int N_each, int K, int group,
                      int sym, uint16_t *h, w4a16_stream_t stream) {
  const int ov = g_override.load();
  if (!x || !packed_gateup || !h) return W4A16_ERR_INVALID_ARG;
  if (!sizes_ok(M, N_each, K, group) || !zero_form(sym) || w4a16_gateup_repacked_bytes(N_each, K, group, sym) == 0)
    return W4A16_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(h, 16) || !aligned(packed_gateup, 256)) return W4A16_ERR_MISALIGNED;
  DeviceInfo d;
  int st = current_device(d);
  if (st != W4A16_OK) return st;
  GemmCall c{x, static_cast<const uint8_t *>(packed_gateup), h, M, N_each, K, group, sym, true,
             reinterpret_cast<cudaStream_t>(stream), d.err, d.device, g_overlap.load() != 0};
  if (use_decode(M, ov)) return finish_launch(launch_decode_kernel(c, d.sm_count, ov));
  return finish_launch(launch_prompt_tc(c, d.sm_count));
}

int w4a16_gemm_argmax(const uint16_t *x, const void *packed, int M, int N, int K, int group, int sym,
                      uint16_t *y, int64_t *argmax, w4a16_stream_t stream) {
  const int ov = g_override.load();
  const bool decode = use_decode(M, ov);
  if (!x || !packed || !argmax) return W4A16_ERR_INVALID_ARG;
  if (!sizes_ok(M, N, K, group) || !zero_form(sym) || (!decode && !y)) return W4A16_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 16) || !aligned(packed, 256) || !aligned(argmax, 8))
    return W4A16_ERR_MISALIGNED;
  DeviceInfo d;
  int st = current_device(d);
  if (st != W4A16_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool overlap = g_overlap.load() != 0;
  cudaError_t e = launch_argmax_init(argmax, M, overlap, s);
  if (e != cudaSuccess) return cuda_fail(e);
  GemmCall c{x, static_cast<const uint8_t *>(packed), y, M, N, K, group, sym, false, s, d.err, d.device, overlap};
  if (decode) {
    c.amax = argmax;  // keys from the decode kernel's epilogue; y may be NULL
    e = launch_decode_kernel(c, d.sm_count, ov);
  } else {
    e = launch_prompt_tc(c, d.sm_count);
    if (e == cudaSuccess) e = launch_row_argmax(y, M, N, argmax, s);
  }
  if (e == cudaSuccess) e = launch_argmax_finalize(argmax, M, overlap, s);
  return finish_launch(e);
}

int w4a16_topk(const uint16_t *y, int M, int N, int k, int64_t *idx, uint16_t *vals, w4a16_stream_t stream) {
  if (!y || !idx) return W4A16_ERR_INVALID_ARG;
  if (!sizes_ok(M, N, 64, 64) || k < 1 || k > N || k > kTopkMaxK) return W4A16_ERR_INVALID_ARG;
  if (!aligned(y, 2) || !aligned(idx, 8) || !aligned(vals, 2)) return W4A16_ERR_MISALIGNED;
  DeviceInfo d;
  int st = current_device(d);
  if (st != W4A16_OK) return st;
  return finish_launch(launch_topk(y, M, N, k, idx, vals, g_overlap.load() != 0, d.device,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

int w4a16_gemm_topk(const uint16_t *x, const void *packed, int M, int N, int K, int group, int sym, int k,
                    uint16_t *y, int64_t *idx, uint16_t *vals, w4a16_stream_t stream) {
  if (k < 1 || k > N || k > kTopkMaxK || !idx) return W4A16_ERR_INVALID_ARG;
  if (!aligned(idx, 8) || !aligned(vals, 2)) return W4A16_ERR_MISALIGNED;
  const int st = w4a16_gemm(x, packed, nullptr, nullptr, M, N, K, group, sym, y, stream);
  if (st != W4A16_OK) return st;
  return w4a16_topk(y, M, N, k, idx, vals, stream);
}

size_t w4a16_xsum_bytes(int M, int K, int group) {
  if (!sizes_ok(M, 1, K, group)) return 0;
  return (size_t)M * (size_t)affine_kb3(K / group) * sizeof(uint16_t);
}

int w4a16_xsum(const uint16_t *x, int M, int K, int group, uint16_t *xsum, w4a16_stream_t stream) {
  if (!x || !xsum) return W4A16_ERR_INVALID_ARG;
  if (!sizes_ok(M, 1, K, group)) return W4A16_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(xsum, 16)) return W4A16_ERR_MISALIGNED;
  DeviceInfo d;
  int st = current_device(d);
  if (st != W4A16_OK) return st;
  return finish_launch(launch_xsum(x, M, K, group, xsum, reinterpret_cast<cudaStream_t>(stream)));
}

int w4a16_gemm_affine(const uint16_t *x, const uint16_t *xsum, const void *packed, int M, int N, int K, int group,
                      uint16_t *y, w4a16_stream_t stream) {
  const int ov = g_override.load();
  if (!x || !packed || !y || (!xsum && affine_uses_tc(M, ov))) return W4A16_ERR_INVALID_ARG;
  if (!sizes_ok(M, N, K, group)) return W4A16_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 16) || !aligned(packed, 256) || !aligned(xsum, 16))
    return W4A16_ERR_MISALIGNED;
  DeviceInfo d;
  int st = current_device(d);
  if (st != W4A16_OK) return st;
  GemmCall c{x, static_cast<const uint8_t *>(packed), y, M, N, K, group, kFormAffine, false,
             reinterpret_cast<cudaStream_t>(stream), d.err, d.device, g_overlap.load() != 0};
  return launch_affine(c, xsum, d, ov);
}

int w4a16_gemm_affine_noalloc(const uint16_t *x, const void *packed, int M, int N, int K, int group, uint16_t *y,
                              w4a16_stream_t stream) {
  const int ov = g_override.load();
  if (!x || !packed || !y) return W4A16_ERR_INVALID_ARG;
  if (!sizes_ok(M, N, K, group)) return W4A16_ERR_INVALID_ARG;
  const bool tc = affine_uses_tc(M, ov);
  if (tc && w4a16_xsum_bytes(M, K, group) > kNoAllocXsumBytes) return W4A16_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 16) || !aligned(packed, 256)) return W4A16_ERR_MISALIGNED;
  DeviceInfo d;
  int st = current_device(d);
  if (st != W4A16_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  GemmCall c{x, static_cast<const uint8_t *>(packed), y, M, N, K, group, kFormAffine, false, s, d.err, d.device,
             g_overlap.load() != 0};
  if (!tc) return launch_affine(c, nullptr, d, ov);
  // every entry the GEMM reads (padding included) is written by this pre-pass
  cudaError_t e = launch_xsum(x, M, K, group, d.noalloc_xsum, s);
  if (e != cudaSuccess) return cuda_fail(e);
  return launch_affine(c, d.noalloc_xsum, d, ov);
}

size_t w4a16_affine_bits_repacked_bytes(int N, int K, int group, int bits) {
  if (!bits_ok(bits) || !sizes_ok(1, N, K, group)) return 0;
  const long long Kp = (long long)K * bits_planes(bits);
  if (!sizes_ok(1, N, Kp, group)) return 0;
  return make_layout(N, (int)Kp, group, kFormAffine).total;
}

size_t w4a16_affine_bits_scratch_bytes(int M, int K, int group, int bits) {
  if (!bits_ok(bits) || !sizes_ok(M, 1, K, group)) return 0;
  const long long Kp = (long long)K * bits_planes(bits);
  if (!sizes_ok(M, 1, Kp, group)) return 0;
  return widened_x_bytes(M, K, bits) + (size_t)M * (size_t)affine_kb3((int)(Kp / group)) * sizeof(uint16_t);
}

int w4a16_repack_affine_bits(const uint32_t *qweight, const uint16_t *scales, const uint16_t *biases, int N, int K,
                             int group, int bits, void *packed, w4a16_stream_t stream) {
  if (!qweight || !scales || !biases || !packed) return W4A16_ERR_INVALID_ARG;
  if (w4a16_affine_bits_repacked_bytes(N, K, group, bits) == 0) return W4A16_ERR_INVALID_ARG;
  if (!aligned(packed, 256) || !aligned(qweight, 4) || !aligned(scales, 2) || !aligned(biases, 2))
    return W4A16_ERR_MISALIGNED;
  DeviceInfo d;
  int st = current_device(d);
  if (st != W4A16_OK) return st;
  const Layout L = make_layout(N, K * bits_planes(bits), group, kFormAffine);
  return finish_launch(launch_repack_affine_bits(reinterpret_cast<const uint32_t *>(qweight), scales, biases, N, K,
                                                 bits, L, static_cast<uint8_t *>(packed),
                                                 reinterpret_cast<cudaStream_t>(stream)));
}

int w4a16_gemm_affine_bits(const uint16_t *x, void *scratch, const void *packed, int M, int N, int K, int group,
                           int bits, uint16_t *y, w4a16_stream_t stream) {
  const int ov = g_override.load();
  if (!x || !scratch || !packed || !y) return W4A16_ERR_INVALID_ARG;
  if (!sizes_ok(M, N, K, group) || w4a16_affine_bits_scratch_bytes(M, K, group, bits) == 0 ||
      w4a16_affine_bits_repacked_bytes(N, K, group, bits) == 0)
    return W4A16_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 16) || !aligned(packed, 256) || !aligned(scratch, 256))
    return W4A16_ERR_MISALIGNED;
  DeviceInfo d;
  int st = current_device(d);
  if (st != W4A16_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t *scr = static_cast<uint8_t *>(scratch);
  const uint16_t *xin = x;
  if (bits > 4) {
    uint16_t *xw = reinterpret_cast<uint16_t *>(scr);
    cudaError_t e = launch_widen_groups(x, M, K, group, xw, s);
    if (e != cudaSuccess) return cuda_fail(e);
    xin = xw;
  }
  const int Kp = K * bits_planes(bits);
  GemmCall c{xin, static_cast<const uint8_t *>(packed), y, M, N, Kp, group, kFormAffine, false, s, d.err, d.device,
             g_overlap.load() != 0};
  if (!affine_uses_tc(M, ov)) return launch_affine(c, nullptr, d, ov);
  uint16_t *xs = reinterpret_cast<uint16_t *>(scr + widened_x_bytes(M, K, bits));
  cudaError_t e = launch_xsum(xin, M, Kp, group, xs, s);
  if (e != cudaSuccess) return cuda_fail(e);
  return launch_affine(c, xs, d, ov);
}

int w4a16_dequantize_affine_bits(const void *packed, int N, int K, int group, int bits, float *w_out,
                                 w4a16_stream_t stream) {
  if (!packed || !w_out) return W4A16_ERR_INVALID_ARG;
  if (w4a16_affine_bits_repacked_bytes(N, K, group, bits) == 0) return W4A16_ERR_INVALID_ARG;
  if (!aligned(packed, 256) || !aligned(w_out, 16)) return W4A16_ERR_MISALIGNED;
  DeviceInfo d;
  int st = current_device(d);
  if (st != W4A16_OK) return st;
  const Layout L = make_layout(N, K * bits_planes(bits), group, kFormAffine);
  return finish_launch(launch_dequantize_affine_bits(static_cast<const uint8_t *>(packed), L, N, K, bits, w_out,
                                                     reinterpret_cast<cudaStream_t>(stream)));
}

int w4a16_gateup_silu_affine(const uint16_t *x, const uint16_t *xsum, const void *packed_gateup, int M, int N_each,
                             int K, int group, uint16_t *h, w4a16_stream_t stream) {
  const int ov = g_override.load();
  if (!x || !packed_gateup || !h || (!xsum && affine_uses_tc(M, ov))) return W4A16_ERR_INVALID_ARG;
  if (!sizes_ok(M, N_each, K, group) || w4a16_gateup_repacked_bytes(N_each, K, group, kFormAffine) == 0)
    return W4A16_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(h, 16) || !aligned(packed_gateup, 256) || !aligned(xsum, 16))
    return W4A16_ERR_MISALIGNED;
  DeviceInfo d;
  int st = current_device(d);
  if (st != W4A16_OK) return st;
  GemmCall c{x, static_cast<const uint8_t *>(packed_gateup), h, M, N_each, K, group, kFormAffine, true,
             reinterpret_cast<cudaStream_t>(stream), d.err, d.device, g_overlap.load() != 0};
  return launch_affine(c, xsum, d, ov);
}

int w4a16_dequantize(const void *packed, int N, int K, int group, int sym, float *w_out,
                     w4a16_stream_t stream) {
  if (!packed || !w_out) return W4A16_ERR_INVALID_ARG;
  if (!sizes_ok(1, N, K, group) || !form_ok(sym)) return W4A16_ERR_INVALID_ARG;
  if (!aligned(packed, 256) || !aligned(w_out, 16)) return W4A16_ERR_MISALIGNED;
  DeviceInfo d;
  int st = current_device(d);
  if (st != W4A16_OK) return st;
  const Layout L = make_layout(N, K, group, sym);
  return finish_launch(launch_dequantize(static_cast<const uint8_t *>(packed), L, N, w_out,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

int w4a16_kernel_status(void) {
  DeviceInfo d;
  int st = current_device(d);
  if (st != W4A16_OK) return st;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e);
  int v = 0;
  if ((e = cudaMemcpyFromSymbol(&v, g_kernel_error, sizeof(int))) != cudaSuccess) return cuda_fail(e);
  if (v != 0) {
    const int zero = 0;
    if ((e = cudaMemcpyToSymbol(g_kernel_error, &zero, sizeof(int))) != cudaSuccess) return cuda_fail(e);
    return W4A16_ERR_TIMEOUT;
  }
  return W4A16_OK;
}

const char *w4a16_strerror(int status) {
  switch (status) {
    case W4A16_OK: return "ok";
    case W4A16_ERR_INVALID_ARG: return "invalid argument (size, group, null pointer or reserved argument)";
    case W4A16_ERR_MISALIGNED: return "misaligned pointer (x, y, h need 16 bytes; packed needs 256)";
    case W4A16_ERR_UNSUPPORTED: return "unsupported device (built for sm_103a)";
    case W4A16_ERR_CUDA: return "CUDA error (see w4a16_last_cuda_error)";
    case W4A16_ERR_TIMEOUT: return "a bounded wait inside a kernel gave up";
    default: return "unknown status";
  }
}

int w4a16_last_cuda_error(void) { return t_last_cuda_error; }

int w4a16_set_kernel_override(int which) {
  if (which < 0 || which > 5) return -1;
  return g_override.exchange(which);
}

int w4a16_set_programmatic_overlap(int on) {
  if (on != 0 && on != 1) return -1;
  return g_overlap.exchange(on);
}

}  // extern "C"
