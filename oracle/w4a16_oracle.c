/*
 * CPU oracle for the group-quantized INT4-weight x bf16-activation matmul.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference leg may load or call this library.
 * It shares no code, header, table or constant with the CUDA library.
 *
 * What it computes (written out as the plain definition, in float64):
 *
 *   q[n][k] = bits 4(k%8)..4(k%8)+3 of qweight[n][k/8]         (4-bit code)
 *   z[n][g] = 8 when symmetric, else nibble g%8 of zeros[n][g/8]
 *   w[n][k] = (q[n][k] - z[n][k/G]) * scale[n][k/G]
 *   y[m][n] = sum_k x[m][k] * w[n][k]          (k ascending, float64)
 *   h[m][n] = SiLU(g) * u,  g = y_gate[m][n],  u = y_up[m][n],  SiLU(v) = v / (1 + exp(-v))
 *
 * Affine form (the *_affine functions): w[n][k] = scale[n][k/G] * q[n][k] +
 * bias[n][k/G], q the unsigned 4-bit code and scale, bias bf16 per (row,
 * group); the MLX affine 4-bit checkpoints of TensorFold PR #859 ("What this
 * changes": every code keeps its value, scale and bias; groups of 64).
 *
 * Sources: the exact "(q - z) * scale" dequantisation of the INT4 decode
 * kernels (GRIMOIRE v1.7 release notes, "What changed"); symmetric GPTQ-Int4
 * at group 128 and AutoRound W4A16 at group 64 (same page, measurement
 * table); the output layer over all verify rows and the prompt path "with the
 * feed-forward gate fused in" (GRIMOIRE v1.8 release notes, "What changed",
 * "INT4 verify faster" and "INT4 prompt processing"). SiLU(gate) * up is the
 * plainest reading of a fused feed-forward gate.
 *
 * Every sum also returns sum_k |x[m][k] * w[n][k]|, the magnitude the error
 * bound of a float32-accumulating kernel is stated against.
 *
 * Parallelism: output rows n are independent, so they are spread over threads
 * with OpenMP when it is available; no sum is split or reordered.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 bit pattern -> exact float64 value */
static double bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* 4-bit code of weight (n, k) in the canonical packing */
int oracle_code(const int32_t *qweight, int K, int n, int k) {
  uint32_t word = (uint32_t)qweight[(size_t)n * (size_t)(K / 8) + (size_t)(k / 8)];
  return (int)((word >> (4 * (k % 8))) & 0xFu);
}

/* zero point of (row n, group g); 8 when symmetric */
int oracle_zero(const int32_t *zeros, int Kg, int sym, int n, int g) {
  if (sym) return 8;
  int words = (Kg + 7) / 8;
  uint32_t word = (uint32_t)zeros[(size_t)n * (size_t)words + (size_t)(g / 8)];
  return (int)((word >> (4 * (g % 8))) & 0xFu);
}

/* w[n][k] = (q - z) * scale, exact in float64 */
double oracle_weight(const int32_t *qweight, const uint16_t *scales, const int32_t *zeros,
                     int K, int G, int sym, int n, int k) {
  int Kg = K / G;
  int g = k / G;
  int q = oracle_code(qweight, K, n, k);
  int z = oracle_zero(zeros, Kg, sym, n, g);
  return (double)(q - z) * bf16_value(scales[(size_t)n * (size_t)Kg + (size_t)g]);
}

/* w[n][k] = scale * q + bias, exact in float64 (a 12-bit product plus a bf16) */
double oracle_weight_affine(const int32_t *qweight, const uint16_t *scales, const uint16_t *biases,
                            int K, int G, int n, int k) {
  int Kg = K / G;
  int g = k / G;
  int q = oracle_code(qweight, K, n, k);
  size_t i = (size_t)n * (size_t)Kg + (size_t)g;
  return bf16_value(scales[i]) * (double)q + bf16_value(biases[i]);
}

/* Affine dequantised weight matrix, float64 [N][K]. */
void oracle_dequant_affine(const int32_t *qweight, const uint16_t *scales, const uint16_t *biases,
                           int N, int K, int G, double *w) {
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < K; ++k)
      w[(size_t)n * K + k] = oracle_weight_affine(qweight, scales, biases, K, G, n, k);
}

/* Dequantised weight matrix, float64 [N][K]. */
void oracle_dequant(const int32_t *qweight, const uint16_t *scales, const int32_t *zeros,
                    int N, int K, int G, int sym, double *w) {
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < K; ++k)
      w[(size_t)n * K + k] = oracle_weight(qweight, scales, zeros, K, G, sym, n, k);
}

/* One output: y = sum_k x[m][k] * w[n][k], and sum_k |x[m][k] * w[n][k]|. */
static void dot_one(const uint16_t *x, const double *wrow, int K, int m, double *y, double *a) {
  double s = 0.0, sa = 0.0;
  const uint16_t *xr = x + (size_t)m * K;
  for (int k = 0; k < K; ++k) {
    double p = bf16_value(xr[k]) * wrow[k];
    s += p;
    sa += fabs(p);
  }
  *y = s;
  *a = sa;
}

/* One weight row; biases != NULL selects the affine form (zeros, sym unused). */
static void weight_row(const int32_t *qweight, const uint16_t *scales, const int32_t *zeros,
                       const uint16_t *biases, int K, int G, int sym, int n, double *wrow) {
  for (int k = 0; k < K; ++k)
    wrow[k] = biases ? oracle_weight_affine(qweight, scales, biases, K, G, n, k)
                     : oracle_weight(qweight, scales, zeros, K, G, sym, n, k);
}

static int pick_threads(int nthreads) {
#ifdef _OPENMP
  return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
  (void)nthreads;
  return 1;
#endif
}

/* Threads the library would use for nthreads (0 = all). */
int oracle_threads(int nthreads) { return pick_threads(nthreads); }

static int gemm_all(const uint16_t *x, const int32_t *qweight, const uint16_t *scales,
                    const int32_t *zeros, const uint16_t *biases, int M, int N, int K, int G, int sym,
                    double *y, double *ysum_abs, int nthreads) {
  if (M < 0 || N < 0 || K <= 0 || G <= 0 || K % G || K % 8) return -1;
  int bad = 0;
  int nt = pick_threads(nthreads);
#pragma omp parallel num_threads(nt)
  {
    double *wrow = (double *)malloc(sizeof(double) * (size_t)K);
    if (!wrow) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(dynamic, 8)
      for (int n = 0; n < N; ++n) {
        weight_row(qweight, scales, zeros, biases, K, G, sym, n, wrow);
        for (int m = 0; m < M; ++m)
          dot_one(x, wrow, K, m, &y[(size_t)m * N + n], &ysum_abs[(size_t)m * N + n]);
      }
      free(wrow);
    }
  }
  return bad ? -1 : 0;
}

static int gemm_some(const uint16_t *x, const int32_t *qweight, const uint16_t *scales,
                     const int32_t *zeros, const uint16_t *biases, int M, int N, int K, int G, int sym,
                     const int64_t *m_idx, const int64_t *n_idx, int64_t count,
                     double *y, double *ysum_abs, int nthreads) {
  if (M < 0 || N < 0 || K <= 0 || G <= 0 || K % G || K % 8) return -1;
  for (int64_t i = 0; i < count; ++i)
    if (m_idx[i] < 0 || m_idx[i] >= M || n_idx[i] < 0 || n_idx[i] >= N) return -1;
  int bad = 0;
  int nt = pick_threads(nthreads);
#pragma omp parallel num_threads(nt)
  {
    double *wrow = (double *)malloc(sizeof(double) * (size_t)K);
    if (!wrow) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(dynamic, 4)
      for (int64_t i = 0; i < count; ++i) {
        weight_row(qweight, scales, zeros, biases, K, G, sym, (int)n_idx[i], wrow);
        dot_one(x, wrow, K, (int)m_idx[i], &y[i], &ysum_abs[i]);
      }
      free(wrow);
    }
  }
  return bad ? -1 : 0;
}

/*
 * y[m][n] (float64 [M][N]) and ysum_abs[m][n] = sum_k |x w| for all outputs.
 * x: bf16 bits [M][K]; qweight int32 [N][K/8]; scales bf16 bits [N][K/G];
 * zeros int32 [N][ceil(K/G/8)] (ignored when sym). Returns 0, or -1 on bad sizes
 * or when memory runs out.
 */
int oracle_gemm(const uint16_t *x, const int32_t *qweight, const uint16_t *scales,
                const int32_t *zeros, int M, int N, int K, int G, int sym,
                double *y, double *ysum_abs, int nthreads) {
  return gemm_all(x, qweight, scales, zeros, NULL, M, N, K, G, sym, y, ysum_abs, nthreads);
}

/* Selected outputs one by one: y[i] = y(m_idx[i], n_idx[i]). */
int oracle_gemm_at(const uint16_t *x, const int32_t *qweight, const uint16_t *scales,
                   const int32_t *zeros, int M, int N, int K, int G, int sym,
                   const int64_t *m_idx, const int64_t *n_idx, int64_t count,
                   double *y, double *ysum_abs, int nthreads) {
  return gemm_some(x, qweight, scales, zeros, NULL, M, N, K, G, sym, m_idx, n_idx, count, y, ysum_abs,
                   nthreads);
}

/* The affine form of oracle_gemm: biases bf16 bits [N][K/G]. */
int oracle_gemm_affine(const uint16_t *x, const int32_t *qweight, const uint16_t *scales,
                       const uint16_t *biases, int M, int N, int K, int G,
                       double *y, double *ysum_abs, int nthreads) {
  if (!biases) return -1;
  return gemm_all(x, qweight, scales, NULL, biases, M, N, K, G, 0, y, ysum_abs, nthreads);
}

/* The affine form of oracle_gemm_at. */
int oracle_gemm_affine_at(const uint16_t *x, const int32_t *qweight, const uint16_t *scales,
                          const uint16_t *biases, int M, int N, int K, int G,
                          const int64_t *m_idx, const int64_t *n_idx, int64_t count,
                          double *y, double *ysum_abs, int nthreads) {
  if (!biases) return -1;
  return gemm_some(x, qweight, scales, NULL, biases, M, N, K, G, 0, m_idx, n_idx, count, y, ysum_abs,
                   nthreads);
}

/* Group sums of x (the X_g of the affine form's bias term), float64
 * [K/G][M]: xs[g][m] = sum_{k in g} x[m][k]. Returns 0, or -1 on bad sizes. */
int oracle_group_sums(const uint16_t *x, int M, int K, int G, double *xs) {
  if (M < 0 || K <= 0 || G <= 0 || K % G) return -1;
  for (int g = 0; g < K / G; ++g)
    for (int m = 0; m < M; ++m) {
      double acc = 0.0;
      for (int k = g * G; k < (g + 1) * G; ++k) acc += bf16_value(x[(size_t)m * K + k]);
      xs[(size_t)g * M + m] = acc;
    }
  return 0;
}

/* SiLU(g) * u in float64 */
double oracle_silu_mul(double g, double u) { return g / (1.0 + exp(-g)) * u; }

/*
 * Fused feed-forward gate over selected outputs: for each i,
 *   g = y_gate(m, n), u = y_up(m, n), h = SiLU(g) * u,
 * returning h, g, u and the two magnitude sums. Gate and up weights are two
 * canonical weights of the same shape [N][K].
 */
int oracle_gateup_silu_at(const uint16_t *x,
                          const int32_t *qw_gate, const uint16_t *sc_gate, const int32_t *z_gate,
                          const int32_t *qw_up, const uint16_t *sc_up, const int32_t *z_up,
                          int M, int N, int K, int G, int sym,
                          const int64_t *m_idx, const int64_t *n_idx, int64_t count,
                          double *h, double *g, double *u, double *gsum_abs, double *usum_abs,
                          int nthreads) {
  if (oracle_gemm_at(x, qw_gate, sc_gate, z_gate, M, N, K, G, sym, m_idx, n_idx, count, g,
                     gsum_abs, nthreads))
    return -1;
  if (oracle_gemm_at(x, qw_up, sc_up, z_up, M, N, K, G, sym, m_idx, n_idx, count, u,
                     usum_abs, nthreads))
    return -1;
  for (int64_t i = 0; i < count; ++i) h[i] = oracle_silu_mul(g[i], u[i]);
  return 0;
}

/* The affine form of oracle_gateup_silu_at: b_gate, b_up bf16 biases [N][K/G]. */
int oracle_gateup_silu_affine_at(const uint16_t *x,
                                 const int32_t *qw_gate, const uint16_t *sc_gate, const uint16_t *b_gate,
                                 const int32_t *qw_up, const uint16_t *sc_up, const uint16_t *b_up,
                                 int M, int N, int K, int G,
                                 const int64_t *m_idx, const int64_t *n_idx, int64_t count,
                                 double *h, double *g, double *u, double *gsum_abs, double *usum_abs,
                                 int nthreads) {
  if (oracle_gemm_affine_at(x, qw_gate, sc_gate, b_gate, M, N, K, G, m_idx, n_idx, count, g, gsum_abs,
                            nthreads))
    return -1;
  if (oracle_gemm_affine_at(x, qw_up, sc_up, b_up, M, N, K, G, m_idx, n_idx, count, u, usum_abs, nthreads))
    return -1;
  for (int64_t i = 0; i < count; ++i) h[i] = oracle_silu_mul(g[i], u[i]);
  return 0;
}

/*
 * Affine form at other code widths: TensorFold PR #859 loads modules of 2 to
 * 8 bits, every code keeping its value, scale and bias ("What this changes";
 * the native 2, 3, 5 and 6-bit tiles note), so w = scale * q + bias with q in
 * 0 .. 2^bits - 1. The canonical layout is read as one little-endian bit
 * stream per row: the row's K codes fill ceil(K * bits / 32) uint32 words and
 * code k occupies bits [bits * k, bits * k + bits) of the stream, running
 * into the next word where it does not fit. At 4 bits this is the nibble
 * packing of oracle_code.
 */
static size_t row_words_bits(int K, int bits) { return ((size_t)K * (size_t)bits + 31) / 32; }

int oracle_code_bits(const uint32_t *qweight, int K, int bits, int n, int k) {
  const size_t words = row_words_bits(K, bits);
  const uint32_t *row = qweight + (size_t)n * words;
  const size_t bit = (size_t)k * (size_t)bits;
  const size_t w = bit / 32;
  uint64_t v = row[w];
  if (w + 1 < words) v |= (uint64_t)row[w + 1] << 32;
  return (int)((v >> (bit % 32)) & ((1u << bits) - 1u));
}

double oracle_weight_affine_bits(const uint32_t *qweight, const uint16_t *scales, const uint16_t *biases,
                                 int K, int G, int bits, int n, int k) {
  const size_t i = (size_t)n * (size_t)(K / G) + (size_t)(k / G);
  return bf16_value(scales[i]) * (double)oracle_code_bits(qweight, K, bits, n, k) + bf16_value(biases[i]);
}

static int bits_args_ok(int M, int N, int K, int G, int bits) {
  return M >= 0 && N >= 0 && K > 0 && G > 0 && K % G == 0 && bits >= 2 && bits <= 8;
}

/* float64 [N][K]: w = scale * q + bias of a bits-wide weight. Returns 0 or -1. */
int oracle_dequant_affine_bits(const uint32_t *qweight, const uint16_t *scales, const uint16_t *biases,
                               int N, int K, int G, int bits, double *w) {
  if (!bits_args_ok(0, N, K, G, bits)) return -1;
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < K; ++k)
      w[(size_t)n * K + k] = oracle_weight_affine_bits(qweight, scales, biases, K, G, bits, n, k);
  return 0;
}

/* y[m][n] and sum_k |x w| of a bits-wide affine weight, as oracle_gemm_affine. */
int oracle_gemm_affine_bits(const uint16_t *x, const uint32_t *qweight, const uint16_t *scales,
                            const uint16_t *biases, int M, int N, int K, int G, int bits,
                            double *y, double *ysum_abs, int nthreads) {
  if (!bits_args_ok(M, N, K, G, bits)) return -1;
  int bad = 0;
  int nt = pick_threads(nthreads);
#pragma omp parallel num_threads(nt)
  {
    double *wrow = (double *)malloc(sizeof(double) * (size_t)K);
    if (!wrow) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(dynamic, 8)
      for (int n = 0; n < N; ++n) {
        for (int k = 0; k < K; ++k) wrow[k] = oracle_weight_affine_bits(qweight, scales, biases, K, G, bits, n, k);
        for (int m = 0; m < M; ++m)
          dot_one(x, wrow, K, m, &y[(size_t)m * N + n], &ysum_abs[(size_t)m * N + n]);
      }
      free(wrow);
    }
  }
  return bad ? -1 : 0;
}
