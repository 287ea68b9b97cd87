"""The oracle's decode steps retyped in numpy, each with a switch that plants
one plausible mistake (test infrastructure for tests/test_oracle_mutants.py).

With no mistake every function here equals the C oracle bit for bit on the
dequantised weights (and the GEMMs within the float64 summation bound), which
the tests check first; so a mutant is the oracle with exactly one mistake, and
each pin that is meant to catch that mistake must reject it.

Mistakes:

  nibble_order_reversed   code k read from nibble 7 - k % 8 of its word
  transposed              w[k][n] used for w[n][k] (square weights)
  zero_word_stride_floor  zero-point words per row floor(K/G/8) instead of
                          ceil(K/G/8)
  zero_mask_3bit          zero points read with a 3-bit mask
  bias_group_off_by_one   the affine bias of group g + 1 used for group g
  straddle_next_word      a b-bit code that runs into the next uint32 word
                          loses its high bits
  nan_lowest              a NaN ranked below every number in the top-k order
  negzero_below_zero      -0 ranked below +0 in the top-k order
  dsilu_sign              SiLU'(g) = s (1 - g (1 - s))
  drop_bu, drop_bg,       one term of the fused gate/up bound left out
  drop_cross
"""
from __future__ import annotations

import numpy as np

import oracle
import synth


def _bf16(bits) -> np.ndarray:
    return synth.bf16_bits_to_f32(np.asarray(bits, dtype=np.uint16)).astype(np.float64)


def codes(qweight, N, K, mistake=None) -> np.ndarray:
    """int64 [N, K]: code k of row n is nibble k % 8 of word k / 8."""
    words = np.ascontiguousarray(qweight).view(np.uint32).reshape(N, K // 8).astype(np.int64)
    k = np.arange(K)
    nib = 7 - k % 8 if mistake == "nibble_order_reversed" else k % 8
    return (words[:, k // 8] >> (4 * nib)) & 0xF


def zero_points(zeros, N, Kg, sym, mistake=None) -> np.ndarray:
    """int64 [N, Kg]: 8 when symmetric, else nibble g % 8 of word g / 8 of the row."""
    if sym:
        return np.full((N, Kg), 8, dtype=np.int64)
    per_row = Kg // 8 if mistake == "zero_word_stride_floor" else (Kg + 7) // 8
    flat = np.ascontiguousarray(zeros).view(np.uint32).reshape(-1).astype(np.int64)
    g = np.arange(Kg)
    idx = np.arange(N)[:, None] * per_row + g[None, :] // 8
    mask = 0x7 if mistake == "zero_mask_3bit" else 0xF
    return (flat[idx] >> (4 * (g % 8))) & mask


def dequant(qweight, scales, zeros, N, K, G, sym, mistake=None) -> np.ndarray:
    """float64 [N, K]: (q - z) * scale."""
    Kg = K // G
    q = codes(qweight, N, K, mistake)
    z = zero_points(zeros, N, Kg, sym, mistake)
    s = _bf16(scales).reshape(N, Kg)
    gi = np.arange(K) // G
    w = (q - z[:, gi]).astype(np.float64) * s[:, gi]
    if mistake == "transposed":
        w = w.T.copy()
    return w


def dequant_affine(qweight, scales, biases, N, K, G, mistake=None) -> np.ndarray:
    """float64 [N, K]: scale * q + bias."""
    Kg = K // G
    q = codes(qweight, N, K, mistake).astype(np.float64)
    s = _bf16(scales).reshape(N, Kg)
    b = _bf16(biases).reshape(N, Kg)
    gi = np.arange(K) // G
    bi = np.minimum(gi + 1, Kg - 1) if mistake == "bias_group_off_by_one" else gi
    return s[:, gi] * q + b[:, bi]


def codes_bits(qweight, N, K, bits, mistake=None) -> np.ndarray:
    """int64 [N, K] of a b-bit weight: code k at bits [b k, b k + b) of the
    row's little-endian bit stream."""
    words = (K * bits + 31) // 32
    row = np.ascontiguousarray(qweight).view(np.uint32).reshape(N, words).astype(np.uint64)
    bit = np.arange(K, dtype=np.int64) * bits
    w = bit // 32
    lo = row[:, w]
    nxt = np.minimum(w + 1, words - 1)
    hi = np.where((w + 1 < words)[None, :], row[:, nxt], 0).astype(np.uint64)
    if mistake == "straddle_next_word":
        hi = np.zeros_like(hi)
    v = lo | (hi << np.uint64(32))
    return ((v >> (bit % 32).astype(np.uint64)) & np.uint64((1 << bits) - 1)).astype(np.int64)


def dequant_affine_bits(qweight, scales, biases, N, K, G, bits, mistake=None) -> np.ndarray:
    Kg = K // G
    q = codes_bits(qweight, N, K, bits, mistake).astype(np.float64)
    s = _bf16(scales).reshape(N, Kg)
    b = _bf16(biases).reshape(N, Kg)
    gi = np.arange(K) // G
    return s[:, gi] * q + b[:, gi]


def gemm_from_weights(x, w):
    """(y, sum|x w|) float64 [M, N] from a dequantised weight [N, K]."""
    xf = _bf16(x)
    return xf @ w.T, np.abs(xf) @ np.abs(w).T


def bf16_rank(bits, mistake=None) -> np.ndarray:
    """Order key of bf16 patterns: sign-magnitude as a signed integer, -0 = +0,
    NaN one step above +inf."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    mag = b & 0x7FFF
    key = np.where(b & 0x8000, -mag, mag)
    if mistake == "negzero_below_zero":
        key = np.where(b == 0x8000, -1, key)
    nan = mag > 0x7F80
    if mistake == "nan_lowest":
        return np.where(nan, -0x7F81, key)
    return np.where(nan, 0x7F81, key)


def topk(y_bits, k, mistake=None):
    """(indices, value bits) of the k largest of every row, ties by column."""
    y = np.atleast_2d(np.asarray(y_bits, dtype=np.uint16))
    order = np.argsort(-bf16_rank(y, mistake), axis=1, kind="stable")[:, :k]
    return order.astype(np.int64), np.take_along_axis(y, order, axis=1)


def dsilu(g, mistake=None):
    s = oracle.sigmoid(g)
    g = np.asarray(g, dtype=np.float64)
    if mistake == "dsilu_sign":
        return s * (1.0 - g * (1.0 - s))
    return s * (1.0 + g * (1.0 - s))


def silu_bound(h_ref, g, u, gsum_abs, usum_abs, mistake=None):
    g = np.asarray(g, dtype=np.float64)
    u = np.asarray(u, dtype=np.float64)
    bg = oracle.ACC_TOL * np.asarray(gsum_abs)
    bu = oracle.ACC_TOL * np.asarray(usum_abs)
    t_g = np.abs(dsilu(g, mistake)) * np.abs(u) * bg
    t_u = np.abs(g * oracle.sigmoid(g)) * bu
    t_x = bg * bu
    if mistake == "drop_bg":
        t_g = 0.0 * t_g
    if mistake == "drop_bu":
        t_u = 0.0 * t_u
    if mistake == "drop_cross":
        t_x = 0.0 * t_x
    return oracle.REL_TOL * np.abs(h_ref) + t_g + t_u + t_x
