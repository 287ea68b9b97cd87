"""Seeded synthetic inputs for the W4A16 group-quantized matmul.

This module builds the inputs that both the CPU oracle and the CUDA path
consume: packed 4-bit codes, bf16 group scales, packed 4-bit zero points and
bf16 activations, all in the canonical layout

    qweight int32 [N, K/8]     nibble j (bits 4j..4j+3) of word c holds k = 8c + j
    scales  bf16  [N, K/G]     one scale per (output row, K-group)
    zeros   int32 [N, ceil(K/G/8)]  nibble j of word c holds group 8c + j
    biases  bf16  [N, K/G]     one bias per (output row, K-group), affine form only

It holds no part of the method's arithmetic (no dequantisation, no products,
no sums): only random-number generation, rounding of the sampled reals to
bf16 and bit packing of the sampled integers.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014), one stream per tensor; uniform reals from
the top 53 bits; normals by the Box-Muller transform (cosine branch); codes
from the top 4 bits.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "splitmix64_stream", "uniform01", "normal01", "f32_to_bf16_bits",
    "bf16_bits_to_f32", "pack_nibbles_rows", "make_codes", "make_qweight",
    "make_scales", "make_zeros", "make_biases", "make_x", "make_problem", "TENSOR_IDS",
    "SCALE_SWEEP", "exhaustive_problem", "planted_max_problem", "pack_bits_rows", "make_codes_bits",
]

def _signed(c: int) -> np.int64:
    return np.int64(c - (1 << 64) if c >= (1 << 63) else c)


# multiplications run on int64 views: two's-complement wrap-around is the same
# modulo-2^64 product, and numpy's int64 multiply is far faster than uint64's
_GAMMA = _signed(0x9E3779B97F4A7C15)
_M1 = _signed(0xBF58476D1CE4E5B9)
_M2 = _signed(0x94D049BB133111EB)

# stream id of every tensor a problem draws
TENSOR_IDS = {"x": 1, "qweight": 2, "scales": 3, "zeros": 4,
              "qweight_up": 5, "scales_up": 6, "zeros_up": 7, "biases": 8, "biases_up": 9, "x_signs": 10}


_BLOCK = 1 << 20  # draws per in-place block (reused buffers keep page faults down)


def _mix_inplace(z: np.ndarray, tmp: np.ndarray) -> None:
    """SplitMix64 output function applied in place to a uint64 array."""
    zi = z.view(np.int64)
    np.right_shift(z, np.uint64(30), out=tmp)
    np.bitwise_xor(z, tmp, out=z)
    np.multiply(zi, _M1, out=zi)
    np.right_shift(z, np.uint64(27), out=tmp)
    np.bitwise_xor(z, tmp, out=z)
    np.multiply(zi, _M2, out=zi)
    np.right_shift(z, np.uint64(31), out=tmp)
    np.bitwise_xor(z, tmp, out=z)


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function on uint64 values (array in, uint64 array out)."""
    z = np.array(z, dtype=np.uint64, copy=True)
    _mix_inplace(z, np.empty_like(z))
    return z


def splitmix64_stream(state0: int, n: int, offset: int = 0) -> np.ndarray:
    """Outputs offset+1 .. offset+n of SplitMix64 started at ``state0``.

    Output i (1-based) is mix(state0 + i * gamma) modulo 2^64.
    """
    out = np.empty(n, dtype=np.uint64)
    s0 = _signed(state0 & 0xFFFFFFFFFFFFFFFF)
    step = min(n, _BLOCK) if n else 0
    idx = np.empty(step, dtype=np.int64)
    tmp = np.empty(step, dtype=np.uint64)
    with np.errstate(over="ignore"):
        for b0 in range(0, n, _BLOCK):
            b1 = min(n, b0 + _BLOCK)
            m = b1 - b0
            zi = out[b0:b1].view(np.int64)
            np.copyto(idx[:m], np.arange(offset + 1 + b0, offset + 1 + b1, dtype=np.int64))
            np.multiply(idx[:m], _GAMMA, out=zi)
            np.add(zi, s0, out=zi)
            _mix_inplace(out[b0:b1], tmp[:m])
    return out


def _stream_state(seed: int, tensor_id: int) -> int:
    with np.errstate(over="ignore"):
        a = _mix(np.array([seed & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64))[0]
        b = _mix(np.array([(tensor_id + 1) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64))[0]
        return int(a ^ b)


def uniform01(bits: np.ndarray) -> np.ndarray:
    """[0, 1) reals in float64 from the top 53 bits of each draw."""
    return (bits >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal01(bits_a: np.ndarray, bits_b: np.ndarray) -> np.ndarray:
    """Standard normals (Box-Muller, cosine branch) in float64."""
    u1 = ((bits_a >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)  # (0, 1]
    u2 = (bits_b >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def f32_to_bf16_bits(a) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); uint16 bits."""
    f = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    bias = np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    r = ((u + bias) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(f)
    if nan.any():
        r = np.where(nan, np.uint16(0x7FC0), r)
    return r


def bf16_bits_to_f32(b) -> np.ndarray:
    b = np.ascontiguousarray(np.asarray(b, dtype=np.uint16))
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def pack_nibbles_rows(vals: np.ndarray) -> np.ndarray:
    """Pack a [R, C] array of 0..15 integers into int32 [R, ceil(C/8)], nibble j of word c = column 8c+j.

    Columns past C in the last word are zero.
    """
    vals = np.asarray(vals, dtype=np.uint32)
    R, C = vals.shape
    W = (C + 7) // 8
    padded = np.zeros((R, W * 8), dtype=np.uint32)
    padded[:, :C] = vals & np.uint32(0xF)
    padded = padded.reshape(R, W, 8)
    words = np.zeros((R, W), dtype=np.uint32)
    for j in range(8):
        words |= padded[:, :, j] << np.uint32(4 * j)
    return words.view(np.int32)



def pack_bits_rows(vals: np.ndarray, bits: int) -> np.ndarray:
    """Pack a [R, C] array of bits-wide integers into uint32 [R, ceil(C*bits/32)]:
    one little-endian bit stream per row, value c at bits [bits*c, bits*c + bits),
    running into the next word where it does not fit; unused high bits zero."""
    vals = np.asarray(vals, dtype=np.uint64) & np.uint64((1 << bits) - 1)
    R, C = vals.shape
    W = (C * bits + 31) // 32
    pos = np.arange(C, dtype=np.uint64) * np.uint64(bits)
    word, shift = (pos // np.uint64(32)).astype(np.int64), pos % np.uint64(32)
    shifted = vals << shift[None, :]
    out = np.zeros((R, W + 1), dtype=np.uint64)
    rows = np.repeat(np.arange(R), C)
    np.bitwise_or.at(out, (rows, np.tile(word, R)), (shifted & np.uint64(0xFFFFFFFF)).ravel())
    np.bitwise_or.at(out, (rows, np.tile(word + 1, R)), (shifted >> np.uint64(32)).ravel())
    return out[:, :W].astype(np.uint32)


def make_codes_bits(N: int, K: int, bits: int, seed: int, tid: int = TENSOR_IDS["qweight"]) -> np.ndarray:
    """Uniform bits-wide codes, uint8 [N, K] (the top `bits` bits of each draw)."""
    draws = splitmix64_stream(_stream_state(seed, tid), N * K)
    return (draws >> np.uint64(64 - bits)).astype(np.uint8).reshape(N, K)

def make_codes(N: int, K: int, seed: int, tid: int) -> np.ndarray:
    """Uniform 4-bit codes q[n][k] in 0..15, uint8 [N, K] (top 4 bits of each draw)."""
    bits = splitmix64_stream(_stream_state(seed, tid), N * K)
    return (bits >> np.uint64(60)).astype(np.uint8).reshape(N, K)


def make_qweight(N: int, K: int, seed: int, tid: int = TENSOR_IDS["qweight"],
                 block_rows: int = 1 << 14) -> np.ndarray:
    """Packed uniform codes, int32 [N, K/8]: word w (row-major) is the low (w even)
    or high (w odd) 32 bits of draw w // 2, i.e. 16 independent uniform 4-bit
    codes per draw. Drawn in row blocks so full-size weights stay cheap."""
    assert K % 8 == 0
    W = K // 8
    state = _stream_state(seed, tid)
    out = np.empty((N, W), dtype=np.uint32)
    for r0 in range(0, N, block_rows):
        r1 = min(N, r0 + block_rows)
        w0, w1 = r0 * W, r1 * W                      # word range [w0, w1)
        d0, d1 = w0 // 2, (w1 + 1) // 2              # draws covering it
        bits = splitmix64_stream(state, d1 - d0, offset=d0)
        words = np.empty(2 * (d1 - d0), dtype=np.uint32)
        words[0::2] = (bits & np.uint64(0xFFFFFFFF)).astype(np.uint32)
        words[1::2] = (bits >> np.uint64(32)).astype(np.uint32)
        out[r0:r1] = words[w0 - 2 * d0: w1 - 2 * d0].reshape(r1 - r0, W)
    return out.view(np.int32)


def make_scales(N: int, Kg: int, lo: float, hi: float, seed: int,
                tid: int = TENSOR_IDS["scales"]) -> np.ndarray:
    """bf16 bits [N, Kg], uniform in [lo, hi) (float64 -> float32 -> bf16, each to nearest even)."""
    u = uniform01(splitmix64_stream(_stream_state(seed, tid), N * Kg))
    return f32_to_bf16_bits((lo + (hi - lo) * u).astype(np.float32)).reshape(N, Kg)


def make_zeros(N: int, Kg: int, seed: int, tid: int = TENSOR_IDS["zeros"]) -> np.ndarray:
    """Packed 4-bit zero points, int32 [N, ceil(Kg/8)], each uniform in 0..15."""
    bits = splitmix64_stream(_stream_state(seed, tid), N * Kg)
    z = (bits >> np.uint64(60)).astype(np.uint8).reshape(N, Kg)
    return pack_nibbles_rows(z)


def make_biases(N: int, Kg: int, lo: float, hi: float, seed: int,
                tid: int = TENSOR_IDS["biases"]) -> np.ndarray:
    """bf16 bits [N, Kg], uniform in [lo, hi), drawn like the scales from their own stream."""
    return make_scales(N, Kg, lo, hi, seed, tid)


def make_x(M: int, K: int, seed: int, x_scale: float = 1.0,
           tid: int = TENSOR_IDS["x"]) -> np.ndarray:
    """bf16 bits [M, K] of N(0, 1) * x_scale (float64 -> float32 -> bf16)."""
    n = M * K
    bits = splitmix64_stream(_stream_state(seed, tid), 2 * n)
    z = normal01(bits[0::2], bits[1::2]) * x_scale
    return f32_to_bf16_bits(z.astype(np.float32)).reshape(M, K)


def make_problem(M: int, N: int, K: int, group: int, sym: bool,
                 scale_range=(0.005, 0.02), x_scale: float = 1.0, seed: int = 0,
                 gateup: bool = False, affine: bool = False, bias_range=(-0.16, -0.04)) -> dict:
    """All host arrays of one problem. With ``gateup`` a second weight (the up
    projection, same shapes) is drawn from its own streams. With ``affine``
    each weight has biases (uniform in ``bias_range``) and no zero points."""
    assert K % group == 0 and K % 8 == 0
    Kg = K // group
    lo, hi = scale_range
    p = {"M": M, "N": N, "K": K, "group": group, "sym": bool(sym), "seed": seed,
         "x": make_x(M, K, seed, x_scale),
         "qweight": make_qweight(N, K, seed),
         "scales": make_scales(N, Kg, lo, hi, seed),
         "zeros": None if (sym or affine) else make_zeros(N, Kg, seed),
         "affine": bool(affine)}
    if affine:
        p["biases"] = make_biases(N, Kg, bias_range[0], bias_range[1], seed)
    if gateup:
        p["qweight_up"] = make_qweight(N, K, seed, TENSOR_IDS["qweight_up"])
        p["scales_up"] = make_scales(N, Kg, lo, hi, seed, TENSOR_IDS["scales_up"])
        p["zeros_up"] = None if (sym or affine) else make_zeros(N, Kg, seed, TENSOR_IDS["zeros_up"])
        if affine:
            p["biases_up"] = make_biases(N, Kg, bias_range[0], bias_range[1], seed, TENSOR_IDS["biases_up"])
    return p


# Scales of the exhaustive weight: normal float32 values that bf16 holds
# exactly, from 2^-100 to 2^100, both signs; times any q - z (|q - z| <= 15)
# each stays a normal float32.
SCALE_SWEEP = (2.0 ** -100, 2.0 ** -40, 2.0 ** -20, 2.0 ** -7, 5 / 1024, 3 / 256, 0.5, 1.0,
               1.5, 201 / 64, -0.25, -3.0, 7.75, 2.0 ** 10, 2.0 ** 40, 2.0 ** 100)


def exhaustive_problem(sym: bool, N: int = 256, group: int = 64) -> dict:
    """A weight in which every (code, zero point) pair meets every scale of
    SCALE_SWEEP (with N = 256): K = 16 groups; row r holds code
    (r + k + r // 16) % 16 at column k, zero point (r + g) % 16 in group g (8
    for the symmetric form) and scale SCALE_SWEEP[(r // 16 + g) % 16].
    Besides the problem's arrays it returns the codes, zero points and scale
    bits it packed ("codes", "zero_points", "scale_bits")."""
    K = 16 * group
    r = np.arange(N)[:, None]
    g = np.arange(16)[None, :]
    codes = ((r + np.arange(K)[None, :] + r // 16) % 16).astype(np.uint8)
    zpts = np.full((N, 16), 8, dtype=np.uint8) if sym else ((r + g) % 16).astype(np.uint8)
    sweep_bits = (np.array(SCALE_SWEEP, dtype=np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    scales = sweep_bits[(r // 16 + g) % 16]
    return {"M": 1, "N": N, "K": K, "group": group, "sym": bool(sym), "seed": 0, "affine": False,
            "x": make_x(1, K, 0), "qweight": pack_nibbles_rows(codes), "scales": scales,
            "zeros": None if sym else pack_nibbles_rows(zpts),
            "codes": codes, "zero_points": zpts, "scale_bits": scales}


def planted_max_problem(M: int, N: int, K: int, group: int, planted, seed: int = 0,
                        scale_range=(0.002, 0.01)) -> dict:
    """A symmetric weight of uniform random codes and x rows of +1 and -1
    (signs from their own stream), in which row planted[m] of the weight is
    recoded to 15 where x[m] is +1 and to 0 where it is -1. Every product
    x[m][k] * (q - 8) of that row is then +7 or +8 times a positive scale, so
    row m's output is largest at column planted[m] by a wide margin."""
    planted = [int(n) for n in planted]
    assert len(planted) == M and len(set(planted)) == M
    p = make_problem(M, N, K, group, True, scale_range=scale_range, seed=seed)
    pos = (make_codes(M, K, seed, TENSOR_IDS["x_signs"]) & 1).astype(bool)
    p["x"] = np.where(pos, np.uint16(0x3F80), np.uint16(0xBF80)).astype(np.uint16)
    q = p["qweight"].copy()
    for m, n in enumerate(planted):
        q[n] = pack_nibbles_rows(np.where(pos[m], 15, 0)[None, :])[0]
    p["qweight"], p["planted"], p["x_positive"] = q, planted, pos
    return p
