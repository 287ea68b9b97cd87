"""CPU oracle for the W4A16 group-quantized matmul (float64, plain definition).

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` are the only code that may import
this package. The product path (``gemm_w4a16_group_gb300``) never does, and
this package never imports the product path.

The arithmetic lives in ``w4a16_oracle.c`` (plain C, float64); this module only
compiles it with gcc on first use and marshals numpy arrays. Besides the
zero-point form w = (q - z) * scale it holds the affine form w = scale * q +
bias of the MLX 4-bit checkpoints (TensorFold PR #859).

Error bounds (used by the parity tests):

* GEMM output y (bf16, float32 accumulation):
  ``|y - ref| <= 2^-7 |ref| + 1e-5 * sum_k |x_k w_nk|``.
* fused h = SiLU(g) * u, with g and u kept in float32 and never rounded before
  the product, first-order propagation of the two accumulation errors:
  ``|h - ref| <= 2^-7 |ref| + |SiLU'(g)| |u| Bg + |SiLU(g)| Bu + Bg Bu``
  with ``Bg = 1e-5 * sum|x wg|``, ``Bu = 1e-5 * sum|x wu|`` and
  ``SiLU'(g) = s (1 + g (1 - s))``, ``s = 1 / (1 + e^-g)``.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4a16_oracle.c")
_SO = os.path.join(_HERE, "_build", "libw4a16_oracle.so")
_lock = threading.Lock()
_lib = None

REL_TOL = 2.0 ** -7     # relative part of the output bound
ACC_TOL = 1e-5          # accumulation part, times sum_k |x_k w_nk|


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when available). Returns the .so path."""
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
        return _SO
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        raise RuntimeError("oracle: no C compiler found")
    tmp = _SO + f".{os.getpid()}.tmp"
    base = [cc, "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
            _SRC, "-o", tmp, "-lm"]
    r = subprocess.run(base[:1] + ["-fopenmp"] + base[1:], capture_output=True, text=True)
    if r.returncode != 0:  # no OpenMP: serial build
        r = subprocess.run(base, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("oracle build failed:\n" + r.stderr)
    os.replace(tmp, _SO)
    return _SO


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64 = ctypes.c_int, ctypes.c_int64
            L.oracle_code.argtypes = [P, i32, i32, i32]
            L.oracle_code.restype = i32
            L.oracle_zero.argtypes = [P, i32, i32, i32, i32]
            L.oracle_zero.restype = i32
            L.oracle_weight.argtypes = [P, P, P, i32, i32, i32, i32, i32]
            L.oracle_weight.restype = ctypes.c_double
            L.oracle_dequant.argtypes = [P, P, P, i32, i32, i32, i32, P]
            L.oracle_dequant.restype = None
            L.oracle_gemm.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, P, P, i32]
            L.oracle_gemm.restype = i32
            L.oracle_gemm_at.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, P, P, i64, P, P, i32]
            L.oracle_gemm_at.restype = i32
            L.oracle_gateup_silu_at.argtypes = ([P] * 7 + [i32] * 5 + [P, P, i64] + [P] * 5 + [i32])
            L.oracle_gateup_silu_at.restype = i32
            L.oracle_silu_mul.argtypes = [ctypes.c_double, ctypes.c_double]
            L.oracle_silu_mul.restype = ctypes.c_double
            L.oracle_weight_affine.argtypes = [P, P, P, i32, i32, i32, i32]
            L.oracle_weight_affine.restype = ctypes.c_double
            L.oracle_dequant_affine.argtypes = [P, P, P, i32, i32, i32, P]
            L.oracle_dequant_affine.restype = None
            L.oracle_gemm_affine.argtypes = [P, P, P, P, i32, i32, i32, i32, P, P, i32]
            L.oracle_gemm_affine.restype = i32
            L.oracle_gemm_affine_at.argtypes = [P, P, P, P, i32, i32, i32, i32, P, P, i64, P, P, i32]
            L.oracle_gemm_affine_at.restype = i32
            L.oracle_gateup_silu_affine_at.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, P, P, i64,
                                                       P, P, P, P, P, i32]
            L.oracle_gateup_silu_affine_at.restype = i32
            L.oracle_group_sums.argtypes = [P, i32, i32, i32, P]
            L.oracle_group_sums.restype = i32
            L.oracle_threads.argtypes = [i32]
            L.oracle_threads.restype = i32
            L.oracle_code_bits.argtypes = [P, i32, i32, i32, i32]
            L.oracle_code_bits.restype = i32
            L.oracle_dequant_affine_bits.argtypes = [P, P, P, i32, i32, i32, i32, P]
            L.oracle_dequant_affine_bits.restype = i32
            L.oracle_gemm_affine_bits.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, P, P, i32]
            L.oracle_gemm_affine_bits.restype = i32
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def _c(a, dt):
    return None if a is None else np.ascontiguousarray(a, dtype=dt)


def threads(nthreads: int = 0) -> int:
    """Threads a call with ``nthreads`` uses (0 = every core OpenMP sees)."""
    return lib().oracle_threads(nthreads)


def code(qweight, K, n, k) -> int:
    q = _c(qweight, np.int32)
    return lib().oracle_code(_p(q), K, n, k)


def zero(zeros, Kg, sym, n, g) -> int:
    z = _c(zeros, np.int32)
    return lib().oracle_zero(_p(z), Kg, int(sym), n, g)


def dequant(qweight, scales, zeros, N, K, group, sym) -> np.ndarray:
    """float64 [N, K]: w = (q - z) * scale."""
    q, s, z = _c(qweight, np.int32), _c(scales, np.uint16), _c(zeros, np.int32)
    w = np.empty((N, K), dtype=np.float64)
    lib().oracle_dequant(_p(q), _p(s), _p(z), N, K, group, int(sym), _p(w))
    return w


def dequant_affine(qweight, scales, biases, N, K, group) -> np.ndarray:
    """float64 [N, K]: w = scale * q + bias (the affine form)."""
    q, s, b = _c(qweight, np.int32), _c(scales, np.uint16), _c(biases, np.uint16)
    w = np.empty((N, K), dtype=np.float64)
    lib().oracle_dequant_affine(_p(q), _p(s), _p(b), N, K, group, _p(w))
    return w


def gemm_affine(x, qweight, scales, biases, M, N, K, group, nthreads: int = 0):
    """(y, sum_abs) of the affine form, float64 [M, N] each."""
    x, q, s, b = (_c(x, np.uint16), _c(qweight, np.int32), _c(scales, np.uint16), _c(biases, np.uint16))
    y = np.empty((M, N), dtype=np.float64)
    a = np.empty((M, N), dtype=np.float64)
    rc = lib().oracle_gemm_affine(_p(x), _p(q), _p(s), _p(b), M, N, K, group, _p(y), _p(a), nthreads)
    if rc:
        raise ValueError("oracle_gemm_affine: bad arguments")
    return y, a


def gemm_affine_at(x, qweight, scales, biases, M, N, K, group, m_idx, n_idx, nthreads: int = 0):
    """(y, sum_abs) of the affine form at the given (m, n) pairs."""
    x, q, s, b = (_c(x, np.uint16), _c(qweight, np.int32), _c(scales, np.uint16), _c(biases, np.uint16))
    mi, ni = _c(m_idx, np.int64), _c(n_idx, np.int64)
    cnt = mi.size
    y = np.empty(cnt, dtype=np.float64)
    a = np.empty(cnt, dtype=np.float64)
    rc = lib().oracle_gemm_affine_at(_p(x), _p(q), _p(s), _p(b), M, N, K, group, _p(mi), _p(ni), cnt,
                                     _p(y), _p(a), nthreads)
    if rc:
        raise ValueError("oracle_gemm_affine_at: bad arguments")
    return y, a


def gemm(x, qweight, scales, zeros, M, N, K, group, sym, nthreads: int = 0):
    """(y, sum_abs), float64 [M, N] each."""
    x, q, s, z = (_c(x, np.uint16), _c(qweight, np.int32), _c(scales, np.uint16),
                  _c(zeros, np.int32))
    y = np.empty((M, N), dtype=np.float64)
    a = np.empty((M, N), dtype=np.float64)
    rc = lib().oracle_gemm(_p(x), _p(q), _p(s), _p(z), M, N, K, group, int(sym),
                           _p(y), _p(a), nthreads)
    if rc:
        raise ValueError("oracle_gemm: bad arguments")
    return y, a


def gemm_at(x, qweight, scales, zeros, M, N, K, group, sym, m_idx, n_idx, nthreads: int = 0):
    """(y, sum_abs) at the given (m, n) pairs, float64 [count] each."""
    x, q, s, z = (_c(x, np.uint16), _c(qweight, np.int32), _c(scales, np.uint16),
                  _c(zeros, np.int32))
    mi, ni = _c(m_idx, np.int64), _c(n_idx, np.int64)
    cnt = mi.size
    y = np.empty(cnt, dtype=np.float64)
    a = np.empty(cnt, dtype=np.float64)
    rc = lib().oracle_gemm_at(_p(x), _p(q), _p(s), _p(z), M, N, K, group, int(sym),
                              _p(mi), _p(ni), cnt, _p(y), _p(a), nthreads)
    if rc:
        raise ValueError("oracle_gemm_at: bad arguments")
    return y, a


def gateup_silu_at(x, qg, sg, zg, qu, su, zu, M, N, K, group, sym, m_idx, n_idx,
                   nthreads: int = 0):
    """(h, g, u, gsum_abs, usum_abs) at the given (m, n) pairs."""
    x = _c(x, np.uint16)
    qg, sg, zg = _c(qg, np.int32), _c(sg, np.uint16), _c(zg, np.int32)
    qu, su, zu = _c(qu, np.int32), _c(su, np.uint16), _c(zu, np.int32)
    mi, ni = _c(m_idx, np.int64), _c(n_idx, np.int64)
    cnt = mi.size
    outs = [np.empty(cnt, dtype=np.float64) for _ in range(5)]
    rc = lib().oracle_gateup_silu_at(_p(x), _p(qg), _p(sg), _p(zg), _p(qu), _p(su), _p(zu),
                                     M, N, K, group, int(sym), _p(mi), _p(ni), cnt,
                                     *[_p(o) for o in outs], nthreads)
    if rc:
        raise ValueError("oracle_gateup_silu_at: bad arguments")
    return tuple(outs)


def gateup_silu_affine_at(x, qg, sg, bg, qu, su, bu, M, N, K, group, m_idx, n_idx, nthreads: int = 0):
    """(h, g, u, gsum_abs, usum_abs) of the affine form at the given (m, n) pairs."""
    x = _c(x, np.uint16)
    qg, sg, bg = _c(qg, np.int32), _c(sg, np.uint16), _c(bg, np.uint16)
    qu, su, bu = _c(qu, np.int32), _c(su, np.uint16), _c(bu, np.uint16)
    mi, ni = _c(m_idx, np.int64), _c(n_idx, np.int64)
    cnt = mi.size
    outs = [np.empty(cnt, dtype=np.float64) for _ in range(5)]
    rc = lib().oracle_gateup_silu_affine_at(_p(x), _p(qg), _p(sg), _p(bg), _p(qu), _p(su), _p(bu),
                                            M, N, K, group, _p(mi), _p(ni), cnt, *[_p(o) for o in outs],
                                            nthreads)
    if rc:
        raise ValueError("oracle_gateup_silu_affine_at: bad arguments")
    return tuple(outs)



def code_bits(qweight, K, bits, n, k) -> int:
    """Code k of row n of a bits-wide weight (uint32 [N, ceil(K*bits/32)], one
    little-endian bit stream per row)."""
    q = _c(qweight, np.uint32)
    return lib().oracle_code_bits(_p(q), K, bits, n, k)


def dequant_affine_bits(qweight, scales, biases, N, K, group, bits) -> np.ndarray:
    """float64 [N, K]: w = scale * q + bias of a bits-wide affine weight."""
    q, s, b = _c(qweight, np.uint32), _c(scales, np.uint16), _c(biases, np.uint16)
    w = np.empty((N, K), dtype=np.float64)
    if lib().oracle_dequant_affine_bits(_p(q), _p(s), _p(b), N, K, group, bits, _p(w)):
        raise ValueError("oracle_dequant_affine_bits: bad arguments")
    return w


def gemm_affine_bits(x, qweight, scales, biases, M, N, K, group, bits, nthreads: int = 0):
    """(y, sum_abs), float64 [M, N] each, of a bits-wide affine weight."""
    x, q, s, b = (_c(x, np.uint16), _c(qweight, np.uint32), _c(scales, np.uint16), _c(biases, np.uint16))
    y = np.empty((M, N), dtype=np.float64)
    a = np.empty((M, N), dtype=np.float64)
    rc = lib().oracle_gemm_affine_bits(_p(x), _p(q), _p(s), _p(b), M, N, K, group, bits, _p(y), _p(a), nthreads)
    if rc:
        raise ValueError("oracle_gemm_affine_bits: bad arguments")
    return y, a

def group_sums(x, M, K, group) -> np.ndarray:
    """float64 [K/G, M]: the sum of x[m] over each group of K."""
    x = _c(x, np.uint16)
    xs = np.empty((K // group, M), dtype=np.float64)
    if lib().oracle_group_sums(_p(x), M, K, group, _p(xs)):
        raise ValueError("oracle_group_sums: bad arguments")
    return xs


def silu_mul(g: float, u: float) -> float:
    return lib().oracle_silu_mul(float(g), float(u))


def gemm_bound(ref, sum_abs):
    """Allowed |y - ref| for a bf16 output of a float32-accumulated sum."""
    return REL_TOL * np.abs(ref) + ACC_TOL * np.asarray(sum_abs)


def sigmoid(g):
    """The logistic function 1 / (1 + e^-g), float64 (0 where e^-g overflows)."""
    g = np.asarray(g, dtype=np.float64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-g))


def dsilu(g):
    """SiLU'(g) = d/dg [g s(g)] = s (1 + g (1 - s)), s the logistic function."""
    g = np.asarray(g, dtype=np.float64)
    s = sigmoid(g)
    return s * (1.0 + g * (1.0 - s))


def silu_bound(h_ref, g, u, gsum_abs, usum_abs):
    """Allowed |h - ref| for the fused SiLU(g) * u output (first-order propagation)."""
    g = np.asarray(g, dtype=np.float64)
    u = np.asarray(u, dtype=np.float64)
    bg = ACC_TOL * np.asarray(gsum_abs)
    bu = ACC_TOL * np.asarray(usum_abs)
    return (REL_TOL * np.abs(h_ref) + np.abs(dsilu(g)) * np.abs(u) * bg
            + np.abs(g * sigmoid(g)) * bu + bg * bu)


def _bf16_rank(bits) -> np.ndarray:
    """Order key of bf16 bit patterns, larger key = larger value: sign and
    magnitude as a signed integer (so -0 and +0 share the key 0), and every
    NaN one step above +inf."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    mag = b & 0x7FFF
    key = np.where(b & 0x8000, -mag, mag)
    return np.where(mag > 0x7F80, 0x7F81, key)


def topk_bf16(y_bits, k: int):
    """The k largest entries of every row of a bf16 matrix (bits [M, N]), the
    greedy pick of the GPU-side token selection (lucebox PR #823, description)
    widened from 1 to k: largest value first; equal values (-0 and +0 among
    them) lowest column first; a NaN ranks above +inf. Returns (indices int64
    [M, k], value bits uint16 [M, k]). A stable sort of the negated key keeps
    equal keys in column order."""
    y = np.atleast_2d(np.asarray(y_bits, dtype=np.uint16))
    M, N = y.shape
    if not 1 <= k <= N:
        raise ValueError("topk_bf16: need 1 <= k <= N")
    order = np.argsort(-_bf16_rank(y), axis=1, kind="stable")[:, :k]
    return order.astype(np.int64), np.take_along_axis(y, order, axis=1)
