"""GB300 (sm_103a) W4A16 group-quantized matmul: thin Python binding.

Every call marshals torch tensors into the C ABI of ``include/w4a16.h`` and
runs on the current CUDA stream; all arithmetic happens in the CUDA library
(``_build/libw4a16_gb300.so``, built in-tree by ``build.py``). There is no
CPU or PyTorch fallback: if the library cannot be loaded every call raises.

    packed = repack(qweight, scales, zeros, N, K, group, sym)     # once per weight
    y = gemm(x, packed, N, K, group, sym)                          # y = x . dequant(W)^T
    pg = repack_gateup(qg, sg, zg, qu, su, zu, N, K, group, sym)
    h = gateup_silu(x, pg, N, K, group, sym)                       # SiLU(x Wg^T) * (x Wu^T)

Affine form w = scale * q + bias (MLX affine 4-bit checkpoints):

    pa = repack_affine(qweight, scales, biases, N, K, group)
    xs = xsum(x, K, group)                 # group sums of x, shared by every weight on x
    y = gemm_affine(x, pa, N, K, group, xs)
"""
from __future__ import annotations

import ctypes
import functools
import os

from . import build as _build

__all__ = [
    "EXPORTS", "W4A16Error", "lib", "library_path", "repacked_bytes", "gateup_repacked_bytes",
    "repack", "repack_gateup", "gemm", "gemm_argmax", "gateup_silu", "dequantize", "kernel_status",
    "set_kernel_override", "set_programmatic_overlap", "strerror", "KERNEL_AUTO", "KERNEL_GEMV", "KERNEL_SMALLM", "KERNEL_TC",
    "KERNEL_XSTAGED", "KERNEL_DECODE_TC",
    "AFFINE", "repack_affine", "repack_affine_gateup", "xsum_bytes", "xsum", "gemm_affine", "gateup_silu_affine",
    "gemm_affine_noalloc", "topk", "gemm_topk", "affine_bits_repacked_bytes", "repack_affine_bits",
    "affine_bits_scratch_bytes", "gemm_affine_bits", "dequantize_affine_bits",
]

# symbols declared in include/w4a16.h
EXPORTS = (
    "w4a16_repacked_bytes", "w4a16_repack", "w4a16_gateup_repacked_bytes", "w4a16_repack_gateup",
    "w4a16_gemm", "w4a16_gemm_argmax", "w4a16_gateup_silu", "w4a16_dequantize", "w4a16_kernel_status",
    "w4a16_strerror", "w4a16_last_cuda_error", "w4a16_set_kernel_override",
    "w4a16_set_programmatic_overlap", "w4a16_repack_affine", "w4a16_repack_affine_gateup", "w4a16_xsum_bytes",
    "w4a16_xsum", "w4a16_gemm_affine", "w4a16_gateup_silu_affine", "w4a16_gemm_affine_noalloc",
    "w4a16_topk", "w4a16_gemm_topk", "w4a16_affine_bits_repacked_bytes", "w4a16_repack_affine_bits",
    "w4a16_affine_bits_scratch_bytes", "w4a16_gemm_affine_bits", "w4a16_dequantize_affine_bits",
)
KERNEL_AUTO, KERNEL_GEMV, KERNEL_SMALLM, KERNEL_TC, KERNEL_XSTAGED, KERNEL_DECODE_TC = 0, 1, 2, 3, 4, 5
# the `sym` argument: 0 zero points, 1 symmetric (z = 8), AFFINE scale * q + bias
AFFINE = 2


class W4A16Error(RuntimeError):
    pass


_lib = None


def library_path() -> str:
    return _build.LIB


def lib(auto_build: bool = True) -> ctypes.CDLL:
    """The loaded CUDA library (compiled first if missing or stale and nvcc is present)."""
    global _lib
    if _lib is not None:
        return _lib
    if auto_build and not _build.up_to_date():
        try:
            _build.build()
        except Exception as e:  # fall through to the load error below
            if not os.path.exists(_build.LIB):
                raise W4A16Error(f"CUDA library missing and build failed: {e}") from e
    if not os.path.exists(_build.LIB):
        raise W4A16Error(f"CUDA library not built: {_build.LIB}")
    L = ctypes.CDLL(_build.LIB)
    P, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    L.w4a16_repacked_bytes.argtypes = [i32, i32, i32, i32]
    L.w4a16_repacked_bytes.restype = sz
    L.w4a16_gateup_repacked_bytes.argtypes = [i32, i32, i32, i32]
    L.w4a16_gateup_repacked_bytes.restype = sz
    L.w4a16_repack.argtypes = [P, P, P, i32, i32, i32, i32, P, P]
    L.w4a16_repack.restype = i32
    L.w4a16_repack_gateup.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, P, P]
    L.w4a16_repack_gateup.restype = i32
    L.w4a16_gemm.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, P, P]
    L.w4a16_gemm.restype = i32
    L.w4a16_gemm_argmax.argtypes = [P, P, i32, i32, i32, i32, i32, P, P, P]
    L.w4a16_gemm_argmax.restype = i32
    L.w4a16_gateup_silu.argtypes = [P, P, i32, i32, i32, i32, i32, P, P]
    L.w4a16_gateup_silu.restype = i32
    L.w4a16_dequantize.argtypes = [P, i32, i32, i32, i32, P, P]
    L.w4a16_dequantize.restype = i32
    L.w4a16_kernel_status.argtypes = []
    L.w4a16_kernel_status.restype = i32
    L.w4a16_strerror.argtypes = [i32]
    L.w4a16_strerror.restype = ctypes.c_char_p
    L.w4a16_last_cuda_error.argtypes = []
    L.w4a16_last_cuda_error.restype = i32
    L.w4a16_set_kernel_override.argtypes = [i32]
    L.w4a16_set_kernel_override.restype = i32
    L.w4a16_set_programmatic_overlap.argtypes = [i32]
    L.w4a16_set_programmatic_overlap.restype = i32
    L.w4a16_repack_affine.argtypes = [P, P, P, i32, i32, i32, P, P]
    L.w4a16_repack_affine.restype = i32
    L.w4a16_repack_affine_gateup.argtypes = [P, P, P, P, P, P, i32, i32, i32, P, P]
    L.w4a16_repack_affine_gateup.restype = i32
    L.w4a16_xsum_bytes.argtypes = [i32, i32, i32]
    L.w4a16_xsum_bytes.restype = sz
    L.w4a16_xsum.argtypes = [P, i32, i32, i32, P, P]
    L.w4a16_xsum.restype = i32
    L.w4a16_gemm_affine.argtypes = [P, P, P, i32, i32, i32, i32, P, P]
    L.w4a16_gemm_affine.restype = i32
    L.w4a16_gateup_silu_affine.argtypes = [P, P, P, i32, i32, i32, i32, P, P]
    L.w4a16_gateup_silu_affine.restype = i32
    L.w4a16_gemm_affine_noalloc.argtypes = [P, P, i32, i32, i32, i32, P, P]
    L.w4a16_gemm_affine_noalloc.restype = i32
    L.w4a16_topk.argtypes = [P, i32, i32, i32, P, P, P]
    L.w4a16_topk.restype = i32
    L.w4a16_gemm_topk.argtypes = [P, P, i32, i32, i32, i32, i32, i32, P, P, P, P]
    L.w4a16_gemm_topk.restype = i32
    L.w4a16_affine_bits_repacked_bytes.argtypes = [i32, i32, i32, i32]
    L.w4a16_affine_bits_repacked_bytes.restype = ctypes.c_size_t
    L.w4a16_repack_affine_bits.argtypes = [P, P, P, i32, i32, i32, i32, P, P]
    L.w4a16_repack_affine_bits.restype = i32
    L.w4a16_affine_bits_scratch_bytes.argtypes = [i32, i32, i32, i32]
    L.w4a16_affine_bits_scratch_bytes.restype = ctypes.c_size_t
    L.w4a16_gemm_affine_bits.argtypes = [P, P, P, i32, i32, i32, i32, i32, P, P]
    L.w4a16_gemm_affine_bits.restype = i32
    L.w4a16_dequantize_affine_bits.argtypes = [P, i32, i32, i32, i32, P, P]
    L.w4a16_dequantize_affine_bits.restype = i32
    _lib = L
    return L


def strerror(rc: int) -> str:
    return lib().w4a16_strerror(rc).decode()


def _check(rc: int, what: str):
    if rc != 0:
        msg = f"{what}: {strerror(rc)} (status {rc}"
        if rc == -4:
            msg += f", cudaError {lib().w4a16_last_cuda_error()}"
        raise W4A16Error(msg + ")")


def _torch():
    import torch
    return torch


@functools.lru_cache(maxsize=1)
def _device_count() -> int:
    return _torch().cuda.device_count()


def _stream(stream, device=None):
    """The call's stream handle. The library launches on the current CUDA
    device, so the call's tensors (on `device`) must live there; with one
    visible device they always do."""
    torch = _torch()
    if device is not None and _device_count() > 1 and device.index != torch.cuda.current_device():
        raise ValueError(f"the tensors are on {device} but the current CUDA device is "
                         f"cuda:{torch.cuda.current_device()}: the library launches on the current device")
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _is_device_tensor(t) -> bool:
    return t.is_cuda


def _ptr(t, dtypes, name, nbytes=0, device=None):
    """Data pointer of `t` after the checks a plain C pointer cannot carry:
    dtype, residency on the call's device, contiguity, and room for the
    `nbytes` bytes the call reads or writes through it."""
    if t is None:
        return None
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if not _is_device_tensor(t):
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, the call's other tensors on {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.nbytes < nbytes:
        raise ValueError(f"{name} holds {t.nbytes} bytes, the call needs {nbytes}")
    return ctypes.c_void_p(t.data_ptr())


_BF16 = None


def _bf16_types():
    global _BF16
    if _BF16 is None:
        torch = _torch()
        _BF16 = (torch.bfloat16, torch.int16, torch.uint16)
    return _BF16


@functools.lru_cache(maxsize=1024)
def _packed_bytes(N: int, K: int, group: int, form: int, gateup: bool) -> int:
    L = lib()
    f = L.w4a16_gateup_repacked_bytes if gateup else L.w4a16_repacked_bytes
    return int(f(N, K, group, form))


def _canonical_bytes(N: int, K: int, group: int):
    """Bytes of a canonical weight's qweight (int32 [N, K/8]), scales or
    biases (bf16 [N, K/G]) and zeros (int32 [N, ceil(K/G/8)])."""
    groups = K // group if group > 0 else 0
    return N * K // 2, N * groups * 2, N * ((groups + 7) // 8) * 4


def _x_rows(x, K) -> int:
    if x.dim() != 2:
        raise ValueError("x must be [M, K]")
    M, k = x.shape
    if k != K:
        raise ValueError("x must be [M, K]")
    return M


def repacked_bytes(N: int, K: int, group: int, sym: bool) -> int:
    return int(lib().w4a16_repacked_bytes(N, K, group, int(sym)))


def gateup_repacked_bytes(N_each: int, K: int, group: int, sym: bool) -> int:
    return int(lib().w4a16_gateup_repacked_bytes(N_each, K, group, int(sym)))


def repack(qweight, scales, zeros, N, K, group, sym, stream=None, out=None):
    """Canonical (qweight int32 [N, K/8], scales bf16 [N, K/G], zeros int32) -> packed uint8 tensor."""
    torch = _torch()
    nbytes = repacked_bytes(N, K, group, sym)
    if nbytes == 0:
        raise W4A16Error("repack: unsupported sizes")
    d = qweight.device
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=d)
    bq, bs, bz = _canonical_bytes(N, K, group)
    rc = lib().w4a16_repack(_ptr(qweight, (torch.int32,), "qweight", bq, d),
                            _ptr(scales, _bf16_types(), "scales", bs, d),
                            _ptr(zeros, (torch.int32,), "zeros", bz, d), N, K, group, int(sym),
                            _ptr(out, (torch.uint8,), "out", nbytes, d), _stream(stream, d))
    _check(rc, "w4a16_repack")
    return out


def repack_gateup(qw_gate, sc_gate, z_gate, qw_up, sc_up, z_up, N_each, K, group, sym, stream=None):
    torch = _torch()
    nbytes = gateup_repacked_bytes(N_each, K, group, sym)
    if nbytes == 0:
        raise W4A16Error("repack_gateup: unsupported sizes")
    d = qw_gate.device
    out = torch.empty(nbytes, dtype=torch.uint8, device=d)
    i32, b16 = (torch.int32,), _bf16_types()
    bq, bs, bz = _canonical_bytes(N_each, K, group)
    rc = lib().w4a16_repack_gateup(_ptr(qw_gate, i32, "qw_gate", bq, d), _ptr(sc_gate, b16, "sc_gate", bs, d),
                                   _ptr(z_gate, i32, "z_gate", bz, d), _ptr(qw_up, i32, "qw_up", bq, d),
                                   _ptr(sc_up, b16, "sc_up", bs, d), _ptr(z_up, i32, "z_up", bz, d), N_each, K,
                                   group, int(sym), ctypes.c_void_p(out.data_ptr()), _stream(stream, d))
    _check(rc, "w4a16_repack_gateup")
    return out


def gemm(x, packed, N, K, group, sym, out=None, stream=None):
    """y[M, N] (bf16) = x[M, K] (bf16) . dequant(W)^T."""
    torch = _torch()
    M = _x_rows(x, K)
    d = x.device
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=d)
    rc = lib().w4a16_gemm(_ptr(x, _bf16_types(), "x", 0, d),
                          _ptr(packed, (torch.uint8,), "packed", _packed_bytes(N, K, group, int(sym), False), d),
                          None, None, M, N, K, group, int(sym), _ptr(out, _bf16_types(), "out", 2 * M * N, d),
                          _stream(stream, d))
    _check(rc, "w4a16_gemm")
    return out


def gemm_argmax(x, packed, N, K, group, sym, out=None, logits=False, stream=None, index_out=None):
    """int64 [M]: the first column of each row of y = x . dequant(W)^T (bf16)
    at which y is largest (torch.argmax over the bf16 row). For M <= 32 the
    logits are stored only when `logits` is true or `out` is given; returns
    (argmax, y or None)."""
    torch = _torch()
    M = _x_rows(x, K)
    d = x.device
    if out is None and (logits or M > 32):
        out = torch.empty((M, N), dtype=torch.bfloat16, device=d)
    idx = index_out if index_out is not None else torch.empty(M, dtype=torch.int64, device=d)
    rc = lib().w4a16_gemm_argmax(_ptr(x, _bf16_types(), "x", 0, d),
                                 _ptr(packed, (torch.uint8,), "packed", _packed_bytes(N, K, group, int(sym), False),
                                      d),
                                 M, N, K, group, int(sym), _ptr(out, _bf16_types(), "out", 2 * M * N, d),
                                 _ptr(idx, (torch.int64,), "index_out", 8 * M, d), _stream(stream, d))
    _check(rc, "w4a16_gemm_argmax")
    return idx, out


TOPK_MAX_K = 1024


def _topk_outs(M, k, d, index_out, values_out, values):
    torch = _torch()
    idx = index_out if index_out is not None else torch.empty((M, k), dtype=torch.int64, device=d)
    vals = values_out
    if vals is None and values:
        vals = torch.empty((M, k), dtype=torch.bfloat16, device=d)
    return idx, vals


def topk(y, k, index_out=None, values_out=None, values=True, stream=None):
    """The k largest entries of every row of the bf16 logits y [M, N], largest
    first (equal values lowest column first, -0 = +0, NaN above +inf).
    Returns (indices int64 [M, k], values bf16 [M, k] or None)."""
    torch = _torch()
    if y.dim() != 2:
        raise ValueError("y must be [M, N]")
    M, N = y.shape
    d = y.device
    idx, vals = _topk_outs(M, k, d, index_out, values_out, values)
    rc = lib().w4a16_topk(_ptr(y, _bf16_types(), "y", 2 * M * N, d), M, N, k,
                          _ptr(idx, (torch.int64,), "index_out", 8 * M * k, d),
                          _ptr(vals, _bf16_types(), "values_out", 2 * M * k, d), _stream(stream, d))
    _check(rc, "w4a16_topk")
    return idx, vals


def gemm_topk(x, packed, N, K, group, sym, k, out=None, index_out=None, values_out=None, values=True, stream=None):
    """y = x . dequant(W)^T (bf16, into `out` or a new tensor), then the top-k
    of each row of y. Returns (indices, values or None, y)."""
    torch = _torch()
    M = _x_rows(x, K)
    d = x.device
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=d)
    idx, vals = _topk_outs(M, k, d, index_out, values_out, values)
    rc = lib().w4a16_gemm_topk(_ptr(x, _bf16_types(), "x", 0, d),
                               _ptr(packed, (torch.uint8,), "packed", _packed_bytes(N, K, group, int(sym), False), d),
                               M, N, K, group, int(sym), k, _ptr(out, _bf16_types(), "out", 2 * M * N, d),
                               _ptr(idx, (torch.int64,), "index_out", 8 * M * k, d),
                               _ptr(vals, _bf16_types(), "values_out", 2 * M * k, d), _stream(stream, d))
    _check(rc, "w4a16_gemm_topk")
    return idx, vals, out


def gateup_silu(x, packed_gateup, N_each, K, group, sym, out=None, stream=None):
    """h[M, N_each] (bf16) = SiLU(x Wg^T) * (x Wu^T)."""
    torch = _torch()
    M = _x_rows(x, K)
    d = x.device
    if out is None:
        out = torch.empty((M, N_each), dtype=torch.bfloat16, device=d)
    rc = lib().w4a16_gateup_silu(_ptr(x, _bf16_types(), "x", 0, d),
                                 _ptr(packed_gateup, (torch.uint8,), "packed",
                                      _packed_bytes(N_each, K, group, int(sym), True), d),
                                 M, N_each, K, group, int(sym), _ptr(out, _bf16_types(), "out", 2 * M * N_each, d),
                                 _stream(stream, d))
    _check(rc, "w4a16_gateup_silu")
    return out


def repack_affine(qweight, scales, biases, N, K, group, stream=None):
    """Canonical affine weight (qweight int32 [N, K/8], scales and biases bf16 [N, K/G]) -> packed uint8."""
    torch = _torch()
    nbytes = repacked_bytes(N, K, group, AFFINE)
    if nbytes == 0:
        raise W4A16Error("repack_affine: unsupported sizes")
    d = qweight.device
    out = torch.empty(nbytes, dtype=torch.uint8, device=d)
    b16 = _bf16_types()
    bq, bs, _ = _canonical_bytes(N, K, group)
    rc = lib().w4a16_repack_affine(_ptr(qweight, (torch.int32,), "qweight", bq, d),
                                   _ptr(scales, b16, "scales", bs, d), _ptr(biases, b16, "biases", bs, d), N, K,
                                   group, ctypes.c_void_p(out.data_ptr()), _stream(stream, d))
    _check(rc, "w4a16_repack_affine")
    return out


def repack_affine_gateup(qw_gate, sc_gate, b_gate, qw_up, sc_up, b_up, N_each, K, group, stream=None):
    torch = _torch()
    nbytes = gateup_repacked_bytes(N_each, K, group, AFFINE)
    if nbytes == 0:
        raise W4A16Error("repack_affine_gateup: unsupported sizes")
    d = qw_gate.device
    out = torch.empty(nbytes, dtype=torch.uint8, device=d)
    i32, b16 = (torch.int32,), _bf16_types()
    bq, bs, _ = _canonical_bytes(N_each, K, group)
    rc = lib().w4a16_repack_affine_gateup(_ptr(qw_gate, i32, "qw_gate", bq, d), _ptr(sc_gate, b16, "sc_gate", bs, d),
                                          _ptr(b_gate, b16, "b_gate", bs, d), _ptr(qw_up, i32, "qw_up", bq, d),
                                          _ptr(sc_up, b16, "sc_up", bs, d), _ptr(b_up, b16, "b_up", bs, d), N_each,
                                          K, group, ctypes.c_void_p(out.data_ptr()), _stream(stream, d))
    _check(rc, "w4a16_repack_affine_gateup")
    return out


def xsum_bytes(M: int, K: int, group: int) -> int:
    return int(lib().w4a16_xsum_bytes(M, K, group))


def xsum(x, K, group, out=None, stream=None):
    """bf16 [M, kb3]: the sum of x[m] over each group g as three bf16 parts
    (hi, mid, lo at columns 3g .. 3g+2) that add up to the float32 sum exactly."""
    torch = _torch()
    M = _x_rows(x, K)
    nbytes = xsum_bytes(M, K, group)
    if nbytes == 0:
        raise W4A16Error("xsum: unsupported sizes")
    d = x.device
    if out is None:
        out = torch.empty((M, nbytes // 2 // M), dtype=torch.bfloat16, device=d)
    rc = lib().w4a16_xsum(_ptr(x, _bf16_types(), "x", 0, d), M, K, group,
                          _ptr(out, _bf16_types(), "out", nbytes, d), _stream(stream, d))
    _check(rc, "w4a16_xsum")
    return out


def _xs_ptr(xs, M, K, group, d):
    # the table is read only by the tcgen05 GEMM (M > 32), but whenever one is
    # passed it must be whole
    return None if xs is None else _ptr(xs, _bf16_types(), "xsum", xsum_bytes(M, K, group), d)


def gemm_affine(x, packed, N, K, group, xs=None, out=None, stream=None):
    """y[M, N] (bf16) = x . (scale * q + bias)^T. `xs` (from xsum) is needed
    for M > 32; None lets the M <= 32 kernels form the group sums themselves."""
    torch = _torch()
    M = _x_rows(x, K)
    d = x.device
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=d)
    rc = lib().w4a16_gemm_affine(_ptr(x, _bf16_types(), "x", 0, d), _xs_ptr(xs, M, K, group, d),
                                 _ptr(packed, (torch.uint8,), "packed", _packed_bytes(N, K, group, AFFINE, False), d),
                                 M, N, K, group, _ptr(out, _bf16_types(), "out", 2 * M * N, d), _stream(stream, d))
    _check(rc, "w4a16_gemm_affine")
    return out


def gemm_affine_noalloc(x, packed, N, K, group, out=None, stream=None):
    """gemm_affine with the group sums in the library's fixed device array (no
    table argument; calls in flight at once on one device race on it)."""
    torch = _torch()
    M = _x_rows(x, K)
    d = x.device
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=d)
    rc = lib().w4a16_gemm_affine_noalloc(_ptr(x, _bf16_types(), "x", 0, d),
                                         _ptr(packed, (torch.uint8,), "packed",
                                              _packed_bytes(N, K, group, AFFINE, False), d),
                                         M, N, K, group, _ptr(out, _bf16_types(), "out", 2 * M * N, d),
                                         _stream(stream, d))
    _check(rc, "w4a16_gemm_affine_noalloc")
    return out


def affine_bits_repacked_bytes(N: int, K: int, group: int, bits: int) -> int:
    return int(lib().w4a16_affine_bits_repacked_bytes(N, K, group, bits))


def affine_bits_scratch_bytes(M: int, K: int, group: int, bits: int) -> int:
    return int(lib().w4a16_affine_bits_scratch_bytes(M, K, group, bits))


def repack_affine_bits(qweight, scales, biases, N, K, group, bits, stream=None):
    """Canonical b-bit affine weight (qweight uint32/int32 [N, ceil(K*bits/32)],
    one bit stream per row; scales and biases bf16 [N, K/G]) -> packed uint8."""
    torch = _torch()
    nbytes = affine_bits_repacked_bytes(N, K, group, bits)
    if nbytes == 0:
        raise W4A16Error(f"unsupported b-bit affine weight N={N} K={K} group={group} bits={bits}")
    d = qweight.device
    out = torch.empty(nbytes, dtype=torch.uint8, device=d)
    qbytes = N * ((K * bits + 31) // 32) * 4
    _, sbytes, _ = _canonical_bytes(N, K, group)
    rc = lib().w4a16_repack_affine_bits(_ptr(qweight, (torch.int32, torch.uint32), "qweight", qbytes, d),
                                        _ptr(scales, _bf16_types(), "scales", sbytes, d),
                                        _ptr(biases, _bf16_types(), "biases", sbytes, d), N, K, group, bits,
                                        _ptr(out, (torch.uint8,), "packed", nbytes, d), _stream(stream, d))
    _check(rc, "w4a16_repack_affine_bits")
    return out


def gemm_affine_bits(x, packed, N, K, group, bits, scratch=None, out=None, stream=None):
    """y[M, N] (bf16) = x . (scale * q + bias)^T of a b-bit affine weight;
    `scratch` (uint8, affine_bits_scratch_bytes) is allocated when not given."""
    torch = _torch()
    M = _x_rows(x, K)
    d = x.device
    sbytes = affine_bits_scratch_bytes(M, K, group, bits)
    if sbytes == 0:
        raise W4A16Error(f"unsupported b-bit affine call M={M} K={K} group={group} bits={bits}")
    if scratch is None:
        scratch = torch.empty(sbytes, dtype=torch.uint8, device=d)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=d)
    rc = lib().w4a16_gemm_affine_bits(_ptr(x, _bf16_types(), "x", 2 * M * K, d),
                                      _ptr(scratch, (torch.uint8,), "scratch", sbytes, d),
                                      _ptr(packed, (torch.uint8,), "packed", affine_bits_repacked_bytes(N, K, group, bits),
                                           d),
                                      M, N, K, group, bits, _ptr(out, _bf16_types(), "out", 2 * M * N, d),
                                      _stream(stream, d))
    _check(rc, "w4a16_gemm_affine_bits")
    return out


def dequantize_affine_bits(packed, N, K, group, bits, stream=None):
    """float32 [N, K]: scale * q + bias read back from a b-bit packed weight."""
    torch = _torch()
    d = packed.device
    w = torch.empty((N, K), dtype=torch.float32, device=d)
    rc = lib().w4a16_dequantize_affine_bits(_ptr(packed, (torch.uint8,), "packed",
                                                 affine_bits_repacked_bytes(N, K, group, bits), d),
                                            N, K, group, bits, _ptr(w, (torch.float32,), "w_out", 4 * N * K, d),
                                            _stream(stream, d))
    _check(rc, "w4a16_dequantize_affine_bits")
    return w


def gateup_silu_affine(x, packed_gateup, N_each, K, group, xs=None, out=None, stream=None):
    """h[M, N_each] (bf16) = SiLU(x Wg^T) * (x Wu^T), affine weights."""
    torch = _torch()
    M = _x_rows(x, K)
    d = x.device
    if out is None:
        out = torch.empty((M, N_each), dtype=torch.bfloat16, device=d)
    rc = lib().w4a16_gateup_silu_affine(_ptr(x, _bf16_types(), "x", 0, d), _xs_ptr(xs, M, K, group, d),
                                        _ptr(packed_gateup, (torch.uint8,), "packed",
                                             _packed_bytes(N_each, K, group, AFFINE, True), d),
                                        M, N_each, K, group, _ptr(out, _bf16_types(), "out", 2 * M * N_each, d),
                                        _stream(stream, d))
    _check(rc, "w4a16_gateup_silu_affine")
    return out


def dequantize(packed, N, K, group, sym, stream=None):
    """float32 [N, K] = (q - z) * scale (exact), or scale * q + bias rounded once
    to float32 for sym = AFFINE, read back through the kernels' unpack."""
    torch = _torch()
    d = packed.device
    need = _packed_bytes(N, K, group, int(sym), False)
    p = _ptr(packed, (torch.uint8,), "packed", need, d)
    out = torch.empty((N, K), dtype=torch.float32, device=d)
    rc = lib().w4a16_dequantize(p, N, K, group, int(sym), ctypes.c_void_p(out.data_ptr()), _stream(stream, d))
    _check(rc, "w4a16_dequantize")
    return out


def kernel_status() -> int:
    """Synchronise and return (and clear) the kernels' timeout flag: 0 or -5."""
    return int(lib().w4a16_kernel_status())


def set_kernel_override(which: int) -> int:
    return int(lib().w4a16_set_kernel_override(which))


def set_programmatic_overlap(on: bool) -> bool:
    """Let each M <= 32 call start streaming its weights while the previous
    kernel on the stream finishes (x and y are touched only after it has).
    Only while packed weights are read-only and complete; returns the previous
    setting."""
    prev = int(lib().w4a16_set_programmatic_overlap(int(bool(on))))
    if prev < 0:
        raise W4A16Error("w4a16_set_programmatic_overlap: bad value")
    return bool(prev)
