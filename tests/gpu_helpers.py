"""Shared helpers of the GPU parity tests: upload seeded inputs, run the CUDA
path through the C ABI, and compare with the oracle under the stated bounds."""
from contextlib import contextmanager

import numpy as np

import oracle
import synth

import gemm_w4a16_group_gb300 as w4


def torch():
    import torch as _t
    return _t


def dev(a):
    """numpy -> CUDA tensor; uint16 (bf16 bits) travels as int16."""
    t = torch()
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return t.from_numpy(a).cuda()


def host_bits(y):
    """bf16 CUDA tensor -> uint16 numpy bits."""
    t = torch()
    return y.view(t.int16).cpu().numpy().view(np.uint16)


def bf16_f64(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


@contextmanager
def kernel(which):
    prev = w4.set_kernel_override(which)
    try:
        yield
    finally:
        w4.set_kernel_override(prev)


def upload(p):
    d = {"x": dev(p["x"]), "qweight": dev(p["qweight"]), "scales": dev(p["scales"]),
         "zeros": None if p["zeros"] is None else dev(p["zeros"])}
    for k in ("qweight_up", "scales_up", "zeros_up"):
        if k in p:
            d[k] = None if p[k] is None else dev(p[k])
    return d


def packed_of(p, d):
    return w4.repack(d["qweight"], d["scales"], d["zeros"], p["N"], p["K"], p["group"], p["sym"])


def packed_gateup_of(p, d):
    return w4.repack_gateup(d["qweight"], d["scales"], d["zeros"], d["qweight_up"], d["scales_up"],
                            d["zeros_up"], p["N"], p["K"], p["group"], p["sym"])


def run_gemm(p, which=w4.KERNEL_AUTO, d=None, packed=None, x=None):
    d = d or upload(p)
    packed = packed if packed is not None else packed_of(p, d)
    with kernel(which):
        y = w4.gemm(d["x"] if x is None else x, packed, p["N"], p["K"], p["group"], p["sym"])
    torch().cuda.synchronize()
    assert w4.kernel_status() == 0
    return host_bits(y)


def run_gateup(p, which=w4.KERNEL_AUTO, d=None, packed=None):
    d = d or upload(p)
    packed = packed if packed is not None else packed_gateup_of(p, d)
    with kernel(which):
        h = w4.gateup_silu(d["x"], packed, p["N"], p["K"], p["group"], p["sym"])
    torch().cuda.synchronize()
    assert w4.kernel_status() == 0
    return host_bits(h)


def assert_within(y_bits, ref, bound, what=""):
    y = bf16_f64(y_bits)
    err = np.abs(y - ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        ratio = np.max(err / np.maximum(bound, 1e-300))
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside bound, max err/bound "
                             f"{ratio:.3g}; first {idx.tolist()}: got {y[bad][:5]}, ref {ref[bad][:5]}")
    return float(np.max(err / np.maximum(bound, 1e-300))) if err.size else 0.0


def check_gemm_full(p, y_bits):
    ref, sa = oracle.gemm(p["x"], p["qweight"], p["scales"], p["zeros"], p["M"], p["N"], p["K"],
                          p["group"], p["sym"])
    return assert_within(y_bits, ref, oracle.gemm_bound(ref, sa), "gemm")


def sample_pairs(M, N, count, seed=0):
    """Sampled (m, n) output positions: every corner and edge plus uniform draws."""
    rng = np.random.default_rng(seed)
    ms = [0, M - 1, M // 2]
    ns = [0, 1, 15, 16, N - 1, N - 16, N // 2]
    pairs = {(m, n) for m in ms for n in ns if 0 <= n < N}
    mi = rng.integers(0, M, count)
    ni = rng.integers(0, N, count)
    pairs.update(zip(mi.tolist(), ni.tolist()))
    pairs = sorted(pairs)
    return np.array([a for a, _ in pairs], dtype=np.int64), np.array([b for _, b in pairs], dtype=np.int64)
