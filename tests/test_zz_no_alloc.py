"""w4a16_gemm_affine_noalloc: the affine GEMM with its group sums in the
library's fixed device array instead of a caller's table. Two consecutive
calls must give exactly the bits of w4a16_gemm_affine with a caller-owned
table (same kernels, same inputs), on the tcgen05 path (M > 32, the array in
use) and the decode path (M <= 32, no table), and lie within the oracle's
bound. Collected last, so it also runs after every other test has used the
library in the same process."""
import ctypes

import numpy as np
import pytest

import oracle
import synth

import gemm_w4a16_group_gb300 as w4

from gpu_helpers import assert_within, dev, host_bits, torch


def test_noalloc_rejects_tables_over_4_mib():
    L = w4.lib()
    P = ctypes.c_void_p
    fake = 1 << 20
    # K = 5120, group 64: M rows of 256 bf16 parts; 4 MiB holds M <= 8,192
    assert w4.xsum_bytes(8192, 5120, 64) <= 4 << 20 < w4.xsum_bytes(8193, 5120, 64)
    assert L.w4a16_gemm_affine_noalloc(P(fake), P(fake), 8193, 64, 5120, 64, P(fake), None) == -1
    assert L.w4a16_gemm_affine_noalloc(None, P(fake), 17, 64, 128, 64, P(fake), None) == -1
    assert L.w4a16_gemm_affine_noalloc(P(fake + 8), P(fake), 17, 64, 128, 64, P(fake), None) == -2


@pytest.mark.gpu
@pytest.mark.parametrize("M,N,K,group", [(300, 520, 1024, 64), (33, 250, 640, 128), (5, 250, 1024, 64)])
def test_noalloc_matches_the_table_entry_point(M, N, K, group):
    p = synth.make_problem(M, N, K, group, False, seed=M + N, affine=True)
    x = dev(p["x"])
    packed = w4.repack_affine(dev(p["qweight"]), dev(p["scales"]), dev(p["biases"]), N, K, group)
    xs = w4.xsum(x, K, group) if M > 32 else None
    y_ref = w4.gemm_affine(x, packed, N, K, group, xs)
    y1 = w4.gemm_affine_noalloc(x, packed, N, K, group)
    y2 = w4.gemm_affine_noalloc(x, packed, N, K, group)
    torch().cuda.synchronize()
    assert w4.kernel_status() == 0
    b_ref, b1, b2 = host_bits(y_ref), host_bits(y1), host_bits(y2)
    np.testing.assert_array_equal(b1, b_ref)
    np.testing.assert_array_equal(b2, b_ref)
    ref, sa = oracle.gemm_affine(p["x"], p["qweight"], p["scales"], p["biases"], M, N, K, group)
    assert_within(b1, ref, oracle.gemm_bound(ref, sa), "noalloc")


@pytest.mark.gpu
def test_noalloc_consecutive_calls_on_different_x():
    """The second call's table replaces the first's: outputs follow each call's own x."""
    M, N, K, group = 64, 300, 512, 64
    pa = synth.make_problem(M, N, K, group, False, seed=91, affine=True)
    pb = synth.make_problem(M, N, K, group, False, seed=92, affine=True)
    packed = w4.repack_affine(dev(pa["qweight"]), dev(pa["scales"]), dev(pa["biases"]), N, K, group)
    ya = w4.gemm_affine_noalloc(dev(pa["x"]), packed, N, K, group)
    yb = w4.gemm_affine_noalloc(dev(pb["x"]), packed, N, K, group)
    torch().cuda.synchronize()
    for x, y in ((pa["x"], ya), (pb["x"], yb)):
        ref, sa = oracle.gemm_affine(x, pa["qweight"], pa["scales"], pa["biases"], M, N, K, group)
        assert_within(host_bits(y), ref, oracle.gemm_bound(ref, sa), "noalloc x")


@pytest.mark.gpu
def test_noalloc_at_the_4_mib_limit():
    """A table of exactly 4 MiB (M = 8,192 rows at K = 5120, group 64): the
    last rows of the fixed array are written and read. Bitwise equal to the
    table entry point on two consecutive calls, and within the oracle's bound
    on sampled outputs."""
    M, N, K, group = 8192, 64, 5120, 64
    assert w4.xsum_bytes(M, K, group) == 4 << 20
    p = synth.make_problem(M, N, K, group, False, seed=17, affine=True)
    x = dev(p["x"])
    packed = w4.repack_affine(dev(p["qweight"]), dev(p["scales"]), dev(p["biases"]), N, K, group)
    y_ref = w4.gemm_affine(x, packed, N, K, group, w4.xsum(x, K, group))
    y1 = w4.gemm_affine_noalloc(x, packed, N, K, group)
    y2 = w4.gemm_affine_noalloc(x, packed, N, K, group)
    torch().cuda.synchronize()
    assert w4.kernel_status() == 0
    b_ref = host_bits(y_ref)
    np.testing.assert_array_equal(host_bits(y1), b_ref)
    np.testing.assert_array_equal(host_bits(y2), b_ref)
    mi = np.concatenate([np.arange(M - 8, M), np.arange(0, M, 97)]).astype(np.int64)
    mi = np.repeat(mi, 4)
    ni = np.tile(np.array([0, 17, 40, N - 1], dtype=np.int64), mi.size // 4)
    ref, sa = oracle.gemm_affine_at(p["x"], p["qweight"], p["scales"], p["biases"], M, N, K, group, mi, ni)
    assert_within(b_ref[mi, ni], ref, oracle.gemm_bound(ref, sa), "noalloc 4 MiB")
