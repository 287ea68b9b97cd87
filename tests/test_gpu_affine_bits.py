"""Affine weights of 2 to 8 bits (TensorFold PR #859: modules of 2 to 8
bits, every code keeping its value, scale and bias) through the C ABI against
the float64 oracle. 2- and 3-bit codes run widened in the 4-bit tiles, 5- to
8-bit codes as two nibble planes over a doubled K with x's groups repeated:
the read-back is scale * q + bias rounded once to float32, and every matmul
output lies within |y - ref| <= 2^-7 |ref| + 1e-5 sum_k |x_k w_nk|, on the
decode kernels (M <= 32) and the tcgen05 GEMM (M > 32), with ragged N and
K and a K whose bit stream runs across word boundaries."""
import numpy as np
import pytest

import oracle
import synth

import gemm_w4a16_group_gb300 as w4

from gpu_helpers import assert_within, dev, host_bits, kernel, torch

pytestmark = pytest.mark.gpu

BITS = [2, 3, 5, 6, 7, 8]


def problem(M, N, K, group, bits, seed):
    codes = synth.make_codes_bits(N, K, bits, seed)
    return dict(codes=codes, qweight=synth.pack_bits_rows(codes, bits),
                scales=synth.make_scales(N, K // group, 0.005, 0.02, seed),
                biases=synth.make_biases(N, K // group, -0.16, -0.04, seed), x=synth.make_x(M, K, seed))


def packed_of(p, N, K, group, bits):
    return w4.repack_affine_bits(dev(p["qweight"].view(np.int32)), dev(p["scales"]), dev(p["biases"]), N, K, group,
                                 bits)


def finish():
    torch().cuda.synchronize()
    assert w4.kernel_status() == 0


@pytest.mark.parametrize("bits", BITS + [4])
@pytest.mark.parametrize("N,K,group", [(250, 512, 64), (33, 640, 128)])
def test_dequantize_affine_bits(bits, N, K, group):
    p = problem(1, N, K, group, bits, seed=bits + N)
    w = w4.dequantize_affine_bits(packed_of(p, N, K, group, bits), N, K, group, bits).cpu().numpy()
    ref = oracle.dequant_affine_bits(p["qweight"], p["scales"], p["biases"], N, K, group, bits)
    np.testing.assert_array_equal(w, ref.astype(np.float32))  # one rounding of the exact value


CASES = [
    # (M, N, K, group): decode kernels, then the tcgen05 GEMM (split K on few tiles included)
    (1, 250, 512, 64),
    (5, 520, 1024, 128),
    (16, 300, 640, 64),
    (32, 250, 512, 128),
    (40, 250, 512, 128),
    (300, 520, 1024, 64),
    (64, 300, 2048, 64),
]


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("M,N,K,group", CASES)
def test_gemm_affine_bits_parity(bits, M, N, K, group):
    p = problem(M, N, K, group, bits, seed=M * 3 + N + bits)
    y = w4.gemm_affine_bits(dev(p["x"]), packed_of(p, N, K, group, bits), N, K, group, bits)
    finish()
    ref, sa = oracle.gemm_affine_bits(p["x"], p["qweight"], p["scales"], p["biases"], M, N, K, group, bits)
    assert_within(host_bits(y), ref, oracle.gemm_bound(ref, sa), f"bits={bits} M={M}")


@pytest.mark.parametrize("bits", [3, 8])
@pytest.mark.parametrize("which,M", [(w4.KERNEL_XSTAGED, 5), (w4.KERNEL_TC, 16), (w4.KERNEL_SMALLM, 24)])
def test_gemm_affine_bits_forced_kernels(bits, which, M):
    N, K, group = 272, 1024, 64
    p = problem(M, N, K, group, bits, seed=90 + M + bits)
    with kernel(which):
        y = w4.gemm_affine_bits(dev(p["x"]), packed_of(p, N, K, group, bits), N, K, group, bits)
    finish()
    ref, sa = oracle.gemm_affine_bits(p["x"], p["qweight"], p["scales"], p["biases"], M, N, K, group, bits)
    assert_within(host_bits(y), ref, oracle.gemm_bound(ref, sa), f"forced {which}")


def test_four_bits_equal_the_nibble_entry_point():
    """At 4 bits the bit stream is the nibble packing: bitwise the output of
    w4a16_gemm_affine on the same weight."""
    M, N, K, group = 40, 300, 640, 64
    p = problem(M, N, K, group, 4, seed=5)
    x = dev(p["x"])
    y = w4.gemm_affine_bits(x, packed_of(p, N, K, group, 4), N, K, group, 4)
    pa = w4.repack_affine(dev(synth.pack_nibbles_rows(p["codes"])), dev(p["scales"]), dev(p["biases"]), N, K, group)
    y4 = w4.gemm_affine(x, pa, N, K, group, w4.xsum(x, K, group))
    finish()
    np.testing.assert_array_equal(host_bits(y), host_bits(y4))


def test_scratch_reused_across_calls():
    """One scratch buffer, two calls in a row on different x: each output
    follows its own x."""
    M, N, K, group, bits = 48, 250, 512, 64, 6
    pa = problem(M, N, K, group, bits, seed=11)
    xb = synth.make_x(M, K, 12)
    packed = packed_of(pa, N, K, group, bits)
    t = torch()
    scratch = t.empty(w4.affine_bits_scratch_bytes(M, K, group, bits), dtype=t.uint8, device="cuda")
    ya = w4.gemm_affine_bits(dev(pa["x"]), packed, N, K, group, bits, scratch=scratch)
    yb = w4.gemm_affine_bits(dev(xb), packed, N, K, group, bits, scratch=scratch)
    finish()
    for x, y in ((pa["x"], ya), (xb, yb)):
        ref, sa = oracle.gemm_affine_bits(x, pa["qweight"], pa["scales"], pa["biases"], M, N, K, group, bits)
        assert_within(host_bits(y), ref, oracle.gemm_bound(ref, sa), "scratch reuse")
