"""The affine weight form w = scale * q + bias (the MLX affine 4-bit
checkpoints of TensorFold PR #859) through the C ABI against the float64
oracle: the dequantised read-back is scale * q + bias rounded once to float32,
the group sums of x are float32 sums within their summation bound, and every
matmul output lies within |y - ref| <= 2^-7 |ref| + 1e-5 sum_k |x_k w_nk|
(the fused gate/up output within oracle.silu_bound). Sizes span several tiles
with ragged tails in M, N and K, on the decode kernels (M <= 32, group sums
formed in the kernel) and the tcgen05 GEMM (group sums from w4a16_xsum)."""
import numpy as np
import pytest

import oracle
import synth

import gemm_w4a16_group_gb300 as w4

from gpu_helpers import assert_within, dev, host_bits, kernel, sample_pairs, torch

pytestmark = pytest.mark.gpu

AUTO, SMALLM, TC, XS = w4.KERNEL_AUTO, w4.KERNEL_SMALLM, w4.KERNEL_TC, w4.KERNEL_XSTAGED


def _problem(M, N, K, group, seed, gateup=False):
    return synth.make_problem(M, N, K, group, False, seed=seed, gateup=gateup, affine=True)


def _packed(p, gateup=False):
    if gateup:
        return w4.repack_affine_gateup(dev(p["qweight"]), dev(p["scales"]), dev(p["biases"]),
                                       dev(p["qweight_up"]), dev(p["scales_up"]), dev(p["biases_up"]),
                                       p["N"], p["K"], p["group"])
    return w4.repack_affine(dev(p["qweight"]), dev(p["scales"]), dev(p["biases"]), p["N"], p["K"], p["group"])


def _finish():
    torch().cuda.synchronize()
    assert w4.kernel_status() == 0


@pytest.mark.parametrize("N,K,group", [(250, 512, 64), (64, 1024, 128), (1, 128, 64), (33, 640, 128)])
def test_dequantize_affine(N, K, group):
    p = _problem(1, N, K, group, seed=N + K)
    w = w4.dequantize(_packed(p), N, K, group, w4.AFFINE).cpu().numpy()
    ref = oracle.dequant_affine(p["qweight"], p["scales"], p["biases"], N, K, group)
    # scale * q + bias is one rounding of the exact value (fmaf)
    np.testing.assert_array_equal(w, ref.astype(np.float32))


@pytest.mark.parametrize("M,K,group", [(1, 512, 64), (17, 640, 128), (300, 1024, 64), (256, 256, 128)])
def test_xsum_parity(M, K, group):
    """Three bf16 parts per group whose sum is a float32 sum of the group's x
    (within its summation bound of the exact sum); zeros past 3 * K/G."""
    x = synth.make_x(M, K, seed=M + K)
    xs = w4.xsum(dev(x), K, group)
    _finish()
    parts = synth.bf16_bits_to_f32(host_bits(xs)).astype(np.float64)
    G3 = 3 * (K // group)
    assert parts.shape == (M, (G3 + 63) // 64 * 64)
    assert np.all(parts[:, G3:] == 0.0)
    hi, mid, lo = parts[:, 0:G3:3], parts[:, 1:G3:3], parts[:, 2:G3:3]
    got = hi + mid + lo                                   # exact in float64
    assert np.all(got.astype(np.float32).astype(np.float64) == got)  # a float32 value
    assert np.all(synth.f32_to_bf16_bits(got.astype(np.float32)) == host_bits(xs)[:, 0:G3:3])  # hi = bf16(X)
    ref = oracle.group_sums(x, M, K, group).T              # [M, groups]
    absx = oracle.group_sums(x & np.uint16(0x7FFF), M, K, group).T  # sums of |x|
    assert np.all(np.abs(got - ref) <= group * 2.0 ** -24 * absx)


GEMM_CASES = [
    # (kernel, M, N, K, group)
    (AUTO, 1, 250, 512, 64),
    (AUTO, 1, 1040, 2048, 128),
    (AUTO, 2, 520, 1024, 64),
    (AUTO, 5, 250, 1024, 128),
    (AUTO, 8, 1040, 640, 64),
    (AUTO, 13, 250, 512, 64),
    (AUTO, 16, 520, 2048, 128),
    (AUTO, 16, 32, 5120, 64),       # short N: split K across a cluster
    (SMALLM, 24, 250, 512, 64),
    (SMALLM, 32, 520, 1024, 128),
    (XS, 1, 250, 512, 64),
    (XS, 5, 250, 1024, 128),
    (XS, 16, 520, 2048, 128),
    (XS, 16, 32, 5120, 64),
    (TC, 1, 250, 512, 64),
    (TC, 16, 300, 640, 128),
    (AUTO, 17, 520, 1024, 64),
    (AUTO, 64, 520, 1024, 128),
    (AUTO, 65, 300, 640, 64),
    (AUTO, 128, 520, 1024, 128),
    (AUTO, 200, 520, 1024, 64),
    (AUTO, 513, 1040, 768, 128),
    (AUTO, 600, 700, 1024, 64),
    (AUTO, 48, 300, 2048, 64),      # split K: the bias group on the first pair only
    (AUTO, 256, 250, 4096, 128),
]


@pytest.mark.parametrize("which,M,N,K,group", GEMM_CASES)
def test_gemm_affine_parity(which, M, N, K, group):
    p = _problem(M, N, K, group, seed=M * 11 + N + K)
    x = dev(p["x"])
    packed = _packed(p)
    with kernel(which):
        xs = w4.xsum(x, K, group) if (M > 32 or which == TC) else None
        y = w4.gemm_affine(x, packed, N, K, group, xs)
    _finish()
    ref, sa = oracle.gemm_affine(p["x"], p["qweight"], p["scales"], p["biases"], M, N, K, group)
    assert_within(host_bits(y), ref, oracle.gemm_bound(ref, sa), f"affine M={M}")


@pytest.mark.parametrize("M", [1, 8, 16, 40])
def test_affine_one_hot_x_gives_rounded_weight(M):
    """x = e_k: y[n] = scale * q + bias rounded once to float32, then to bf16."""
    N, K, group = 272, 512, 64
    p = _problem(M, N, K, group, seed=5)
    ks = (np.arange(M) * 97 + 5) % K
    x = np.zeros((M, K), np.uint16)
    x[np.arange(M), ks] = 0x3F80
    xd = dev(x)
    xs = w4.xsum(xd, K, group) if M > 32 else None
    y = w4.gemm_affine(xd, _packed(p), N, K, group, xs)
    _finish()
    w = oracle.dequant_affine(p["qweight"], p["scales"], p["biases"], N, K, group)
    expect = synth.f32_to_bf16_bits(w[:, ks].T.astype(np.float32))
    np.testing.assert_array_equal(host_bits(y), expect)


@pytest.mark.parametrize("which,M,N,K,group", [
    (AUTO, 1, 250, 512, 64), (AUTO, 5, 130, 1024, 128), (AUTO, 16, 300, 640, 64),
    (AUTO, 40, 250, 512, 128), (AUTO, 130, 300, 640, 64), (AUTO, 300, 200, 1024, 128), (TC, 3, 128, 512, 64),
    (XS, 2, 250, 512, 64), (XS, 16, 300, 640, 128)])
def test_gateup_affine_parity(which, M, N, K, group):
    p = _problem(M, N, K, group, seed=M + 3 * N + K, gateup=True)
    x = dev(p["x"])
    packed = _packed(p, gateup=True)
    with kernel(which):
        xs = w4.xsum(x, K, group) if (M > 32 or which == TC) else None
        h = w4.gateup_silu_affine(x, packed, N, K, group, xs)
    _finish()
    mi, ni = np.repeat(np.arange(M), N), np.tile(np.arange(N), M)
    if M * N > 20000:
        mi, ni = sample_pairs(M, N, 4000, seed=M)
    ref, g, u, ga, ua = oracle.gateup_silu_affine_at(p["x"], p["qweight"], p["scales"], p["biases"],
                                                     p["qweight_up"], p["scales_up"], p["biases_up"],
                                                     M, N, K, group, mi, ni)
    got = host_bits(h)[mi, ni]
    assert_within(got, ref, oracle.silu_bound(ref, g, u, ga, ua), f"gateup affine M={M}")


def test_affine_xsum_serves_several_weights():
    """One table of group sums, two weights of different N on the same x."""
    M, K, group = 48, 1024, 64
    pa = _problem(M, 96, K, group, seed=71)
    pb = _problem(M, 400, K, group, seed=72)
    pb["x"] = pa["x"]
    x = dev(pa["x"])
    xs = w4.xsum(x, K, group)
    for p in (pa, pb):
        y = w4.gemm_affine(x, _packed(p), p["N"], K, group, xs)
        _finish()
        ref, sa = oracle.gemm_affine(p["x"], p["qweight"], p["scales"], p["biases"], M, p["N"], K, group)
        assert_within(host_bits(y), ref, oracle.gemm_bound(ref, sa), f"N={p['N']}")
