"""The tcgen05 decode kernel (weights dequantised into tensor memory, x rows
as the MMA's N) through the C ABI against the float64 oracle, under the same
bounds as the other GEMM paths: |y - ref| <= 2^-7 |ref| + 1e-5 sum_k |x_k w_nk|.

Cases span its paths: x padded to 16 and to 32 MMA columns (M = 1-16 and
17-32), persistent CTAs walking more 128-row tiles than fit at once, K split
over 2-8 CTAs of a cluster (few tiles; the split is whole blocks of four
groups), a ragged last 128-k stage (an odd number of 64-k chunks), a ragged
last block of four groups, and N that is not a multiple of 16 or 128.
"""
import numpy as np
import pytest

import oracle
import synth

import gemm_w4a16_group_gb300 as w4

from gpu_helpers import check_gemm_full, dev, packed_of, run_gemm, upload

pytestmark = pytest.mark.gpu

DTC = w4.KERNEL_DECODE_TC

CASES = [
    # (M, N, K, group, sym)
    (1, 250, 512, 128, True),
    (2, 1040, 2048, 64, False),      # K split over 4 CTAs
    (5, 250, 1024, 128, False),
    (8, 520, 2048, 64, True),
    (9, 130, 576, 64, False),        # 9 chunks: a one-chunk last stage
    (13, 250, 512, 64, False),
    (16, 1040, 1024, 128, True),
    (16, 32, 5120, 64, False),       # one partial tile, K split over 8 CTAs
    (17, 520, 1024, 64, False),      # 32 MMA columns
    (24, 250, 512, 128, True),
    (32, 300, 640, 128, True),       # 10 chunks: a ragged last block
    (32, 32, 5120, 64, False),
    (1, 5120, 8704, 128, True),      # 40 tiles, K split over 7 CTAs
    (5, 5120, 5120, 64, False),
    (3, 40000, 128, 64, True),       # 313 tiles: persistent CTAs take two
    (20, 39100, 256, 128, False),
    (2, 39000, 576, 64, False),      # 305 tiles of 9 chunks: ragged stages inside a persistent walk
]


@pytest.mark.parametrize("M,N,K,group,sym", CASES)
def test_decode_tc_parity(M, N, K, group, sym):
    p = synth.make_problem(M, N, K, group, sym, seed=M * 11 + N + K)
    check_gemm_full(p, run_gemm(p, DTC))


@pytest.mark.parametrize("M", [1, 16, 32])
@pytest.mark.parametrize("sym", [True, False])
def test_decode_tc_one_hot_x_gives_rounded_weight(M, sym):
    """x = e_k: y[n] = (q - z) * scale exactly in float32, so y is its bf16
    rounding; a wrong k order of x against the weight in tensor memory shows
    here as the weight of another k."""
    N, K, group = 272, 512, 64
    p = synth.make_problem(M, N, K, group, sym, seed=3)
    ks = (np.arange(M) * 97 + 5) % K
    x = np.zeros((M, K), np.uint16)
    x[np.arange(M), ks] = 0x3F80
    p["x"] = x
    y = run_gemm(p, DTC)
    w = oracle.dequant(p["qweight"], p["scales"], p["zeros"], N, K, group, sym)
    np.testing.assert_array_equal(y, synth.f32_to_bf16_bits(w[:, ks].T.astype(np.float32)))


def test_decode_tc_codes_equal_zero_give_exact_zero():
    M, N, K, group = 5, 96, 512, 128
    p = synth.make_problem(M, N, K, group, False, seed=4)
    zmat = synth.make_codes(N, K // group, 4, 9)
    p["zeros"] = synth.pack_nibbles_rows(zmat)
    p["qweight"] = synth.pack_nibbles_rows(np.repeat(zmat, group, axis=1))
    y = run_gemm(p, DTC)
    assert np.all((y & 0x7FFF) == 0)


@pytest.mark.parametrize("M,N,K", [(5, 520, 1024), (24, 520, 1024), (16, 1040, 4096)])
def test_decode_tc_rows_independent_and_deterministic(M, N, K):
    """Bitwise reproducible (the split-K sum runs in rank order); permuting x
    rows permutes y rows bitwise."""
    p = synth.make_problem(M, N, K, 64, False, seed=5)
    d = upload(p)
    packed = packed_of(p, d)
    y1 = run_gemm(p, DTC, d, packed)
    np.testing.assert_array_equal(y1, run_gemm(p, DTC, d, packed))
    perm = np.random.default_rng(0).permutation(M)
    np.testing.assert_array_equal(run_gemm(p, DTC, d, packed, x=dev(p["x"][perm])), y1[perm])


def test_decode_tc_agrees_with_the_mma_sync_kernel_within_bound():
    p = synth.make_problem(16, 2080, 2048, 128, True, seed=6)
    d = upload(p)
    packed = packed_of(p, d)
    check_gemm_full(p, run_gemm(p, DTC, d, packed))
    check_gemm_full(p, run_gemm(p, w4.KERNEL_SMALLM, d, packed))


@pytest.mark.parametrize("name", ["decode_gateup_m1_k5120_n34816", "decode_down_m1_k17408_n5120",
                                  "smallm_m16_k5120_n34816", "verify_m32_k5120_n34816"])
def test_decode_tc_full_size_sampled(name):
    """The full-size workload through this kernel (as `bench.py --kernel
    decode_tc` times it), on sampled outputs the oracle computes one by one."""
    from synth.workloads import WORKLOADS
    from gpu_helpers import assert_within, sample_pairs
    w = WORKLOADS[name]
    p = synth.make_problem(w["M"], w["N"], w["K"], w["group"], w["sym"], scale_range=w["scale_range"],
                           x_scale=w["x_scale"], seed=0)
    y = run_gemm(p, DTC)
    mi, ni = sample_pairs(p["M"], p["N"], 1500, seed=len(name))
    ref, sa = oracle.gemm_at(p["x"], p["qweight"], p["scales"], p["zeros"], p["M"], p["N"], p["K"], p["group"],
                             p["sym"], mi, ni)
    assert_within(y[mi, ni], ref, oracle.gemm_bound(ref, sa), name)
