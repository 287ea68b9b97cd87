"""CUDA path (through the C ABI) against the float64 oracle.

Bounds: dequantisation is bit-exact; matmul outputs satisfy
|y - ref| <= 2^-7 |ref| + 1e-5 sum_k |x_k w_nk|; the fused SiLU(gate) * up
output satisfies the propagated bound in oracle.silu_bound. Sizes here are
small enough for the oracle to compute every output, and span several tiles
with ragged tails in N (not a multiple of 16 or of the 256-row GEMM tile) and
in M (not a multiple of 8 or of the 128-row GEMM tile).
"""
import numpy as np
import pytest

import oracle
import synth

import gemm_w4a16_group_gb300 as w4

from gpu_helpers import (assert_within, bf16_f64, check_gemm_full, dev, host_bits, kernel,
                         packed_gateup_of, packed_of, run_gateup, run_gemm, torch, upload)

pytestmark = pytest.mark.gpu

GEMV, SMALLM, TC, XS = w4.KERNEL_GEMV, w4.KERNEL_SMALLM, w4.KERNEL_TC, w4.KERNEL_XSTAGED


@pytest.mark.parametrize("sym,group", [(True, 128), (False, 64), (True, 64), (False, 128)])
@pytest.mark.parametrize("N,K", [(250, 512), (64, 1024), (1, 128)])
def test_dequantize_bit_exact(sym, group, N, K):
    if K % group:
        pytest.skip("K % G")
    p = synth.make_problem(1, N, K, group, sym, seed=N + K)
    d = upload(p)
    w = w4.dequantize(packed_of(p, d), N, K, group, sym).cpu().numpy().astype(np.float64)
    ref = oracle.dequant(p["qweight"], p["scales"], p["zeros"], N, K, group, sym)
    np.testing.assert_array_equal(w, ref)



@pytest.mark.parametrize("sym", [False, True])
def test_dequantize_every_code_zero_point_and_scale(sym):
    """Every (code, zero point) pair against every scale of a sweep from
    2^-100 to 2^100 (both signs), read back bit for bit."""
    e = synth.exhaustive_problem(sym)
    N, K, G = e["N"], e["K"], e["group"]
    w = w4.dequantize(packed_of(e, upload(e)), N, K, G, sym).cpu().numpy().astype(np.float64)
    np.testing.assert_array_equal(w, oracle.dequant(e["qweight"], e["scales"], e["zeros"], N, K, G, sym))

CASES = [
    # (kernel, M, N, K, group, sym)
    (GEMV, 1, 250, 512, 128, True),
    (GEMV, 1, 1040, 2048, 64, False),
    (GEMV, 1, 16, 17408 // 8, 128, True),
    (SMALLM, 1, 250, 512, 128, True),
    (SMALLM, 2, 1040, 2048, 64, False),
    (SMALLM, 5, 250, 1024, 128, False),
    (SMALLM, 8, 520, 2048, 64, True),
    (SMALLM, 13, 250, 512, 64, False),
    (SMALLM, 16, 1040, 1024, 128, True),
    (SMALLM, 16, 32, 5120, 64, False),
    # 17-32 rows on the small-M kernel (three and four n8 tiles of x rows)
    (SMALLM, 17, 520, 1024, 64, False),
    (SMALLM, 24, 250, 512, 128, True),
    (SMALLM, 25, 1040, 2048, 64, False),
    (SMALLM, 32, 300, 640, 128, True),
    (SMALLM, 32, 32, 5120, 64, False),
    # the small-M kernel that stages x once per CTA: one CTA (8 tiles), ragged
    # N, cluster split-K on short N, a ragged last K unit (K = 640, 1088)
    (XS, 1, 250, 512, 128, True),
    (XS, 2, 1040, 2048, 64, False),
    (XS, 5, 250, 1024, 128, False),
    (XS, 8, 520, 2048, 64, True),
    (XS, 9, 130, 640, 64, False),
    (XS, 13, 250, 512, 64, False),
    (XS, 16, 1040, 1024, 128, True),
    (XS, 16, 32, 5120, 64, False),
    (XS, 16, 2100, 1088, 64, True),
    (TC, 1, 250, 512, 128, True),
    (TC, 17, 520, 1024, 64, False),
    (TC, 200, 520, 1024, 128, True),
    (TC, 130, 300, 640, 64, False),
    (TC, 256, 512, 512, 128, False),
    # the 64- and 128-row x tiles of short M, at and across their boundaries
    (TC, 64, 520, 1024, 128, True),
    (TC, 65, 300, 640, 64, False),
    (TC, 100, 1040, 768, 64, True),
    (TC, 128, 520, 1024, 128, False),
    # several 256 x 256 pair tiles in both directions, ragged in M and N
    (TC, 600, 700, 1024, 64, True),
    (TC, 513, 1040, 768, 128, False),
    # few tiles: K split across 2, 3 or 4 pairs of a cluster (blocks of four
    # groups each), the partial sums added over distributed shared memory
    (TC, 64, 300, 2048, 64, False),
    (TC, 100, 1040, 1536, 64, True),
    (TC, 300, 250, 4096, 128, False),
    (TC, 40, 5120, 1024, 64, True),
]


@pytest.mark.parametrize("which,M,N,K,group,sym", CASES)
def test_gemm_parity(which, M, N, K, group, sym):
    p = synth.make_problem(M, N, K, group, sym, seed=M * 7 + N + K)
    y = run_gemm(p, which)
    check_gemm_full(p, y)


@pytest.mark.parametrize("which,M", [(GEMV, 1), (SMALLM, 1), (SMALLM, 8), (SMALLM, 16), (XS, 3), (XS, 16), (TC, 40)])
@pytest.mark.parametrize("sym", [True, False])
def test_one_hot_x_gives_rounded_weight(which, M, sym):
    """x = e_k: y[n] = (q - z) * scale exactly in float32, so y is its bf16 rounding."""
    N, K, group = 272, 512, 64
    p = synth.make_problem(M, N, K, group, sym, seed=3)
    ks = (np.arange(M) * 97 + 5) % K
    x = np.zeros((M, K), np.uint16)
    x[np.arange(M), ks] = 0x3F80
    p["x"] = x
    y = run_gemm(p, which)
    w = oracle.dequant(p["qweight"], p["scales"], p["zeros"], N, K, group, sym)
    expect = synth.f32_to_bf16_bits(w[:, ks].T.astype(np.float32))
    np.testing.assert_array_equal(y, expect)


@pytest.mark.parametrize("which,M", [(GEMV, 1), (SMALLM, 5), (TC, 33)])
def test_codes_equal_zero_give_exact_zero(which, M):
    N, K, group = 96, 512, 128
    p = synth.make_problem(M, N, K, group, False, seed=4)
    zmat = synth.make_codes(N, K // group, 4, 9)
    p["zeros"] = synth.pack_nibbles_rows(zmat)
    p["qweight"] = synth.pack_nibbles_rows(np.repeat(zmat, group, axis=1))
    y = run_gemm(p, which)
    assert np.all((y & 0x7FFF) == 0)


@pytest.mark.parametrize("which,M", [(SMALLM, 16), (SMALLM, 5), (XS, 16), (XS, 5), (TC, 150)])
def test_rows_independent_and_deterministic(which, M):
    """Runs are bitwise reproducible; permuting x rows permutes y rows bitwise."""
    N, K, group = 520, 1024, 64
    p = synth.make_problem(M, N, K, group, False, seed=5)
    d = upload(p)
    packed = packed_of(p, d)
    y1 = run_gemm(p, which, d, packed)
    y2 = run_gemm(p, which, d, packed)
    np.testing.assert_array_equal(y1, y2)
    perm = np.random.default_rng(0).permutation(M)
    yp = run_gemm(p, which, d, packed, x=dev(p["x"][perm]))
    np.testing.assert_array_equal(yp, y1[perm])


def test_gemv_and_smallm_agree_within_bound():
    p = synth.make_problem(1, 2080, 4096, 128, True, seed=6)
    d = upload(p)
    packed = packed_of(p, d)
    a = run_gemm(p, GEMV, d, packed)
    b = run_gemm(p, SMALLM, d, packed)
    check_gemm_full(p, a)
    check_gemm_full(p, b)


GATEUP_CASES = [
    (SMALLM, 1, 136, 512, 128, True),
    (SMALLM, 5, 300, 1024, 64, False),
    (SMALLM, 16, 128, 2048, 128, True),
    (SMALLM, 20, 136, 512, 128, True),
    (SMALLM, 32, 300, 1024, 64, False),
    (TC, 40, 136, 2048, 64, False),
    (TC, 200, 300, 3072, 128, True),
    (XS, 1, 136, 512, 128, True),
    (XS, 5, 300, 1024, 64, False),
    (XS, 16, 128, 2048, 128, True),
    (TC, 17, 136, 512, 64, False),
    (TC, 64, 300, 1024, 64, False),
    (TC, 120, 136, 512, 128, True),
    (TC, 200, 300, 1024, 128, True),
    (TC, 300, 200, 768, 64, True),
]


@pytest.mark.parametrize("which,M,N,K,group,sym", GATEUP_CASES)
def test_gateup_silu_parity(which, M, N, K, group, sym):
    p = synth.make_problem(M, N, K, group, sym, seed=M + N, gateup=True)
    h = run_gateup(p, which)
    mi, ni = np.repeat(np.arange(M), N), np.tile(np.arange(N), M)
    ref, g, u, ga, ua = oracle.gateup_silu_at(p["x"], p["qweight"], p["scales"], p["zeros"],
                                              p["qweight_up"], p["scales_up"], p["zeros_up"],
                                              M, N, K, group, sym, mi, ni)
    assert_within(h.reshape(-1), ref, oracle.silu_bound(ref, g, u, ga, ua), "gateup")


def test_gateup_buffer_is_a_plain_repack_of_interleaved_rows():
    """The gate/up buffer read as an ordinary weight gives gate and up rows
    alternating in 16-row tiles."""
    M, N, K, group = 3, 128, 512, 128
    p = synth.make_problem(M, N, K, group, True, seed=8, gateup=True)
    d = upload(p)
    pg = packed_gateup_of(p, d)
    y = host_bits(w4.gemm(d["x"], pg, 2 * N, K, group, True))
    yg = run_gemm(p, SMALLM, d)
    pu = dict(p, qweight=p["qweight_up"], scales=p["scales_up"], zeros=p["zeros_up"])
    yu = run_gemm(pu, SMALLM)
    inter = y.reshape(M, N // 16, 2, 16)
    np.testing.assert_array_equal(inter[:, :, 0].reshape(M, N), yg)
    np.testing.assert_array_equal(inter[:, :, 1].reshape(M, N), yu)


ARGMAX_CASES = [
    # (M, N, K, group, sym): one tile pair, ragged N, cluster split-K, tcgen05 path
    (1, 250, 512, 128, True),
    (5, 1040, 2048, 64, False),
    (16, 520, 5120, 64, False),
    (1, 96, 17408, 128, True),
    (24, 300, 640, 128, True),
    (40, 300, 640, 128, True),
]


@pytest.mark.parametrize("which", [w4.KERNEL_AUTO, XS])
@pytest.mark.parametrize("M,N,K,group,sym", ARGMAX_CASES)
def test_gemm_argmax_matches_first_max_of_y(M, N, K, group, sym, which):
    """Fused argmax = numpy's first maximum of the bf16 row that w4a16_gemm
    writes (which is torch.argmax's choice), with and without stored logits."""
    p = synth.make_problem(M, N, K, group, sym, seed=70 + M + N)
    d = upload(p)
    packed = packed_of(p, d)
    y = bf16_f64(run_gemm(p, which, d=d, packed=packed))
    want = np.argmax(y, axis=1)
    with kernel(which):
        a1, y1 = w4.gemm_argmax(d["x"], packed, N, K, group, sym, logits=True)
        a2, y2 = w4.gemm_argmax(d["x"], packed, N, K, group, sym)
    torch().cuda.synchronize()
    assert w4.kernel_status() == 0
    np.testing.assert_array_equal(a1.cpu().numpy(), want)
    np.testing.assert_array_equal(a2.cpu().numpy(), want)
    np.testing.assert_array_equal(bf16_f64(host_bits(y1)), y)
    assert (y2 is None) == (M <= 32)


@pytest.mark.parametrize("M", [1, 7, 30])
def test_gemm_argmax_ties_pick_the_first_column(M):
    """Rows of equal weights give equal outputs: the lowest such column wins.
    Weight rows 40..47 repeat row 40 of a weight whose other rows are scaled
    down, so each x row's maximum is shared by columns 40..47 (or is lower)."""
    N, K, group = 200, 512, 64
    p = synth.make_problem(M, N, K, group, True, seed=81)
    q, sc = p["qweight"].copy(), p["scales"].copy()
    q[40:48] = q[40]
    sc[40:48] = sc[40]
    # x = the sign pattern of row 40's dequantised weight, so row 40 is the largest dot product
    w40 = oracle.dequant(q[40:41], sc[40:41], None, 1, K, group, True)[0]
    x = np.tile(np.where(w40 >= 0, 0x3F80, 0xBF80).astype(np.uint16), (M, 1))
    pp = dict(p, qweight=q, scales=sc, x=x)
    d = upload(pp)
    packed = packed_of(pp, d)
    y = bf16_f64(run_gemm(pp, d=d, packed=packed))
    a, _ = w4.gemm_argmax(d["x"], packed, N, K, group, True, logits=M > 32)
    torch().cuda.synchronize()
    got = a.cpu().numpy()
    np.testing.assert_array_equal(got, np.argmax(y, axis=1))
    assert (got == 40).all()


DEGENERATE_KERNELS = [(GEMV, 1), (SMALLM, 1), (SMALLM, 7), (SMALLM, 16), (XS, 2), (XS, 16), (TC, 20), (TC, 300)]


@pytest.mark.parametrize("which,M", DEGENERATE_KERNELS)
def test_zero_scales_or_zero_x_give_exact_zero(which, M):
    """w = (q - z) * 0 = 0, and x = 0, each give y = +-0 exactly."""
    N, K, group = 72, 256, 64
    p = synth.make_problem(M, N, K, group, False, seed=90 + M)
    y = run_gemm(dict(p, scales=np.zeros_like(p["scales"])), which)
    assert np.all((y & 0x7FFF) == 0)
    y = run_gemm(dict(p, x=np.zeros_like(p["x"])), which)
    assert np.all((y & 0x7FFF) == 0)


@pytest.mark.parametrize("which,M", DEGENERATE_KERNELS)
@pytest.mark.parametrize("N,K,group,sym", [(1, 64, 64, True), (17, 64, 64, False), (1, 128, 128, False)])
def test_smallest_shapes(which, M, N, K, group, sym):
    """One output row and/or one 64-wide K chunk (a single group)."""
    p = synth.make_problem(M, N, K, group, sym, seed=95 + N + K)
    check_gemm_full(p, run_gemm(p, which))



@pytest.mark.parametrize("M,N", [(1, 248320), (5, 248320), (40, 4096)])
def test_argmax_finds_a_planted_maximum(M, N):
    """On the output-vocabulary head shape, x rows of +1 and -1 and one weight
    row per x row recoded to agree with it in sign: the greedy pick of every
    row is its planted column (decode epilogue for M <= 32; stored logits and
    the row argmax for M = 40)."""
    K, G = 5120, 128
    planted = [(7919 * (m + 1)) % N for m in range(M)]
    p = synth.planted_max_problem(M, N, K, G, planted, seed=M)
    d = upload(p)
    idx, _ = w4.gemm_argmax(d["x"], packed_of(p, d), N, K, G, True)
    torch().cuda.synchronize()
    assert w4.kernel_status() == 0
    assert idx.cpu().numpy().tolist() == planted
