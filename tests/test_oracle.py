"""Pins of the CPU oracle against facts that do not come from the oracle itself.

* a hand-worked example (tests/golden/dequant_worked_example.txt);
* exact rational brute force on tiny inputs (fractions.Fraction: every bf16
  value and every product is a dyadic rational, so the exact sum is known and
  the float64 oracle must sit within the float64 summation bound of it);
* closed forms: all codes equal to the zero point give y = 0; constant codes
  give (c - z) * sum_g s_g * sum_{k in g} x_k; a one-hot x selects one
  dequantised weight exactly; power-of-two scaling of the scales scales y
  exactly;
* the logistic function's textbook value sigma(1) = e / (1 + e) for SiLU.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "dequant_worked_example.txt")


def _load_golden():
    d = {}
    with open(GOLDEN) as f:
        for line in f:
            if line.startswith("#") or ":" not in line:
                continue
            k, v = line.split(":", 1)
            d[k.strip()] = v.split()
    N, K, G = int(d["N"][0]), int(d["K"][0]), int(d["G"][0])
    q = np.array([int(h, 16) for h in d["qweight"]], dtype=np.uint32).view(np.int32).reshape(N, K // 8)
    s = np.array([int(h, 16) for h in d["scales"]], dtype=np.uint16).reshape(N, K // G)
    z = np.array([int(h, 16) for h in d["zeros"]], dtype=np.uint32).view(np.int32).reshape(N, -1)
    x = np.array([int(h, 16) for h in d["x"]], dtype=np.uint16).reshape(-1, K)
    f = lambda key: np.array([float(v) for v in d[key]])
    return dict(N=N, K=K, G=G, q=q, s=s, z=z, x=x, w_sym=f("w_sym").reshape(N, K),
                w_asym=f("w_asym").reshape(N, K), y_sym=f("y_sym").reshape(-1, N),
                y_asym=f("y_asym").reshape(-1, N))


def test_golden_codes_nibble_order():
    g = _load_golden()
    codes = [[oracle.code(g["q"], g["K"], n, k) for k in range(g["K"])] for n in range(g["N"])]
    assert codes[0] == list(range(16))
    assert codes[1] == [7, 6, 5, 4, 3, 2, 1, 0, 15, 14, 13, 12, 11, 10, 9, 8]
    assert [oracle.zero(g["z"], 2, False, 0, j) for j in range(2)] == [3, 12]
    assert [oracle.zero(g["z"], 2, False, 1, j) for j in range(2)] == [0, 15]
    assert oracle.zero(g["z"], 2, True, 1, 1) == 8


@pytest.mark.parametrize("sym", [True, False])
def test_golden_dequant_and_gemm(sym):
    g = _load_golden()
    z = None if sym else g["z"]
    w = oracle.dequant(g["q"], g["s"], z, g["N"], g["K"], g["G"], sym)
    np.testing.assert_array_equal(w, g["w_sym"] if sym else g["w_asym"])
    y, a = oracle.gemm(g["x"], g["q"], g["s"], z, 2, g["N"], g["K"], g["G"], sym)
    np.testing.assert_array_equal(y, g["y_sym"] if sym else g["y_asym"])
    # sum |x w| of the first row (x = 1) is the sum of |w| over the row
    np.testing.assert_array_equal(a[0], np.abs(w).sum(axis=1))


# --------------------------------------------------------------------------
# exact rational brute force

def _fr_bf16(bits):
    return Fraction(float(synth.bf16_bits_to_f32(np.array([bits], dtype=np.uint16))[0]))


def _brute(codes, zeros_mat, scales, x, G):
    """Exact y[m][n] from the unpacked code / zero matrices (never from packed words)."""
    M, K = x.shape
    N = codes.shape[0]
    xs = [[_fr_bf16(x[m, k]) for k in range(K)] for m in range(M)]
    y = [[Fraction(0)] * N for _ in range(M)]
    a = [[Fraction(0)] * N for _ in range(M)]
    for n in range(N):
        w = [(int(codes[n, k]) - int(zeros_mat[n, k // G])) * _fr_bf16(scales[n, k // G])
             for k in range(K)]
        for m in range(M):
            y[m][n] = sum((xs[m][k] * w[k] for k in range(K)), Fraction(0))
            a[m][n] = sum((abs(xs[m][k] * w[k]) for k in range(K)), Fraction(0))
    return y, a


# (False, 8, 2, 3, 80) and (False, 16, 1, 5, 272): 10 and 17 groups per row,
# so each row's zero points span two and three int32 words, the last one part
# used (a wrong word stride or nibble index shows up only past 8 groups)
@pytest.mark.parametrize("sym,G,M,N,K", [(True, 8, 3, 5, 32), (False, 8, 2, 4, 64),
                                         (False, 16, 3, 3, 48), (True, 64, 1, 2, 128),
                                         (False, 8, 2, 3, 80), (False, 16, 1, 5, 272)])
def test_bruteforce_exact(sym, G, M, N, K, seed=None):
    seed = 11 + K + N if seed is None else seed
    codes = synth.make_codes(N, K, seed, 2)
    Kg = K // G
    zmat = (np.full((N, Kg), 8, dtype=np.uint8) if sym
            else synth.make_codes(N, Kg, seed, 4))
    q = synth.pack_nibbles_rows(codes)
    z = None if sym else synth.pack_nibbles_rows(zmat)
    s = synth.make_scales(N, Kg, 0.005, 0.02, seed)
    x = synth.make_x(M, K, seed)
    y, a = oracle.gemm(x, q, s, z, M, N, K, G, sym)
    ye, ae = _brute(codes, zmat, s, x, G)
    gamma = 1.01 * K * 2.0 ** -53
    for m in range(M):
        for n in range(N):
            err = abs(Fraction(y[m, n]) - ye[m][n])
            assert err <= gamma * ae[m][n], (m, n, float(err))
            assert abs(Fraction(a[m, n]) - ae[m][n]) <= gamma * ae[m][n]


def test_bruteforce_random_shapes():
    """The same exact comparison over random shapes (1-20 groups of 8 or 16,
    so zero points in one to three int32 words per row), forms and seeds."""
    hyp = pytest.importorskip("hypothesis")
    st = hyp.strategies

    @hyp.settings(max_examples=120, deadline=None, derandomize=True)
    @hyp.given(sym=st.booleans(), G=st.sampled_from([8, 16]), M=st.integers(1, 3), N=st.integers(2, 4),
               Kg=st.integers(1, 20), seed=st.integers(0, 2**31 - 1))
    def run(sym, G, M, N, Kg, seed):
        test_bruteforce_exact(sym, G, M, N, G * Kg, seed=seed)

    run()


def test_bruteforce_detects_transposed_weight():
    """A weight read transposed (w[k][n] for w[n][k]) must disagree with the exact sum."""
    N = K = 16
    codes = synth.make_codes(N, K, 5, 2)
    s = np.full((N, 2), 0x3F80, dtype=np.uint16)  # 1.0
    x = synth.make_x(1, K, 5)
    ye, _ = _brute(codes.T.copy(), np.full((N, 2), 8), s, x, 8)
    y, _ = oracle.gemm(x, synth.pack_nibbles_rows(codes), s, None, 1, N, K, 8, True)
    assert any(abs(Fraction(y[0, n]) - ye[0][n]) > 0 for n in range(N))


# --------------------------------------------------------------------------
# closed forms

@pytest.mark.parametrize("sym", [True, False])
def test_codes_equal_zero_give_zero(sym):
    M, N, K, G = 3, 24, 256, 64
    Kg = K // G
    zmat = np.full((N, Kg), 8, np.uint8) if sym else synth.make_codes(N, Kg, 3, 4)
    codes = np.repeat(zmat, G, axis=1)
    q = synth.pack_nibbles_rows(codes)
    z = None if sym else synth.pack_nibbles_rows(zmat)
    s = synth.make_scales(N, Kg, 0.005, 0.02, 3)
    x = synth.make_x(M, K, 3)
    y, a = oracle.gemm(x, q, s, z, M, N, K, G, sym)
    assert np.all(y == 0.0) and np.all(a == 0.0)


@pytest.mark.parametrize("c,sym", [(0, True), (15, True), (11, False), (3, False)])
def test_constant_code_closed_form(c, sym):
    M, N, K, G = 2, 16, 512, 128
    Kg = K // G
    codes = np.full((N, K), c, np.uint8)
    zmat = np.full((N, Kg), 8, np.uint8) if sym else synth.make_codes(N, Kg, 9, 4)
    q = synth.pack_nibbles_rows(codes)
    z = None if sym else synth.pack_nibbles_rows(zmat)
    s = synth.make_scales(N, Kg, 0.005, 0.02, 9)
    x = synth.make_x(M, K, 9)
    y, a = oracle.gemm(x, q, s, z, M, N, K, G, sym)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    sf = synth.bf16_bits_to_f32(s).astype(np.float64)
    xg = xf.reshape(M, Kg, G).sum(axis=2)                    # sum_{k in g} x_k
    expect = (c - zmat.astype(np.float64))[None] * sf[None] * xg[:, None, :]
    expect = expect.sum(axis=2)                              # sum over groups
    tol = 2 * K * 2.0 ** -53 * a
    assert np.all(np.abs(y - expect) <= tol + 1e-300)


@pytest.mark.parametrize("sym", [True, False])
def test_one_hot_x_selects_weight(sym):
    N, K, G = 20, 256, 64
    Kg = K // G
    codes = synth.make_codes(N, K, 21, 2)
    zmat = np.full((N, Kg), 8, np.uint8) if sym else synth.make_codes(N, Kg, 21, 4)
    q = synth.pack_nibbles_rows(codes)
    z = None if sym else synth.pack_nibbles_rows(zmat)
    s = synth.make_scales(N, Kg, 0.005, 0.02, 21)
    ks = [0, 7, 64, 131, 255]
    x = np.zeros((len(ks), K), np.uint16)
    for i, k in enumerate(ks):
        x[i, k] = 0x3F80  # 1.0
    y, _ = oracle.gemm(x, q, s, z, len(ks), N, K, G, sym)
    sf = synth.bf16_bits_to_f32(s).astype(np.float64)
    for i, k in enumerate(ks):
        expect = (codes[:, k].astype(np.float64) - zmat[:, k // G]) * sf[:, k // G]
        np.testing.assert_array_equal(y[i], expect)


def test_power_of_two_scale_scales_output_exactly():
    M, N, K, G = 2, 12, 256, 128
    p = synth.make_problem(M, N, K, G, False, seed=4)
    y1, _ = oracle.gemm(p["x"], p["qweight"], p["scales"], p["zeros"], M, N, K, G, False)
    s2 = (p["scales"].astype(np.uint32) + (1 << 7)).astype(np.uint16)  # exponent + 1 -> x2
    y2, _ = oracle.gemm(p["x"], p["qweight"], s2, p["zeros"], M, N, K, G, False)
    np.testing.assert_array_equal(y2, 2.0 * y1)


def test_threads_do_not_change_results():
    p = synth.make_problem(3, 40, 512, 64, False, seed=6)
    args = (p["x"], p["qweight"], p["scales"], p["zeros"], 3, 40, 512, 64, False)
    y1, a1 = oracle.gemm(*args, nthreads=1)
    y8, a8 = oracle.gemm(*args, nthreads=0)
    np.testing.assert_array_equal(y1, y8)
    np.testing.assert_array_equal(a1, a8)


def test_gemm_at_matches_full():
    p = synth.make_problem(5, 48, 256, 64, False, seed=8)
    args = (p["x"], p["qweight"], p["scales"], p["zeros"], 5, 48, 256, 64, False)
    y, a = oracle.gemm(*args)
    rng = np.random.default_rng(0)
    mi = rng.integers(0, 5, 50)
    ni = rng.integers(0, 48, 50)
    ys, as_ = oracle.gemm_at(*args, mi, ni)
    np.testing.assert_array_equal(ys, y[mi, ni])
    np.testing.assert_array_equal(as_, a[mi, ni])


def test_bad_arguments_rejected():
    p = synth.make_problem(1, 16, 128, 64, True, seed=1)
    with pytest.raises(ValueError):
        oracle.gemm(p["x"], p["qweight"], p["scales"], None, 1, 16, 128, 48, True)  # K % G
    with pytest.raises(ValueError):
        oracle.gemm_at(p["x"], p["qweight"], p["scales"], None, 1, 16, 128, 64, True, [1], [0])


# --------------------------------------------------------------------------
# fused SiLU(gate) * up

def test_silu_textbook_values():
    assert oracle.silu_mul(1.0, 1.0) == pytest.approx(math.e / (1.0 + math.e), rel=1e-15)
    assert oracle.silu_mul(1.0, 1.0) == pytest.approx(0.7310585786300049, rel=1e-15)
    assert oracle.silu_mul(0.0, 5.0) == 0.0
    assert oracle.silu_mul(40.0, 2.0) == 80.0
    v = oracle.silu_mul(-800.0, 1.0)
    assert v == 0.0 and math.copysign(1.0, v) < 0
    assert oracle.silu_mul(-1.0, 1.0) == pytest.approx(-1.0 / (1.0 + math.e), rel=1e-15)


@pytest.mark.parametrize("sym", [True, False])
def test_gateup_closed_forms(sym):
    M, N, K, G = 3, 16, 256, 64
    Kg = K // G
    p = synth.make_problem(M, N, K, G, sym, seed=13, gateup=True)
    # zero points kept <= 14 so that the code z + 1 below exists
    zmat = np.full((N, Kg), 8, np.uint8) if sym else synth.make_codes(N, Kg, 13, 4) % 15
    z = None if sym else synth.pack_nibbles_rows(zmat)
    mi, ni = np.repeat(np.arange(M), N), np.tile(np.arange(N), M)
    # gate codes equal to the zero point: g = 0 and h = 0
    qg0 = synth.pack_nibbles_rows(np.repeat(zmat, G, axis=1))
    h, g, u, _, _ = oracle.gateup_silu_at(p["x"], qg0, p["scales"], z, p["qweight_up"],
                                          p["scales_up"], z, M, N, K, G, sym, mi, ni)
    assert np.all(g == 0.0) and np.all(h == 0.0)
    # up codes z + 1 with unit scales: u = sum_k x_k exactly (bf16 sums of <= 256 terms
    # stay exact in float64), and h = SiLU(g) * sum_k x_k
    qu1 = synth.pack_nibbles_rows(np.repeat(zmat + 1, G, axis=1))
    ones = np.full((N, Kg), 0x3F80, np.uint16)
    codes_g = synth.make_codes(N, K, 13, 2)
    h, g, u, _, _ = oracle.gateup_silu_at(p["x"], synth.pack_nibbles_rows(codes_g), p["scales"], z,
                                          qu1, ones, z, M, N, K, G, sym, mi, ni)
    xs = [sum(Fraction(float(v)) for v in synth.bf16_bits_to_f32(p["x"][m])) for m in range(M)]
    np.testing.assert_array_equal(u, np.array([float(xs[m]) for m in mi]))
    ge, _ = _brute(codes_g, zmat, p["scales"], p["x"], G)
    for i, (m, n) in enumerate(zip(mi, ni)):
        gv = float(ge[m][n])
        assert g[i] == pytest.approx(gv, rel=1e-13, abs=1e-300)
        assert h[i] == pytest.approx(gv / (1.0 + math.exp(-gv)) * float(xs[m]), rel=1e-12)


def test_silu_bound_reduces_to_gemm_part_when_exact():
    # with no accumulation error allowed the bound is the relative part only
    b = oracle.silu_bound(np.array([2.0]), np.array([1.0]), np.array([3.0]),
                          np.array([0.0]), np.array([0.0]))
    assert b[0] == 2.0 * 2.0 ** -7


# --------------------------------------------------------------------------
# affine form w = scale * q + bias (MLX affine 4-bit checkpoints)

AFFINE_GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "affine_worked_example.txt")


def _load_affine_golden():
    d = {}
    with open(AFFINE_GOLDEN) as f:
        for line in f:
            if line.startswith("#") or ":" not in line:
                continue
            k, v = line.split(":", 1)
            d[k.strip()] = v.split()
    N, K, G = int(d["N"][0]), int(d["K"][0]), int(d["G"][0])
    hexes = lambda key, dt: np.array([int(h, 16) for h in d[key]], dtype=dt)
    f = lambda key: np.array([float(v) for v in d[key]])
    return dict(N=N, K=K, G=G, q=hexes("qweight", np.uint32).view(np.int32).reshape(N, K // 8),
                s=hexes("scales", np.uint16).reshape(N, K // G), b=hexes("biases", np.uint16).reshape(N, K // G),
                x=hexes("x", np.uint16).reshape(-1, K), w=f("w").reshape(N, K), y=f("y").reshape(-1, N),
                xsum=f("xsum").reshape(K // G, -1))


def test_affine_golden_dequant_gemm_and_group_sums():
    g = _load_affine_golden()
    N, K, G = g["N"], g["K"], g["G"]
    np.testing.assert_array_equal(oracle.dequant_affine(g["q"], g["s"], g["b"], N, K, G), g["w"])
    y, a = oracle.gemm_affine(g["x"], g["q"], g["s"], g["b"], 2, N, K, G)
    np.testing.assert_array_equal(y, g["y"])
    np.testing.assert_array_equal(a[0], np.abs(g["w"]).sum(axis=1))
    np.testing.assert_array_equal(oracle.group_sums(g["x"], 2, K, G), g["xsum"])


def _brute_affine(codes, scales, biases, x, G):
    """Exact y[m][n] and sum |x w| of the affine form from the unpacked codes."""
    M, K = x.shape
    N = codes.shape[0]
    xs = [[_fr_bf16(x[m, k]) for k in range(K)] for m in range(M)]
    y = [[Fraction(0)] * N for _ in range(M)]
    a = [[Fraction(0)] * N for _ in range(M)]
    for n in range(N):
        w = [_fr_bf16(scales[n, k // G]) * int(codes[n, k]) + _fr_bf16(biases[n, k // G]) for k in range(K)]
        for m in range(M):
            y[m][n] = sum((xs[m][k] * w[k] for k in range(K)), Fraction(0))
            a[m][n] = sum((abs(xs[m][k] * w[k]) for k in range(K)), Fraction(0))
    return y, a


@pytest.mark.parametrize("G,M,N,K", [(8, 3, 5, 32), (16, 2, 4, 64), (64, 1, 3, 128), (8, 2, 3, 88)])
def test_affine_bruteforce_exact(G, M, N, K, seed=None):
    seed = 31 + K + N if seed is None else seed
    Kg = K // G
    codes = synth.make_codes(N, K, seed, 2)
    s = synth.make_scales(N, Kg, 0.005, 0.02, seed)
    b = synth.make_biases(N, Kg, -0.16, -0.04, seed)
    x = synth.make_x(M, K, seed)
    y, a = oracle.gemm_affine(x, synth.pack_nibbles_rows(codes), s, b, M, N, K, G)
    ye, ae = _brute_affine(codes, s, b, x, G)
    gamma = 1.01 * K * 2.0 ** -53
    for m in range(M):
        for n in range(N):
            assert abs(Fraction(y[m, n]) - ye[m][n]) <= gamma * ae[m][n], (m, n)
            assert abs(Fraction(a[m, n]) - ae[m][n]) <= gamma * ae[m][n]


def test_affine_bruteforce_random_shapes():
    """The affine exact comparison over random shapes (1-20 groups of 8 or
    16) and seeds."""
    hyp = pytest.importorskip("hypothesis")
    st = hyp.strategies

    @hyp.settings(max_examples=60, deadline=None, derandomize=True)
    @hyp.given(G=st.sampled_from([8, 16]), M=st.integers(1, 3), N=st.integers(2, 4), Kg=st.integers(1, 20),
               seed=st.integers(0, 2**31 - 1))
    def run(G, M, N, Kg, seed):
        test_affine_bruteforce_exact(G, M, N, G * Kg, seed=seed)

    run()


def test_affine_zero_codes_leave_bias_times_group_sums():
    """q = 0 everywhere: y = sum_g bias_g * X_g, with X_g summed exactly."""
    M, N, K, G = 3, 8, 256, 64
    Kg = K // G
    q = synth.pack_nibbles_rows(np.zeros((N, K), np.uint8))
    s = synth.make_scales(N, Kg, 0.005, 0.02, 41)
    b = synth.make_biases(N, Kg, -0.16, -0.04, 41)
    x = synth.make_x(M, K, 41)
    y, a = oracle.gemm_affine(x, q, s, b, M, N, K, G)
    for m in range(M):
        xg = [sum((_fr_bf16(x[m, k]) for k in range(g * G, (g + 1) * G)), Fraction(0)) for g in range(Kg)]
        for n in range(N):
            expect = sum((_fr_bf16(b[n, g]) * xg[g] for g in range(Kg)), Fraction(0))
            assert abs(Fraction(y[m, n]) - expect) <= 1.01 * K * 2.0 ** -53 * Fraction(a[m, n])


def test_affine_without_bias_is_the_zero_point_form_with_zero_points_0():
    M, N, K, G = 2, 24, 256, 64
    Kg = K // G
    p = synth.make_problem(M, N, K, G, False, seed=43)
    zeros0 = synth.pack_nibbles_rows(np.zeros((N, Kg), np.uint8))
    b0 = np.zeros((N, Kg), np.uint16)
    ya, aa = oracle.gemm_affine(p["x"], p["qweight"], p["scales"], b0, M, N, K, G)
    yz, az = oracle.gemm(p["x"], p["qweight"], p["scales"], zeros0, M, N, K, G, False)
    np.testing.assert_array_equal(ya, yz)
    np.testing.assert_array_equal(aa, az)


def test_affine_one_hot_x_selects_weight():
    N, K, G = 20, 256, 64
    Kg = K // G
    codes = synth.make_codes(N, K, 45, 2)
    s = synth.make_scales(N, Kg, 0.005, 0.02, 45)
    b = synth.make_biases(N, Kg, -0.16, -0.04, 45)
    ks = [0, 9, 64, 200, 255]
    x = np.zeros((len(ks), K), np.uint16)
    for i, k in enumerate(ks):
        x[i, k] = 0x3F80
    y, _ = oracle.gemm_affine(x, synth.pack_nibbles_rows(codes), s, b, len(ks), N, K, G)
    sf = synth.bf16_bits_to_f32(s).astype(np.float64)
    bf = synth.bf16_bits_to_f32(b).astype(np.float64)
    for i, k in enumerate(ks):
        np.testing.assert_array_equal(y[i], sf[:, k // G] * codes[:, k] + bf[:, k // G])


def test_affine_gemm_at_and_gateup_match_their_parts():
    M, N, K, G = 4, 32, 256, 64
    p = synth.make_problem(M, N, K, G, False, seed=47, gateup=True, affine=True)
    assert p["zeros"] is None and p["zeros_up"] is None
    y, a = oracle.gemm_affine(p["x"], p["qweight"], p["scales"], p["biases"], M, N, K, G)
    rng = np.random.default_rng(1)
    mi, ni = rng.integers(0, M, 40), rng.integers(0, N, 40)
    ys, as_ = oracle.gemm_affine_at(p["x"], p["qweight"], p["scales"], p["biases"], M, N, K, G, mi, ni)
    np.testing.assert_array_equal(ys, y[mi, ni])
    np.testing.assert_array_equal(as_, a[mi, ni])
    h, g, u, _, _ = oracle.gateup_silu_affine_at(p["x"], p["qweight"], p["scales"], p["biases"],
                                                 p["qweight_up"], p["scales_up"], p["biases_up"], M, N, K, G, mi, ni)
    np.testing.assert_array_equal(g, ys)
    yu, _ = oracle.gemm_affine(p["x"], p["qweight_up"], p["scales_up"], p["biases_up"], M, N, K, G)
    np.testing.assert_array_equal(u, yu[mi, ni])
    for i in range(len(mi)):
        assert h[i] == pytest.approx(g[i] / (1.0 + math.exp(-g[i])) * u[i], rel=1e-14)


def test_group_sums_closed_forms():
    K, G = 512, 128
    ones = np.full((2, K), 0x3F80, np.uint16)
    np.testing.assert_array_equal(oracle.group_sums(ones, 2, K, G), np.full((K // G, 2), float(G)))
    x = synth.make_x(3, K, 49)
    xs = oracle.group_sums(x, 3, K, G)
    for m in range(3):
        for g in range(K // G):
            exact = sum((_fr_bf16(x[m, k]) for k in range(g * G, (g + 1) * G)), Fraction(0))
            assert xs[g, m] == float(exact)  # at most 128 bf16 terms: exact in float64


# --------------------------------------------------------------------------
# every code, zero point and scale; a planted maximum

@pytest.mark.parametrize("sym", [False, True])
def test_dequant_every_code_zero_point_and_scale(sym):
    """Every (code, zero point) pair meets every scale of a sweep from 2^-100
    to 2^100, both signs, in every nibble position of a word (codes 8-15 in
    the top nibble make the int32 word negative). The oracle's unpack of the
    packed words must give back exactly the q - z the input was built from,
    times the scale."""
    e = synth.exhaustive_problem(sym)
    N, K, G = e["N"], e["K"], e["group"]
    w = oracle.dequant(e["qweight"], e["scales"], e["zeros"], N, K, G, sym)
    s = synth.bf16_bits_to_f32(e["scale_bits"]).astype(np.float64)
    qz = e["codes"].astype(np.float64) - np.repeat(e["zero_points"], G, axis=1).astype(np.float64)
    np.testing.assert_array_equal(w, qz * np.repeat(s, G, axis=1))


def test_planted_maximum_is_the_argmax():
    """A weight row recoded to agree in sign with x row m (code 15 where x is
    +1, 0 where it is -1; z = 8) gives x[m] . w = sum_g s_g (7 P_g + 8 (G - P_g))
    with P_g the +1 entries of x[m] in group g: exact in float64 (every term
    is a short dyadic rational of nearby exponents), and the row's maximum."""
    M, N, K, G = 3, 300, 512, 128
    planted = [17, 250, 299]
    p = synth.planted_max_problem(M, N, K, G, planted, seed=3)
    y, _ = oracle.gemm(p["x"], p["qweight"], p["scales"], None, M, N, K, G, True)
    for m, n in enumerate(planted):
        P = p["x_positive"][m].reshape(K // G, G).sum(axis=1)
        exact = sum((_fr_bf16(p["scales"][n, g]) * (7 * int(P[g]) + 8 * (G - int(P[g]))) for g in range(K // G)),
                    Fraction(0))
        assert Fraction(y[m, n]) == exact
        assert int(np.argmax(y[m])) == n


# --------------------------------------------------------------------------
# top-k selection of a bf16 row

TOPK_GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "topk_worked_example.txt")


def test_topk_golden_worked_example():
    d = {}
    with open(TOPK_GOLDEN) as f:
        for line in f:
            if line.startswith("#") or ":" not in line:
                continue
            key, v = line.split(":", 1)
            d[key.strip()] = v.split()
    row = np.array([int(h, 16) for h in d["row"]], dtype=np.uint16)
    for key in ("k1", "k3", "k6", "k8", "k10"):
        k = int(key[1:])
        idx, vals = oracle.topk_bf16(row, k)
        assert idx[0].tolist() == [int(v) for v in d[key]], key
        np.testing.assert_array_equal(vals[0], row[idx[0]])


def _rank_by_comparison(vals):
    """Column order by repeated pairwise comparison of Python floats: a
    before b when a > b, or a NaN against a number, or equal (or both NaN)
    and a's column is lower."""
    import functools

    def cmp(i, j):
        a, b = vals[i], vals[j]
        an, bn = math.isnan(a), math.isnan(b)
        if an != bn:
            return -1 if an else 1
        if not an and a != b:
            return -1 if a > b else 1
        return -1 if i < j else (1 if i > j else 0)

    return sorted(range(len(vals)), key=functools.cmp_to_key(cmp))


def test_topk_against_pairwise_comparison():
    """Random rows mixing normal values, repeats, +-0, +-inf and NaNs, every
    k: the oracle's order equals a sort by pairwise float comparison."""
    rng = np.random.default_rng(7)
    specials = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0xFFC1, 0x3F80, 0xBF80], dtype=np.uint16)
    for trial in range(60):
        N = int(rng.integers(1, 40))
        row = rng.integers(0, 1 << 16, N).astype(np.uint16)
        mask = rng.random(N) < 0.35
        row[mask] = rng.choice(specials, int(mask.sum()))
        vals = [float(v) for v in synth.bf16_bits_to_f32(row)]
        want = _rank_by_comparison(vals)
        for k in range(1, N + 1):
            idx, _ = oracle.topk_bf16(row, k)
            assert idx[0].tolist() == want[:k], (trial, k)


def test_topk_k1_is_the_first_maximum_and_k_n_a_permutation():
    """k = 1 is numpy's argmax of the float values (first maximum, first NaN
    if any); k = N orders every column exactly once."""
    rng = np.random.default_rng(11)
    y = rng.integers(0, 1 << 16, (50, 300)).astype(np.uint16)
    y[:, rng.integers(0, 300, 20)] = 0x4040  # repeated values
    f = synth.bf16_bits_to_f32(y)
    idx, vals = oracle.topk_bf16(y, 1)
    np.testing.assert_array_equal(idx[:, 0], np.argmax(f, axis=1))
    full, _ = oracle.topk_bf16(y, 300)
    assert all(sorted(r) == list(range(300)) for r in full.tolist())
    with pytest.raises(ValueError):
        oracle.topk_bf16(y, 0)
    with pytest.raises(ValueError):
        oracle.topk_bf16(y, 301)


# --------------------------------------------------------------------------
# affine form at 2, 3, 5, 6 and 8 bits

BITS_GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "affine_bits_worked_example.txt")


def _load_bits_golden():
    d = {}
    with open(BITS_GOLDEN) as f:
        for line in f:
            if line.startswith("#") or ":" not in line:
                continue
            key, v = line.split(":", 1)
            d[key.strip()] = v.split()
    return d


@pytest.mark.parametrize("bits,G,M", [(3, 8, 2), (6, 16, 1)])
def test_affine_bits_golden_worked_example(bits, G, M):
    d = _load_bits_golden()
    pre = f"bits{bits}_"
    codes = np.array([int(v) for v in d[pre + "codes"]], dtype=np.uint8)[None, :]
    words = np.array([int(h, 16) for h in d[pre + "words"]], dtype=np.uint32)[None, :]
    s = np.array([int(h, 16) for h in d[pre + "scales"]], dtype=np.uint16)[None, :]
    b = np.array([int(h, 16) for h in d[pre + "biases"]], dtype=np.uint16)[None, :]
    x = np.array([int(h, 16) for h in d[pre + "x"]], dtype=np.uint16).reshape(M, 16)
    np.testing.assert_array_equal(synth.pack_bits_rows(codes, bits), words)
    assert [oracle.code_bits(words, 16, bits, 0, k) for k in range(16)] == codes[0].tolist()
    y, _ = oracle.gemm_affine_bits(x, words, s, b, M, 1, 16, G, bits)
    np.testing.assert_array_equal(y[:, 0], [float(v) for v in d[pre + "y"]])


def _pack_by_bigint(codes, bits):
    """Reference packer: one Python integer per row, code k shifted to bit bits*k."""
    R, C = codes.shape
    W = (C * bits + 31) // 32
    out = np.zeros((R, W), dtype=np.uint32)
    for r in range(R):
        v = 0
        for k in range(C):
            v |= int(codes[r, k]) << (bits * k)
        for i in range(W):
            out[r, i] = (v >> (32 * i)) & 0xFFFFFFFF
    return out


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6, 7, 8])
def test_bit_stream_packing(bits):
    codes = synth.make_codes_bits(5, 77, bits, seed=bits)
    assert codes.max() < (1 << bits)
    np.testing.assert_array_equal(synth.pack_bits_rows(codes, bits), _pack_by_bigint(codes, bits))
    q = synth.pack_bits_rows(codes, bits)
    got = [[oracle.code_bits(q, 77, bits, n, k) for k in range(77)] for n in range(5)]
    np.testing.assert_array_equal(np.array(got), codes)


def test_affine_bits4_is_the_nibble_form():
    """At 4 bits the stream is the nibble packing, and the b-bit GEMM equals
    the 4-bit affine GEMM on the same words exactly."""
    M, N, K, G = 3, 20, 256, 64
    codes = synth.make_codes(N, K, 5, 2)
    assert np.array_equal(synth.pack_bits_rows(codes, 4).view(np.int32), synth.pack_nibbles_rows(codes))
    s = synth.make_scales(N, K // G, 0.005, 0.02, 5)
    b = synth.make_biases(N, K // G, -0.16, -0.04, 5)
    x = synth.make_x(M, K, 5)
    y4, a4 = oracle.gemm_affine(x, synth.pack_nibbles_rows(codes), s, b, M, N, K, G)
    yb, ab = oracle.gemm_affine_bits(x, synth.pack_bits_rows(codes, 4), s, b, M, N, K, G, 4)
    np.testing.assert_array_equal(y4, yb)
    np.testing.assert_array_equal(a4, ab)


def _affine_bits_case(bits, M, N, K, G, seed):
    codes = synth.make_codes_bits(N, K, bits, seed)
    s = synth.make_scales(N, K // G, 0.005, 0.02, seed)
    b = synth.make_biases(N, K // G, -0.16, -0.04, seed)
    x = synth.make_x(M, K, seed)
    return codes, synth.pack_bits_rows(codes, bits), s, b, x


@pytest.mark.parametrize("bits", [2, 3, 5, 6, 8])
@pytest.mark.parametrize("G,M,N,K", [(8, 2, 3, 40), (16, 3, 2, 96), (64, 1, 3, 128)])
def test_affine_bits_bruteforce_exact(bits, G, M, N, K):
    """Exact rational sums from the codes the packer was given (not from the
    packed words), within the float64 summation bound."""
    codes, q, s, b, x = _affine_bits_case(bits, M, N, K, G, 40 + bits + K)
    y, a = oracle.gemm_affine_bits(x, q, s, b, M, N, K, G, bits)
    gamma = 1.01 * K * 2.0 ** -53
    for n in range(N):
        w = [_fr_bf16(s[n, k // G]) * int(codes[n, k]) + _fr_bf16(b[n, k // G]) for k in range(K)]
        for m in range(M):
            xs = [_fr_bf16(x[m, k]) for k in range(K)]
            ye = sum((xs[k] * w[k] for k in range(K)), Fraction(0))
            ae = sum((abs(xs[k] * w[k]) for k in range(K)), Fraction(0))
            assert abs(Fraction(y[m, n]) - ye) <= gamma * ae, (bits, m, n)
            assert abs(Fraction(a[m, n]) - ae) <= gamma * ae


@pytest.mark.parametrize("bits", [2, 3, 5, 6, 8])
def test_affine_bits_one_hot_x_and_dequant(bits):
    """One-hot x at column k gives s * q + b of that column exactly, and the
    dequantised matrix holds the same values."""
    N, K, G = 4, 64, 16
    codes, q, s, b, _ = _affine_bits_case(bits, 1, N, K, G, 70 + bits)
    w = oracle.dequant_affine_bits(q, s, b, N, K, G, bits)
    for k in (0, 1, 31, 63):
        x = np.zeros((1, K), dtype=np.uint16)
        x[0, k] = 0x3F80
        y, _ = oracle.gemm_affine_bits(x, q, s, b, 1, N, K, G, bits)
        for n in range(N):
            exact = _fr_bf16(s[n, k // G]) * int(codes[n, k]) + _fr_bf16(b[n, k // G])
            assert Fraction(y[0, n]) == exact and Fraction(w[n, k]) == exact
    # the pages' modules hold 2 to 8 bits
    for bad in (1, 9):
        with pytest.raises(ValueError):
            oracle.gemm_affine_bits(np.zeros((1, K), np.uint16), q, s, b, 1, N, K, G, bad)
        with pytest.raises(ValueError):
            oracle.dequant_affine_bits(q, s, b, N, K, G, bad)
