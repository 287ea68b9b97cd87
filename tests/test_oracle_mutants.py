"""Each pin of the oracle rejects the mistakes it is there to catch.

tests/oracle_mutants.py retypes the oracle's decode steps in numpy with one
switch per planted mistake. Every test below first checks that the unmutated
retyping passes the pin (and equals the C oracle), then that the mutant fails
it, so the pins are shown to have the power they are relied on for:

  pin                                      mistakes it must catch
  hand-worked dequant example              nibble order reversed
  exact rational brute force               transposed weight, zero-point word
                                           stride floor(K/G/8), nibble order
  every code x zero point x scale          zero points read with a 3-bit mask
  affine exact brute force                 bias of the next group
  b-bit exact brute force                  a code straddling two words
  top-k by pairwise comparison, golden     NaN ranked lowest, -0 below +0
  SiLU' against a centred difference       a sign flip in SiLU'
  the bound against the interval of        each term of the fused gate/up
  reachable SiLU(g') u'                    bound left out

The fused gate/up bound (oracle.silu_bound) is pinned here too: SiLU' against
a centred finite difference of the oracle's own SiLU(g) * u, each term of the
bound against an independent evaluation, and the bound against the largest
|SiLU(g') u' - SiLU(g) u| over g' in [g - Bg, g + Bg] and u' in [u - Bu, u + Bu]
(sampled densely), plus a second-order slack derived below.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
import oracle_mutants as om
from test_oracle import _brute, _brute_affine, _fr_bf16, _load_golden

TOPK_GOLDEN_ROW = [0x3F80, 0x8000, 0x7FC0, 0x4040, 0x4040, 0x7F80, 0xFF80, 0x0000, 0x4020, 0x7FC1]
TOPK_GOLDEN_K10 = [2, 9, 5, 3, 4, 8, 0, 1, 7, 6]


# --------------------------------------------------------------------------
# the pins, each a function of the implementation under test

def _within_fp64_sum(y, a, ye, ae, K):
    gamma = 1.01 * K * 2.0 ** -53
    M, N = y.shape
    return all(abs(Fraction(y[m, n]) - ye[m][n]) <= gamma * ae[m][n] for m in range(M) for n in range(N))


def _zero_point_case(sym, G, M, N, K, seed):
    codes = synth.make_codes(N, K, seed, 2)
    Kg = K // G
    zmat = np.full((N, Kg), 8, dtype=np.uint8) if sym else synth.make_codes(N, Kg, seed, 4)
    q = synth.pack_nibbles_rows(codes)
    z = None if sym else synth.pack_nibbles_rows(zmat)
    s = synth.make_scales(N, Kg, 0.005, 0.02, seed)
    x = synth.make_x(M, K, seed)
    return codes, zmat, q, z, s, x


BRUTE_CASES = [(True, 8, 3, 5, 32), (False, 8, 2, 4, 64), (False, 16, 3, 3, 48), (True, 64, 1, 2, 128),
               (False, 8, 2, 3, 80), (False, 16, 1, 5, 272)]


def bruteforce_passes(mistake):
    """The exact rational brute force over the oracle test's fixed shapes."""
    for sym, G, M, N, K in BRUTE_CASES:
        codes, zmat, q, z, s, x = _zero_point_case(sym, G, M, N, K, 11 + K + N)
        y, a = om.gemm_from_weights(x, om.dequant(q, s, z, N, K, G, sym, mistake))
        ye, ae = _brute(codes, zmat, s, x, G)
        if not _within_fp64_sum(y, a, ye, ae, K):
            return False
    return True


def bruteforce_square_passes(mistake):
    """The brute force on a square weight (where a transposed read has the right shape)."""
    N = K = 16
    codes = synth.make_codes(N, K, 5, 2)
    s = np.full((N, 2), 0x3F80, dtype=np.uint16)
    x = synth.make_x(1, K, 5)
    y, a = om.gemm_from_weights(x, om.dequant(synth.pack_nibbles_rows(codes), s, None, N, K, 8, True, mistake))
    ye, ae = _brute(codes, np.full((N, 2), 8), s, x, 8)
    return _within_fp64_sum(y, a, ye, ae, K)


def golden_passes(mistake):
    g = _load_golden()
    for sym in (True, False):
        w = om.dequant(g["q"], g["s"], None if sym else g["z"], g["N"], g["K"], g["G"], sym, mistake)
        if not np.array_equal(w, g["w_sym"] if sym else g["w_asym"]):
            return False
    return True


def exhaustive_passes(mistake):
    e = synth.exhaustive_problem(False)
    N, K, G = e["N"], e["K"], e["group"]
    w = om.dequant(e["qweight"], e["scales"], e["zeros"], N, K, G, False, mistake)
    s = synth.bf16_bits_to_f32(e["scale_bits"]).astype(np.float64)
    qz = e["codes"].astype(np.float64) - np.repeat(e["zero_points"], G, axis=1).astype(np.float64)
    return np.array_equal(w, qz * np.repeat(s, G, axis=1))


AFFINE_CASES = [(8, 3, 5, 32), (16, 2, 4, 64), (64, 1, 3, 128), (8, 2, 3, 88)]


def affine_bruteforce_passes(mistake):
    for G, M, N, K in AFFINE_CASES:
        seed = 31 + K + N
        codes = synth.make_codes(N, K, seed, 2)
        s = synth.make_scales(N, K // G, 0.005, 0.02, seed)
        b = synth.make_biases(N, K // G, -0.16, -0.04, seed)
        x = synth.make_x(M, K, seed)
        y, a = om.gemm_from_weights(x, om.dequant_affine(synth.pack_nibbles_rows(codes), s, b, N, K, G, mistake))
        ye, ae = _brute_affine(codes, s, b, x, G)
        if not _within_fp64_sum(y, a, ye, ae, K):
            return False
    return True


def bits_bruteforce_passes(mistake, bits):
    for G, M, N, K in [(8, 2, 3, 40), (16, 3, 2, 96), (64, 1, 3, 128)]:
        seed = 40 + bits + K
        codes = synth.make_codes_bits(N, K, bits, seed)
        s = synth.make_scales(N, K // G, 0.005, 0.02, seed)
        b = synth.make_biases(N, K // G, -0.16, -0.04, seed)
        x = synth.make_x(M, K, seed)
        q = synth.pack_bits_rows(codes, bits)
        y, a = om.gemm_from_weights(x, om.dequant_affine_bits(q, s, b, N, K, G, bits, mistake))
        ye, ae = _brute_affine(codes, s, b, x, G)
        if not _within_fp64_sum(y, a, ye, ae, K):
            return False
    return True


def topk_pairwise_passes(mistake):
    from test_oracle import _rank_by_comparison
    rng = np.random.default_rng(7)
    specials = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0xFFC1, 0x3F80, 0xBF80], dtype=np.uint16)
    for _ in range(60):
        N = int(rng.integers(1, 40))
        row = rng.integers(0, 1 << 16, N).astype(np.uint16)
        mask = rng.random(N) < 0.35
        row[mask] = rng.choice(specials, int(mask.sum()))
        want = _rank_by_comparison([float(v) for v in synth.bf16_bits_to_f32(row)])
        idx, _ = om.topk(row, N, mistake)
        if idx[0].tolist() != want:
            return False
    return True


def topk_golden_passes(mistake):
    idx, _ = om.topk(np.array(TOPK_GOLDEN_ROW, dtype=np.uint16), 10, mistake)
    return idx[0].tolist() == TOPK_GOLDEN_K10


SILU_G = (-20.0, -3.0, -0.5, 0.0, 0.5, 3.0, 20.0)


def _silu(g):
    """SiLU(g) from the C oracle's SiLU(g) * u at u = 1."""
    return oracle.silu_mul(float(g), 1.0)


def dsilu_fd_passes(mistake):
    """SiLU'(g) against the centred difference (SiLU(g + h) - SiLU(g - h)) / 2h
    of the C oracle, h = 1e-4 max(1, |g|): truncation below 1e-9 and rounding
    below 1e-11 here, so 1e-7 separates a right derivative from a wrong one."""
    for g in SILU_G:
        h = 1e-4 * max(1.0, abs(g))
        fd = (_silu(g + h) - _silu(g - h)) / (2 * h)
        if abs(float(om.dsilu(g, mistake)) - fd) > 1e-7 * max(1.0, abs(fd)):
            return False
    return True


# Second-order slack of the first-order bound. With f(g, u) = SiLU(g) u and
# |dg| <= Bg, |du| <= Bu, Taylor's theorem gives
#   f(g + dg, u + du) - f(g, u) = SiLU(g) du + SiLU'(g) dg (u + du) + SiLU''(xi) dg^2 (u + du) / 2,
# so |f' - f| <= |SiLU| Bu + |SiLU'| |u| Bg + |SiLU'| Bg Bu + max|SiLU''| Bg^2 (|u| + Bu) / 2.
# The bound carries Bg Bu for the cross term; with max|SiLU'| < 1.1 and
# max|SiLU''| = SiLU''(0) = 1/2 (both checked in test_silu_slack_constants) the
# remainder is at most 0.1 Bg Bu + 0.25 Bg^2 (|u| + Bu).
MAX_DSILU, MAX_D2SILU = 1.1, 0.5


def _slack(u, bg, bu):
    return (MAX_DSILU - 1.0) * bg * bu + 0.5 * MAX_D2SILU * bg * bg * (abs(u) + bu)


def silu_interval_passes(mistake):
    """The bound (less its relative part) against the largest reachable
    |SiLU(g') u' - SiLU(g) u|: 401 points g' across [g - Bg, g + Bg] (ends
    included) and both ends of [u - Bu, u + Bu] (the deviation is convex in
    u'), every (g, u, Bg, Bu) of the grid."""
    for g in SILU_G + (2.4, -1.3):
        for u in (-2.0, 0.0, 0.7, 5.0):
            h = oracle.silu_mul(g, u)
            for bg in (1e-3, 0.05, 0.3):
                for bu in (1e-3, 0.05, 0.3):
                    gp = np.linspace(g - bg, g + bg, 401)
                    sg = np.array([_silu(v) for v in gp])
                    dev = max(np.max(np.abs(sg * (u - bu) - h)), np.max(np.abs(sg * (u + bu) - h)))
                    first = float(om.silu_bound(h, g, u, bg / oracle.ACC_TOL, bu / oracle.ACC_TOL, mistake)
                                  - oracle.REL_TOL * abs(h))
                    if dev > first + _slack(u, bg, bu) + 1e-14 * (1.0 + abs(h)):
                        return False
    return True


# --------------------------------------------------------------------------
# the retyping equals the oracle

@pytest.mark.parametrize("sym,G,M,N,K", BRUTE_CASES)
def test_retyped_dequant_equals_oracle(sym, G, M, N, K):
    _, _, q, z, s, x = _zero_point_case(sym, G, M, N, K, 11 + K + N)
    np.testing.assert_array_equal(om.dequant(q, s, z, N, K, G, sym), oracle.dequant(q, s, z, N, K, G, sym))


def test_retyped_affine_bits_and_topk_equal_oracle():
    for G, _, N, K in AFFINE_CASES:
        codes = synth.make_codes(N, K, 3, 2)
        q = synth.pack_nibbles_rows(codes)
        s = synth.make_scales(N, K // G, 0.005, 0.02, 3)
        b = synth.make_biases(N, K // G, -0.16, -0.04, 3)
        np.testing.assert_array_equal(om.dequant_affine(q, s, b, N, K, G), oracle.dequant_affine(q, s, b, N, K, G))
    for bits in (2, 3, 5, 6, 7, 8):
        codes = synth.make_codes_bits(3, 96, bits, bits)
        q = synth.pack_bits_rows(codes, bits)
        s = synth.make_scales(3, 6, 0.005, 0.02, bits)
        b = synth.make_biases(3, 6, -0.16, -0.04, bits)
        np.testing.assert_array_equal(om.dequant_affine_bits(q, s, b, 3, 96, 16, bits),
                                      oracle.dequant_affine_bits(q, s, b, 3, 96, 16, bits))
    rng = np.random.default_rng(3)
    y = rng.integers(0, 1 << 16, (20, 50)).astype(np.uint16)
    y[:, ::7] = 0x8000
    y[:, ::11] = 0x7FC0
    for k in (1, 5, 50):
        a, av = om.topk(y, k)
        b_, bv = oracle.topk_bf16(y, k)
        np.testing.assert_array_equal(a, b_)
        np.testing.assert_array_equal(av, bv)


def test_retyped_silu_bound_equals_oracle():
    rng = np.random.default_rng(5)
    g = rng.normal(0, 6, 200)
    u = rng.normal(0, 3, 200)
    h = np.array([oracle.silu_mul(a, b) for a, b in zip(g, u)])
    ga, ua = rng.uniform(0, 1e4, 200), rng.uniform(0, 1e4, 200)
    np.testing.assert_array_equal(om.silu_bound(h, g, u, ga, ua), oracle.silu_bound(h, g, u, ga, ua))
    np.testing.assert_array_equal(om.dsilu(g), oracle.dsilu(g))


# --------------------------------------------------------------------------
# the fused gate/up bound, pinned

def test_dsilu_against_centred_difference():
    assert dsilu_fd_passes(None)


def test_silu_bound_terms_against_independent_evaluations():
    """With Bu = 0 the bound less its relative part is |SiLU'(g)| |u| Bg, with
    SiLU' from the centred difference; with Bg = 0 it is |SiLU(g)| Bu, with
    SiLU from the C oracle; with both it adds Bg Bu."""
    for g in SILU_G:
        h_ = 1e-4 * max(1.0, abs(g))
        fd = (_silu(g + h_) - _silu(g - h_)) / (2 * h_)
        for u in (-2.0, 0.7, 5.0):
            h = oracle.silu_mul(g, u)
            rel = oracle.REL_TOL * abs(h)
            bg_only = float(oracle.silu_bound(h, g, u, 3e3, 0.0)) - rel
            assert bg_only == pytest.approx(abs(fd) * abs(u) * 3e3 * oracle.ACC_TOL, rel=1e-6, abs=1e-300)
            bu_only = float(oracle.silu_bound(h, g, u, 0.0, 4e3)) - rel
            assert bu_only == pytest.approx(abs(_silu(g)) * 4e3 * oracle.ACC_TOL, rel=1e-12, abs=1e-300)
            both = float(oracle.silu_bound(h, g, u, 3e3, 4e3)) - rel
            assert both == pytest.approx(bg_only + bu_only + 3e3 * 4e3 * oracle.ACC_TOL ** 2, rel=1e-12)


def test_silu_slack_constants():
    """max |SiLU'| < 1.1 (it peaks near g = 2.4 at about 1.0998) and
    max |SiLU''| = 1/2 at g = 0, from centred differences of the C oracle's
    SiLU on a dense grid."""
    gs = np.linspace(-40.0, 40.0, 16001)
    h = 1e-3
    d1 = [(_silu(g + h) - _silu(g - h)) / (2 * h) for g in gs]
    d2 = [(_silu(g + h) - 2 * _silu(g) + _silu(g - h)) / (h * h) for g in gs]
    assert max(np.abs(d1)) < MAX_DSILU
    assert max(np.abs(d2)) <= MAX_D2SILU + 1e-5
    assert abs(d2[8000] - 0.5) < 1e-5  # g = 0


def test_silu_bound_covers_the_reachable_interval():
    assert silu_interval_passes(None)


# --------------------------------------------------------------------------
# each pin rejects its mistakes

def test_golden_rejects_reversed_nibble_order():
    assert golden_passes(None)
    assert not golden_passes("nibble_order_reversed")


@pytest.mark.parametrize("mistake", ["nibble_order_reversed", "zero_word_stride_floor"])
def test_bruteforce_rejects(mistake):
    assert bruteforce_passes(None)
    assert not bruteforce_passes(mistake)


def test_bruteforce_rejects_transposed_weight():
    assert bruteforce_square_passes(None)
    assert not bruteforce_square_passes("transposed")


def test_exhaustive_rejects_three_bit_zero_mask():
    assert exhaustive_passes(None)
    assert not exhaustive_passes("zero_mask_3bit")


def test_affine_bruteforce_rejects_next_group_bias():
    assert affine_bruteforce_passes(None)
    assert not affine_bruteforce_passes("bias_group_off_by_one")


@pytest.mark.parametrize("bits", [3, 5, 6, 7])
def test_bits_bruteforce_rejects_straddle(bits):
    """Widths that do not divide 32 have codes running into the next word."""
    assert bits_bruteforce_passes(None, bits)
    assert not bits_bruteforce_passes("straddle_next_word", bits)


@pytest.mark.parametrize("mistake", ["nan_lowest", "negzero_below_zero"])
def test_topk_pins_reject(mistake):
    assert topk_pairwise_passes(None) and topk_golden_passes(None)
    assert not topk_pairwise_passes(mistake)
    assert not topk_golden_passes(mistake)


def test_dsilu_pin_rejects_sign_flip():
    assert not dsilu_fd_passes("dsilu_sign")


@pytest.mark.parametrize("mistake", ["drop_bg", "drop_bu", "drop_cross"])
def test_interval_pin_rejects_dropped_terms(mistake):
    assert not silu_interval_passes(mistake)
