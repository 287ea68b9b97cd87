"""Pins of the seeded input generators (shared by oracle and CUDA path)."""
import numpy as np
import pytest

import synth
from synth import workloads


def test_splitmix64_published_outputs():
    # SplitMix64 started at state 0 (Steele, Lea and Flood 2014; the reference
    # outputs quoted with Vigna's xoshiro seeding code)
    out = [int(v) for v in synth.splitmix64_stream(0, 4)]
    assert out == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F, 0xF88BB8A8724C81EC]
    # offsets continue the same sequence
    assert int(synth.splitmix64_stream(0, 1, offset=2)[0]) == 0x06C45D188009454F


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(1)
    f = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 10,
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 3.4e38, -1e-30,
                                  np.inf, -np.inf], dtype=np.float32)])
    # exact ties: 1 + 2^-8 (even below), 1 + 3 * 2^-8 (odd below)
    mine = synth.f32_to_bf16_bits(f)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(mine, ref)
    np.testing.assert_array_equal(synth.bf16_bits_to_f32(mine),
                                  torch.from_numpy(f).to(torch.bfloat16).float().numpy())


def test_pack_nibbles_hand_word():
    w = synth.pack_nibbles_rows(np.array([[0, 1, 2, 3, 4, 5, 6, 7, 15, 14]]))
    assert w.view(np.uint32).tolist() == [[0x76543210, 0x0000000EF]]


def test_distributions():
    c = synth.make_codes(64, 1024, 0, 2)
    assert c.min() == 0 and c.max() == 15
    counts = np.bincount(c.ravel(), minlength=16)
    assert counts.min() > 0.9 * c.size / 16
    # whole-word draws: 16 codes per SplitMix64 output, every nibble uniform
    w = synth.make_qweight(64, 1024, 0).view(np.uint32)
    nib = (w[..., None] >> (4 * np.arange(8, dtype=np.uint32))) & np.uint32(15)
    counts = np.bincount(nib.ravel(), minlength=16)
    assert counts.min() > 0.9 * nib.size / 16
    s = synth.bf16_bits_to_f32(synth.make_scales(256, 40, 0.005, 0.02, 0))
    assert s.min() >= 0.005 * (1 - 2 ** -8) and s.max() <= 0.02 * (1 + 2 ** -8)
    x = synth.bf16_bits_to_f32(synth.make_x(4, 4096, 0)).astype(np.float64)
    assert abs(x.mean()) < 0.05 and abs(x.std() - 1.0) < 0.05


def test_streams_differ_and_are_seeded():
    a = synth.make_qweight(16, 64, 0)
    b = synth.make_qweight(16, 64, 0, synth.TENSOR_IDS["qweight_up"])
    c = synth.make_qweight(16, 64, 1)
    assert not np.array_equal(a, b) and not np.array_equal(a, c)
    np.testing.assert_array_equal(a, synth.make_qweight(16, 64, 0))


def test_workload_table():
    w = workloads.WORKLOADS
    assert w[workloads.HEADLINE]["N"] == 34816
    assert workloads.algorithmic_bytes(1, 34816, 5120, 128, True) == 91_994_112
    assert w["prompt_gateup_m4096_k5120_n17408"]["kind"] == "gateup"
    assert sum(1 for k in w if k.startswith("smallm_")) == 15


def test_qweight_words_are_draw_halves_and_blocking_is_invisible():
    w = synth.make_qweight(10, 64, 3).view(np.uint32).ravel()
    d = synth.splitmix64_stream(synth._stream_state(3, synth.TENSOR_IDS["qweight"]), 40)
    assert w[0] == int(d[0]) & 0xFFFFFFFF and w[1] == int(d[0]) >> 32
    assert w[79] == int(d[39]) >> 32
    np.testing.assert_array_equal(synth.make_qweight(37, 128, 5, block_rows=4),
                                  synth.make_qweight(37, 128, 5))
    np.testing.assert_array_equal(synth.splitmix64_stream(9, 10, offset=5),
                                  synth.splitmix64_stream(9, 15)[5:])


@pytest.mark.parametrize("sym", [False, True])
def test_exhaustive_problem_meets_every_code_zero_point_and_scale(sym):
    e = synth.exhaustive_problem(sym)
    G = e["group"]
    c = e["codes"].reshape(e["N"], 16, G)
    seen = set()
    for r in range(e["N"]):
        for g in range(16):
            z, s = int(e["zero_points"][r, g]), int(e["scale_bits"][r, g])
            seen.update((int(q), z, s) for q in np.unique(c[r, g]))
    assert len(seen) == (16 * 16 * 16 if not sym else 16 * 16)
    # the packed words hold the codes and zero points, nibble j of word c = column 8c + j
    np.testing.assert_array_equal(e["qweight"], synth.pack_nibbles_rows(e["codes"]))
    if not sym:
        np.testing.assert_array_equal(e["zeros"], synth.pack_nibbles_rows(e["zero_points"]))
    # every scale of the sweep, exactly, and normal in float32 times any |q - z| <= 15
    vals = set(synth.bf16_bits_to_f32(e["scale_bits"]).astype(np.float64).ravel().tolist())
    assert vals == set(synth.SCALE_SWEEP)
    tiny = np.float32(min(abs(v) for v in synth.SCALE_SWEEP))
    assert tiny >= np.finfo(np.float32).tiny and 15 * max(abs(v) for v in synth.SCALE_SWEEP) < np.finfo(np.float32).max


def test_planted_max_problem_recodes_the_planted_rows():
    M, N, K, G = 3, 64, 256, 128
    p = synth.planted_max_problem(M, N, K, G, [5, 40, 63], seed=2)
    assert p["x"].dtype == np.uint16 and set(np.unique(p["x"]).tolist()) <= {0x3F80, 0xBF80}
    base = synth.make_problem(M, N, K, G, True, scale_range=(0.002, 0.01), seed=2)
    for m, n in enumerate([5, 40, 63]):
        want = np.where(p["x"][m] == 0x3F80, 15, 0)
        np.testing.assert_array_equal(p["qweight"][n], synth.pack_nibbles_rows(want[None, :])[0])
    others = [r for r in range(N) if r not in (5, 40, 63)]
    np.testing.assert_array_equal(p["qweight"][others], base["qweight"][others])
    np.testing.assert_array_equal(p["scales"], base["scales"])
    with pytest.raises(AssertionError):
        synth.planted_max_problem(2, N, K, G, [7, 7])
