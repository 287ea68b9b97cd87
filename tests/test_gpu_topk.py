"""Device top-k of bf16 rows (w4a16_topk) against the oracle's top-k,
element by element: the same columns in the same order and the same value
bits. Rows mix ordinary values with repeats, +-0, +-inf and NaNs; widths are
ragged (rows off 16-byte boundaries take the one-value-per-thread path) and
long enough for clusters of 2 to 16 CTAs per row; k runs from 1 to 1024."""
import numpy as np
import pytest

import oracle
import synth

import gemm_w4a16_group_gb300 as w4

from gpu_helpers import dev, host_bits, torch

pytestmark = pytest.mark.gpu

SPECIALS = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0xFFC1, 0x3F80, 0xBF80], dtype=np.uint16)


def rows(M, N, seed, kind):
    rng = np.random.default_rng(seed)
    if kind == "bits":  # any 16-bit pattern, specials sprinkled in
        y = rng.integers(0, 1 << 16, (M, N)).astype(np.uint16)
        mask = rng.random((M, N)) < 0.05
        y[mask] = rng.choice(SPECIALS, int(mask.sum()))
    elif kind == "logits":  # bf16 of normal draws: many repeated values
        y = synth.f32_to_bf16_bits(rng.normal(0, 2, (M, N)).astype(np.float32))
    else:  # a handful of distinct values: long runs of ties at every threshold
        y = rng.choice(np.array([0x3F80, 0x4000, 0x0000, 0x8000, 0xBF80], dtype=np.uint16), (M, N))
    return np.ascontiguousarray(y)


def check(y, k):
    M, N = y.shape
    idx, vals = w4.topk(dev(y), k)
    torch().cuda.synchronize()
    want_i, want_v = oracle.topk_bf16(y, k)
    np.testing.assert_array_equal(idx.cpu().numpy(), want_i)
    np.testing.assert_array_equal(host_bits(vals), want_v)


@pytest.mark.parametrize("N", [1, 7, 300, 1000, 4096, 20000, 65539, 131080])
@pytest.mark.parametrize("kind", ["bits", "logits", "ties"])
def test_topk_matches_oracle(N, kind):
    M = 3
    y = rows(M, N, seed=N + len(kind), kind=kind)
    for k in sorted({1, min(N, 2), min(N, 8), min(N, 64), min(N, 1024), min(N, 777)}):
        check(y, k)


def test_topk_without_values_and_into_given_buffers():
    t = torch()
    y = rows(4, 5000, seed=3, kind="logits")
    idx = t.empty((4, 16), dtype=t.int64, device="cuda")
    got, vals = w4.topk(dev(y), 16, index_out=idx, values=False)
    t.cuda.synchronize()
    assert vals is None and got.data_ptr() == idx.data_ptr()
    np.testing.assert_array_equal(idx.cpu().numpy(), oracle.topk_bf16(y, 16)[0])


def test_topk_all_equal_and_all_nan_rows():
    """Every value equal: the first k columns; every value NaN: likewise."""
    for v in (0x4040, 0x7FC0, 0x8000):
        y = np.full((2, 3000), v, dtype=np.uint16)
        y[1, ::2] = 0x0000 if v == 0x8000 else v  # -0 and +0 mixed in row 1
        check(y, 100)
        check(y, 1024)


def test_topk_one_is_the_argmax_of_the_same_logits():
    M, N, K, G = 5, 4096, 1024, 128
    p = synth.make_problem(M, N, K, G, True, seed=9)
    x = dev(p["x"])
    packed = w4.repack(dev(p["qweight"]), dev(p["scales"]), None, N, K, G, True)
    idx, vals, y = w4.gemm_topk(x, packed, N, K, G, True, 1)
    am, _ = w4.gemm_argmax(x, packed, N, K, G, True)
    torch().cuda.synchronize()
    assert w4.kernel_status() == 0
    np.testing.assert_array_equal(idx.cpu().numpy()[:, 0], am.cpu().numpy())
    np.testing.assert_array_equal(host_bits(vals)[:, 0], host_bits(y)[np.arange(M), am.cpu().numpy()])
