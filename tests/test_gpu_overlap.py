"""Programmatic overlap of consecutive decode calls: a call that reads the
previous call's output must see all of it.

Two M <= 16 matmuls are chained (the second one's x is the first one's y),
on the automatic kernel choice and on the tcgen05 decode kernel, and run many
times back to back, eagerly and from a CUDA graph, with the overlap
switch on. The kernels are deterministic, so every result must equal, bit for
bit, the same chain run with the switch off; the chain's final output is also
checked against the oracle, given the first call's output as its input.
"""
import numpy as np
import pytest

import oracle
import synth

import gemm_w4a16_group_gb300 as w4

from gpu_helpers import assert_within, bf16_f64, host_bits, kernel, packed_of, torch, upload

pytestmark = pytest.mark.gpu


@pytest.fixture
def overlap_off_after():
    prev = w4.set_programmatic_overlap(False)
    yield
    w4.set_programmatic_overlap(prev)


@pytest.mark.parametrize("which", [w4.KERNEL_AUTO, w4.KERNEL_DECODE_TC])
@pytest.mark.parametrize("M", [1, 5, 16])
def test_chained_calls_overlap(M, which, overlap_off_after):
    with kernel(which):
        _chained_calls_overlap(M)


def _chained_calls_overlap(M):
    t = torch()
    K1, N1, N2, G = 1024, 2048, 520, 64
    pa = synth.make_problem(M, N1, K1, G, False, seed=31 + M)
    pb = synth.make_problem(M, N2, N1, G, True, seed=47 + M)
    da, db = upload(pa), upload(pb)
    wa, wb = packed_of(pa, da), packed_of(pb, db)
    y1 = t.empty((M, N1), dtype=t.bfloat16, device="cuda")
    y2 = t.empty((M, N2), dtype=t.bfloat16, device="cuda")
    t.cuda.synchronize()  # the packed weights are complete before any overlapped call

    def chain(n):
        for _ in range(n):
            w4.gemm(da["x"], wa, N1, K1, G, False, out=y1)
            w4.gemm(y1, wb, N2, N1, G, True, out=y2)

    w4.set_programmatic_overlap(False)
    chain(1)
    t.cuda.synchronize()
    ref1, ref2 = host_bits(y1), host_bits(y2)

    w4.set_programmatic_overlap(True)
    y1.zero_()
    y2.zero_()
    chain(20)
    t.cuda.synchronize()
    assert w4.kernel_status() == 0
    np.testing.assert_array_equal(host_bits(y1), ref1)
    np.testing.assert_array_equal(host_bits(y2), ref2)

    s = t.cuda.Stream()
    g = t.cuda.CUDAGraph()
    with t.cuda.graph(g, stream=s):
        chain(10)
    y1.zero_()
    y2.zero_()
    t.cuda.synchronize()
    for _ in range(3):
        g.replay()
    t.cuda.synchronize()
    assert w4.kernel_status() == 0
    np.testing.assert_array_equal(host_bits(y1), ref1)
    np.testing.assert_array_equal(host_bits(y2), ref2)

    # the second call against the oracle, on the first call's output
    x2 = ref1.reshape(M, N1)
    r, sa = oracle.gemm(x2, pb["qweight"], pb["scales"], None, M, N2, N1, G, True)
    assert_within(ref2, r, oracle.gemm_bound(r, sa), "chained second call")
    r1, sa1 = oracle.gemm(pa["x"], pa["qweight"], pa["scales"], pa["zeros"], M, N1, K1, G, False)
    assert_within(ref1, r1, oracle.gemm_bound(r1, sa1), "chained first call")
    assert np.isfinite(bf16_f64(ref2)).all()
