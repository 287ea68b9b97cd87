"""Every measured workload at full size, in the launch configuration bench.py
times (automatic kernel choice), checked against the oracle on sampled
outputs it computes one by one (the affine workloads through the affine
entry points and oracle); the output-vocabulary head also on its argmax over
all 248,320 columns."""
import numpy as np
import pytest

import oracle
import synth
from synth.workloads import WORKLOADS

import gemm_w4a16_group_gb300 as w4

from gpu_helpers import (assert_within, bf16_f64, dev, host_bits, packed_of, run_gateup, run_gemm, sample_pairs, torch,
                         upload)

pytestmark = pytest.mark.gpu

_cache = {}


def problem(name):
    if name not in _cache:
        w = WORKLOADS[name]
        _cache.clear()  # keep one full-size problem in host memory at a time
        _cache[name] = synth.make_problem(w["M"], w["N"], w["K"], w["group"], w["sym"],
                                          scale_range=w["scale_range"], x_scale=w["x_scale"], seed=0,
                                          gateup=w["kind"] == "gateup", affine=w["affine"])
    return _cache[name]


def run_affine(p, gateup):
    """The affine workload through its public calls, as bench.py makes them
    (group sums from w4a16_xsum above 32 rows)."""
    x = dev(p["x"])
    xs = w4.xsum(x, p["K"], p["group"]) if p["M"] > 32 else None
    if gateup:
        packed = w4.repack_affine_gateup(dev(p["qweight"]), dev(p["scales"]), dev(p["biases"]), dev(p["qweight_up"]),
                                         dev(p["scales_up"]), dev(p["biases_up"]), p["N"], p["K"], p["group"])
        out = w4.gateup_silu_affine(x, packed, p["N"], p["K"], p["group"], xs)
    else:
        packed = w4.repack_affine(dev(p["qweight"]), dev(p["scales"]), dev(p["biases"]), p["N"], p["K"], p["group"])
        out = w4.gemm_affine(x, packed, p["N"], p["K"], p["group"], xs)
    torch().cuda.synchronize()
    assert w4.kernel_status() == 0
    return host_bits(out)


GEMM_NAMES = [n for n, w in WORKLOADS.items() if w["kind"] in ("gemm", "lm_head")]


@pytest.mark.parametrize("name", GEMM_NAMES)
def test_workload_sampled(name):
    p = problem(name)
    mi, ni = sample_pairs(p["M"], p["N"], 1500, seed=len(name))
    if p["affine"]:
        y = run_affine(p, gateup=False)
        ref, sa = oracle.gemm_affine_at(p["x"], p["qweight"], p["scales"], p["biases"], p["M"], p["N"], p["K"],
                                        p["group"], mi, ni)
    else:
        y = run_gemm(p)
        ref, sa = oracle.gemm_at(p["x"], p["qweight"], p["scales"], p["zeros"], p["M"], p["N"], p["K"],
                                 p["group"], p["sym"], mi, ni)
    assert_within(y[mi, ni], ref, oracle.gemm_bound(ref, sa), name)
    assert np.isfinite(bf16_f64(y)).all()


@pytest.mark.parametrize("M", [1, 5, 16])
def test_lm_head_argmax(M):
    """The head's greedy pick, from the logits and from the fused device
    argmax (which stores no logits), against the oracle's exact maximum."""
    name = f"lm_head_m{M}_k5120_n248320"
    p = problem(name)
    d = upload(p)
    packed = packed_of(p, d)
    yb = run_gemm(p, d=d, packed=packed)
    fused, none = w4.gemm_argmax(d["x"], packed, p["N"], p["K"], p["group"], p["sym"])
    torch().cuda.synchronize()
    assert none is None and w4.kernel_status() == 0
    y = bf16_f64(yb)
    np.testing.assert_array_equal(fused.cpu().numpy(), np.argmax(y, axis=1))
    ref, sa = oracle.gemm(p["x"], p["qweight"], p["scales"], p["zeros"], p["M"], p["N"], p["K"],
                          p["group"], p["sym"])
    bound = oracle.gemm_bound(ref, sa)
    exact = 0
    for m in range(M):
        a_gpu, a_ref = int(np.argmax(y[m])), int(np.argmax(ref[m]))
        if a_gpu == a_ref:
            exact += 1
        else:
            # a near-tie: the GPU's pick is within the bound of the true maximum
            assert ref[m, a_ref] - ref[m, a_gpu] <= bound[m, a_gpu] + bound[m, a_ref], (m, a_gpu, a_ref)
    assert exact >= M - 1


@pytest.mark.parametrize("M", [16, 5, 1])
def test_lm_head_topk(M):
    """Top-k over all 248,320 columns of the head's logits (w4a16_gemm_topk),
    element by element against the oracle's top-k of the same logits, at
    k = 1, 8 and 64; k = 1 is the fused argmax's pick."""
    name = f"lm_head_m{M}_k5120_n248320"
    p = problem(name)
    d = upload(p)
    packed = packed_of(p, d)
    fused, _ = w4.gemm_argmax(d["x"], packed, p["N"], p["K"], p["group"], p["sym"])
    for k in (1, 8, 64):
        idx, vals, y = w4.gemm_topk(d["x"], packed, p["N"], p["K"], p["group"], p["sym"], k)
        torch().cuda.synchronize()
        assert w4.kernel_status() == 0
        yb = host_bits(y)
        want_i, want_v = oracle.topk_bf16(yb, k)
        np.testing.assert_array_equal(idx.cpu().numpy(), want_i)
        np.testing.assert_array_equal(host_bits(vals), want_v)
        if k == 1:
            np.testing.assert_array_equal(idx.cpu().numpy()[:, 0], fused.cpu().numpy())


GATEUP_NAMES = [n for n, w in WORKLOADS.items() if w["kind"] == "gateup"]


@pytest.mark.parametrize("name", GATEUP_NAMES)
def test_gateup_workload_sampled(name):
    p = problem(name)
    mi, ni = sample_pairs(p["M"], p["N"], 2000, seed=1)
    if p["affine"]:
        h = run_affine(p, gateup=True)
        ref, g, u, ga, ua = oracle.gateup_silu_affine_at(p["x"], p["qweight"], p["scales"], p["biases"],
                                                         p["qweight_up"], p["scales_up"], p["biases_up"], p["M"],
                                                         p["N"], p["K"], p["group"], mi, ni)
    else:
        h = run_gateup(p)
        ref, g, u, ga, ua = oracle.gateup_silu_at(p["x"], p["qweight"], p["scales"], p["zeros"],
                                                  p["qweight_up"], p["scales_up"], p["zeros_up"], p["M"],
                                                  p["N"], p["K"], p["group"], p["sym"], mi, ni)
    assert_within(h[mi, ni], ref, oracle.silu_bound(ref, g, u, ga, ua), name)
    assert np.isfinite(bf16_f64(h)).all()
