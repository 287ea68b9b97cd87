"""The workloads the library is measured and checked on.

Shapes are the projection shapes of a 27B dense decoder with hidden size 5120
and feed-forward width 17408 (GRIMOIRE v1.7 release notes, "What changed":
single-user decode, 2-16 rows for batching and speculative verify; GRIMOIRE
v1.8 release notes, "What changed": the output layer checked in one pass, the
prompt path with the feed-forward gate fused, 4,096-token prompts). Group 128
with the symmetric zero point 8 is the GPTQ-Int4 checkpoint and group 64 with
packed 4-bit zero points the AutoRound W4A16 one (v1.7, measurement table).
The affine workloads take the same shapes in the MLX affine 4-bit form, group
64 with a bf16 bias per group (TensorFold PR #859, "What this changes").
"""
from __future__ import annotations

import math

HIDDEN, FFN, VOCAB = 5120, 17408, 248320

# name -> problem parameters (make_problem keywords plus "kind")
WORKLOADS: dict[str, dict] = {}


def _add(name, **kw):
    kw.setdefault("kind", "gemm")
    kw.setdefault("affine", False)
    kw.setdefault("scale_range", (0.005, 0.02))
    kw.setdefault("x_scale", 1.0)
    WORKLOADS[name] = kw


# tiny single-row case, small enough for the oracle in milliseconds
_add("tiny_gemv_m1_k512_n256", M=1, K=512, N=256, group=128, sym=True)
# single-user decode: fused gate+up rows, and the down projection
_add("decode_gateup_m1_k5120_n34816", M=1, K=HIDDEN, N=2 * FFN, group=128, sym=True)
_add("decode_down_m1_k17408_n5120", M=1, K=FFN, N=HIDDEN, group=128, sym=True)
# batched decode / speculative verify rows, asymmetric group 64
for _M in (2, 4, 5, 8, 16):
    for _K, _N in ((HIDDEN, HIDDEN), (HIDDEN, 2 * FFN), (FFN, HIDDEN)):
        _add(f"smallm_m{_M}_k{_K}_n{_N}", M=_M, K=_K, N=_N, group=64, sym=False)
# 17-32 rows (a longer verify window) on the decode kernel, and a 256-row
# prompt chunk through the down projection (few output tiles: split K)
_add("verify_m32_k5120_n34816", M=32, K=HIDDEN, N=2 * FFN, group=64, sym=False)
_add("chunk_m256_k17408_n5120", M=256, K=FFN, N=HIDDEN, group=128, sym=True)
# single-user decode through the fused gate/up: h = SiLU(x Wg^T) * (x Wu^T),
# both weights read once (the same 34,816 weight rows as above)
_add("decode_gateup_silu_m1_k5120_n17408", M=1, K=HIDDEN, N=FFN, group=128, sym=True, kind="gateup")
# output-vocabulary head
for _M in (1, 5, 16):
    _add(f"lm_head_m{_M}_k5120_n248320", M=_M, K=HIDDEN, N=VOCAB, group=128, sym=True,
         scale_range=(0.002, 0.01), x_scale=64.0 / math.sqrt(HIDDEN), kind="lm_head")
# prompt processing with the feed-forward gate fused: h = SiLU(x Wg^T) * (x Wu^T)
_add("prompt_gateup_m4096_k5120_n17408", M=4096, K=HIDDEN, N=FFN, group=128, sym=True,
     kind="gateup")

# the affine form (scale * q + bias, group 64): decode rows, verify rows, and
# the prompt with the fused gate
_add("affine_decode_m1_k5120_n34816", M=1, K=HIDDEN, N=2 * FFN, group=64, sym=False, affine=True)
_add("affine_smallm_m16_k5120_n34816", M=16, K=HIDDEN, N=2 * FFN, group=64, sym=False, affine=True)
_add("affine_prompt_gateup_m4096_k5120_n17408", M=4096, K=HIDDEN, N=FFN, group=64, sym=False, affine=True,
     kind="gateup")
# the same prompt rows through the plain GEMM of the 34,816 gate+up rows (the
# form w4a16_gemm_affine_noalloc runs)
_add("affine_prompt_m4096_k5120_n34816", M=4096, K=HIDDEN, N=2 * FFN, group=64, sym=False, affine=True)

# the configuration the headline throughput line is quoted on
HEADLINE = "decode_gateup_m1_k5120_n34816"


def algorithmic_bytes(M: int, N: int, K: int, group: int, sym: bool, affine: bool = False) -> int:
    """Bytes one call must move at least: packed codes, scales, zero points (or
    affine biases), x and y."""
    Kg = K // group
    b = N * K // 2 + N * Kg * 2 + M * K * 2 + M * N * 2
    if affine:
        b += N * Kg * 2
    elif not sym:
        b += N * Kg // 2
    return b


def gemm_flops(M: int, N: int, K: int) -> int:
    return 2 * M * N * K


def gateup_bytes(M: int, N_each: int, K: int, group: int, sym: bool, affine: bool = False) -> int:
    """Bytes a fused gate/up call must move at least: both packed weights with
    their scales (and zero points or biases), x, and the N_each-wide output h."""
    w = algorithmic_bytes(0, N_each, K, group, sym, affine)  # one weight, no x or y
    return 2 * w + M * K * 2 + M * N_each * 2
