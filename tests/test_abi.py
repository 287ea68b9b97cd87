"""The C-ABI library builds, loads and exports every function include/w4a16.h
declares; argument checks that need no GPU return their status codes without
touching CUDA (no device is needed, so these run on CPU-only hosts too)."""
import ctypes
import os
import re

import pytest

import gemm_w4a16_group_gb300 as w4

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "w4a16.h")

OK, INVALID, MISALIGNED = 0, -1, -2


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(w4a16_[a-z_0-9]+)\s*\(", src)))


@pytest.fixture(scope="module")
def L():
    return w4.lib()


def test_exports_match_header(L):
    declared = _declared()
    assert declared, "no declarations parsed"
    assert sorted(w4.EXPORTS) == declared
    for name in declared:
        assert hasattr(L, name), name


def test_library_is_in_tree(L):
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    assert os.path.commonpath([w4.library_path(), root]) == root


def test_repacked_bytes_layout(L):
    # N=256, K=512, G=128: 16 tiles x 8 chunks x 512 B of codes, then one
    # 4-group block of scales per tile (128 B), then (asym) 32 B of zeros per tile
    assert w4.repacked_bytes(256, 512, 128, True) == 65536 + 2048
    assert w4.repacked_bytes(256, 512, 128, False) == 65536 + 2048 + 512
    # ragged N pads to 16 rows; every section is 256-byte aligned
    n = w4.repacked_bytes(250, 5120, 64, False)
    assert n % 256 == 0 and n == 16 * 80 * 512 + 16 * 20 * 128 + 16 * 20 * 32
    # gate/up: N_each padded to 128, two weights
    assert w4.gateup_repacked_bytes(100, 512, 128, True) == w4.repacked_bytes(256, 512, 128, True)
    for bad in [(0, 512, 128), (16, 512, 96), (16, 100, 64), (16, 32, 64), (16, 192, 128)]:
        assert w4.repacked_bytes(*bad, True) == 0


FAKE = 1 << 20  # an aligned non-null address; never dereferenced on these paths


def _gemm(L, x=FAKE, packed=FAKE, scales=None, zeros=None, M=4, N=64, K=128, group=64, sym=1, y=FAKE):
    P = ctypes.c_void_p
    return L.w4a16_gemm(P(x), P(packed), P(scales), P(zeros), M, N, K, group, sym, P(y), None)


def test_gemm_argument_checks(L):
    assert _gemm(L, x=None) == INVALID
    assert _gemm(L, y=None) == INVALID
    assert _gemm(L, packed=None) == INVALID
    assert _gemm(L, scales=FAKE) == INVALID       # reserved: must be NULL
    assert _gemm(L, zeros=FAKE) == INVALID
    assert _gemm(L, M=0) == INVALID
    assert _gemm(L, N=0) == INVALID
    assert _gemm(L, K=96, group=64) == INVALID    # K % G
    assert _gemm(L, group=32) == INVALID
    assert _gemm(L, K=0) == INVALID
    assert _gemm(L, x=FAKE + 8) == MISALIGNED
    assert _gemm(L, y=FAKE + 2) == MISALIGNED
    assert _gemm(L, packed=FAKE + 128) == MISALIGNED


def test_other_entry_points_argument_checks(L):
    P = ctypes.c_void_p
    assert L.w4a16_gateup_silu(P(FAKE), None, 4, 64, 128, 64, 1, P(FAKE), None) == INVALID
    assert L.w4a16_gateup_silu(P(FAKE), P(FAKE), 4, 64, 100, 64, 1, P(FAKE), None) == INVALID
    assert L.w4a16_gateup_silu(P(FAKE + 4), P(FAKE), 4, 64, 128, 64, 1, P(FAKE), None) == MISALIGNED
    assert L.w4a16_repack(None, P(FAKE), None, 64, 128, 64, 1, P(FAKE), None) == INVALID
    assert L.w4a16_repack(P(FAKE), P(FAKE), None, 64, 128, 64, 0, P(FAKE), None) == INVALID  # asym needs zeros
    assert L.w4a16_repack(P(FAKE), P(FAKE), None, 64, 128, 64, 1, P(FAKE + 16), None) == MISALIGNED
    assert L.w4a16_repack_gateup(P(FAKE), P(FAKE), None, None, P(FAKE), None, 64, 128, 64, 1,
                                 P(FAKE), None) == INVALID
    assert L.w4a16_dequantize(P(FAKE), 64, 128, 64, 1, None, None) == INVALID
    assert L.w4a16_dequantize(P(FAKE), 64, 128, 48, 1, P(FAKE), None) == INVALID


def test_strerror_and_override(L):
    for rc in (0, -1, -2, -3, -4, -5):
        assert len(w4.strerror(rc)) >= 2
    assert w4.strerror(-99) == "unknown status"
    prev = w4.set_kernel_override(w4.KERNEL_SMALLM)
    assert w4.set_kernel_override(prev) == w4.KERNEL_SMALLM
    assert w4.set_kernel_override(7) == -1
    assert w4.set_kernel_override(6) == -1
    prev = w4.set_kernel_override(w4.KERNEL_DECODE_TC)
    assert w4.set_kernel_override(prev) == w4.KERNEL_DECODE_TC


def test_programmatic_overlap_switch(L):
    assert L.w4a16_set_programmatic_overlap(2) == -1
    prev = L.w4a16_set_programmatic_overlap(1)
    assert prev in (0, 1)
    assert L.w4a16_set_programmatic_overlap(prev) == 1
    assert w4.set_programmatic_overlap(False) == bool(prev)
    assert w4.set_programmatic_overlap(prev) is False


def test_argmax_entry_point_argument_checks(L):
    P = ctypes.c_void_p
    g = L.w4a16_gemm_argmax
    assert g(None, P(FAKE), 4, 64, 128, 64, 1, P(FAKE), P(FAKE), None) == INVALID
    assert g(P(FAKE), P(FAKE), 4, 64, 128, 64, 1, P(FAKE), None, None) == INVALID     # no output
    assert g(P(FAKE), P(FAKE), 33, 64, 128, 64, 1, None, P(FAKE), None) == INVALID    # M > 32 needs y
    assert g(P(FAKE), P(FAKE), 4, 64, 96, 64, 1, None, P(FAKE), None) == INVALID      # K % G
    assert g(P(FAKE), P(FAKE), 4, 64, 128, 64, 1, None, P(FAKE + 4), None) == MISALIGNED
    assert g(P(FAKE), P(FAKE), 4, 64, 128, 64, 1, P(FAKE + 2), P(FAKE), None) == MISALIGNED


def test_topk_entry_points_argument_checks(L):
    P = ctypes.c_void_p
    t = L.w4a16_topk
    assert t(None, 2, 300, 8, P(FAKE), None, None) == INVALID                    # no y
    assert t(P(FAKE), 2, 300, 8, None, None, None) == INVALID                    # no idx
    assert t(P(FAKE), 2, 300, 0, P(FAKE), None, None) == INVALID                 # k < 1
    assert t(P(FAKE), 2, 300, 301, P(FAKE), None, None) == INVALID               # k > N
    assert t(P(FAKE), 2, 5000, 1025, P(FAKE), None, None) == INVALID             # k > 1024
    assert t(P(FAKE), 0, 300, 8, P(FAKE), None, None) == INVALID                 # M < 1
    assert t(P(FAKE + 1), 2, 300, 8, P(FAKE), None, None) == MISALIGNED          # y
    assert t(P(FAKE), 2, 300, 8, P(FAKE + 4), None, None) == MISALIGNED          # idx
    assert t(P(FAKE), 2, 300, 8, P(FAKE), P(FAKE + 1), None) == MISALIGNED       # vals
    g = L.w4a16_gemm_topk
    assert g(P(FAKE), P(FAKE), 2, 300, 128, 64, 1, 0, P(FAKE), P(FAKE), None, None) == INVALID
    assert g(P(FAKE), P(FAKE), 2, 300, 128, 64, 1, 8, None, P(FAKE), None, None) == INVALID   # y required
    assert g(P(FAKE), P(FAKE), 2, 300, 128, 64, 1, 8, P(FAKE), None, None, None) == INVALID   # no idx
    assert g(P(FAKE), P(FAKE), 2, 300, 96, 64, 1, 8, P(FAKE), P(FAKE), None, None) == INVALID  # K % G
    assert g(P(FAKE), P(FAKE), 2, 300, 128, 64, 1, 8, P(FAKE), P(FAKE + 4), None, None) == MISALIGNED


def test_affine_bits_sizes_and_argument_checks(L):
    P = ctypes.c_void_p
    rb = L.w4a16_affine_bits_repacked_bytes
    # 2-4 bits: the 4-bit affine layout; 5-8 bits: the layout of K' = 2K
    for bits in (2, 3, 4):
        assert rb(300, 512, 64, bits) == L.w4a16_repacked_bytes(300, 512, 64, 2)
    for bits in (5, 6, 7, 8):
        assert rb(300, 512, 64, bits) == L.w4a16_repacked_bytes(300, 1024, 64, 2)
    assert rb(300, 512, 64, 1) == 0 and rb(300, 512, 64, 9) == 0 and rb(300, 96, 64, 4) == 0
    sb = L.w4a16_affine_bits_scratch_bytes
    # the group-sum table (3 parts per group, rounded up to 64 columns), after
    # the widened x for 5-8 bits
    assert sb(3, 512, 64, 3) == 3 * 64 * 2
    assert sb(3, 512, 64, 8) == 3 * 2 * 512 * 2 + 3 * 64 * 2
    assert sb(300, 5120, 64, 6) == 300 * 2 * 5120 * 2 + 300 * 512 * 2  # 160 groups of the widened K
    assert sb(3, 512, 64, 1) == 0 and sb(0, 512, 64, 4) == 0
    r = L.w4a16_repack_affine_bits
    assert r(P(FAKE), P(FAKE), P(FAKE), 300, 512, 64, 1, P(FAKE), None) == INVALID
    assert r(P(FAKE), P(FAKE), None, 300, 512, 64, 5, P(FAKE), None) == INVALID
    assert r(P(FAKE), P(FAKE), P(FAKE), 300, 512, 64, 5, P(FAKE + 16), None) == MISALIGNED
    g = L.w4a16_gemm_affine_bits
    assert g(P(FAKE), None, P(FAKE), 4, 64, 512, 64, 6, P(FAKE), None) == INVALID        # no scratch
    assert g(P(FAKE), P(FAKE), P(FAKE), 4, 64, 512, 64, 9, P(FAKE), None) == INVALID     # bits
    assert g(P(FAKE), P(FAKE), P(FAKE), 4, 64, 96, 64, 6, P(FAKE), None) == INVALID      # K % G
    assert g(P(FAKE), P(FAKE + 16), P(FAKE), 4, 64, 512, 64, 6, P(FAKE), None) == MISALIGNED
    assert g(P(FAKE + 8), P(FAKE), P(FAKE), 4, 64, 512, 64, 6, P(FAKE), None) == MISALIGNED
    dq = L.w4a16_dequantize_affine_bits
    assert dq(P(FAKE), 64, 512, 64, 1, P(FAKE), None) == INVALID
    assert dq(None, 64, 512, 64, 3, P(FAKE), None) == INVALID


def test_affine_layout_and_argument_checks(L):
    P = ctypes.c_void_p
    # the bias section is the scales' size (N=256, K=512, G=128 -> 2048 B), then
    # the bias operand: 256 rows of 3 * 4 columns rounded up to 64, bf16
    assert w4.repacked_bytes(256, 512, 128, w4.AFFINE) == 65536 + 2048 + 2048 + 256 * 64 * 2
    assert w4.gateup_repacked_bytes(100, 512, 128, w4.AFFINE) == w4.repacked_bytes(256, 512, 128, w4.AFFINE)
    assert w4.repacked_bytes(256, 512, 128, 3) == 0  # no such form
    # group sums: M rows of 3 * K/G bf16 parts rounded up to 64
    assert w4.xsum_bytes(17, 512, 64) == 17 * 64 * 2
    assert w4.xsum_bytes(300, 5120, 128) == 300 * 128 * 2
    assert w4.xsum_bytes(4, 5120, 64) == 4 * 256 * 2
    assert w4.xsum_bytes(0, 512, 64) == 0 and w4.xsum_bytes(4, 100, 64) == 0
    # the zero-point calls reject the affine form, and the affine repack needs biases
    assert _gemm(L, sym=2) == INVALID
    assert L.w4a16_gateup_silu(P(FAKE), P(FAKE), 4, 64, 128, 64, 2, P(FAKE), None) == INVALID
    assert L.w4a16_gemm_argmax(P(FAKE), P(FAKE), 4, 64, 128, 64, 2, None, P(FAKE), None) == INVALID
    assert L.w4a16_repack(P(FAKE), P(FAKE), P(FAKE), 64, 128, 64, 2, P(FAKE), None) == INVALID
    assert L.w4a16_repack_affine(P(FAKE), P(FAKE), None, 64, 128, 64, P(FAKE), None) == INVALID
    assert L.w4a16_repack_affine(P(FAKE), P(FAKE), P(FAKE + 1), 64, 128, 64, P(FAKE), None) == MISALIGNED
    assert L.w4a16_repack_affine_gateup(P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), None, 64, 128, 64,
                                        P(FAKE), None) == INVALID
    # M > 32 runs the tcgen05 GEMM, which reads the group sums: they are required
    ga = L.w4a16_gemm_affine
    assert ga(P(FAKE), None, P(FAKE), 33, 64, 128, 64, P(FAKE), None) == INVALID
    assert ga(P(FAKE), P(FAKE + 4), P(FAKE), 33, 64, 128, 64, P(FAKE), None) == MISALIGNED
    assert ga(P(FAKE), P(FAKE), P(FAKE), 33, 64, 96, 64, P(FAKE), None) == INVALID
    assert L.w4a16_gateup_silu_affine(P(FAKE), None, P(FAKE), 300, 64, 128, 64, P(FAKE), None) == INVALID
    assert L.w4a16_xsum(P(FAKE), 4, 128, 64, None, None) == INVALID
    assert L.w4a16_xsum(P(FAKE), 4, 128, 64, P(FAKE + 8), None) == MISALIGNED


def test_noalloc_entry_point_argument_checks(L):
    # the no-alloc affine GEMM keeps its group sums in a fixed 4 MiB device
    # array: at K = 5120, group 64 a row of sums is 256 bf16 (512 B), so
    # M = 8192 fills it exactly and M = 8193 is refused before any CUDA call
    P = ctypes.c_void_p
    na = L.w4a16_gemm_affine_noalloc
    assert w4.xsum_bytes(8192, 5120, 64) == 4 << 20
    assert w4.xsum_bytes(8193, 5120, 64) > 4 << 20
    assert na(P(FAKE), P(FAKE), 8193, 64, 5120, 64, P(FAKE), None) == INVALID
    assert na(P(FAKE), P(FAKE), 16385, 64, 5120, 128, P(FAKE), None) == INVALID
    assert na(None, P(FAKE), 4, 64, 128, 64, P(FAKE), None) == INVALID
    assert na(P(FAKE), None, 4, 64, 128, 64, P(FAKE), None) == INVALID
    assert na(P(FAKE), P(FAKE), 4, 64, 128, 64, None, None) == INVALID
    assert na(P(FAKE), P(FAKE), 0, 64, 128, 64, P(FAKE), None) == INVALID
    assert na(P(FAKE), P(FAKE), 4, 64, 96, 64, P(FAKE), None) == INVALID     # K % G
    assert na(P(FAKE), P(FAKE), 4, 64, 128, 32, P(FAKE), None) == INVALID    # group
    assert na(P(FAKE + 8), P(FAKE), 4, 64, 128, 64, P(FAKE), None) == MISALIGNED
    assert na(P(FAKE), P(FAKE + 128), 4, 64, 128, 64, P(FAKE), None) == MISALIGNED
    assert na(P(FAKE), P(FAKE), 40, 64, 128, 64, P(FAKE + 2), None) == MISALIGNED
