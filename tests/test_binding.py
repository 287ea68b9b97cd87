"""The Python binding's own checks, on CPU: every buffer a call reads or
writes must hold the bytes the call needs (the C ABI takes plain pointers and
cannot tell), index_out must be int64, all tensors must share one device, and
the arguments reach the C entry point in the header's order.

The compute entry points are replaced by a recorder (no CUDA call is made);
the size queries are the real library's."""
import ctypes

import pytest
import torch

import gemm_w4a16_group_gb300 as w4

BF = torch.bfloat16


class FakeLib:
    def __init__(self, real):
        self.real = real
        self.calls = []

    def __getattr__(self, name):
        if name.endswith("_bytes") or name in ("w4a16_strerror", "w4a16_last_cuda_error"):
            return getattr(self.real, name)

        def record(*args):
            self.calls.append((name, args))
            return 0

        return record


@pytest.fixture
def fake(monkeypatch):
    f = FakeLib(w4.lib())
    monkeypatch.setattr(w4, "lib", lambda auto_build=True: f)
    monkeypatch.setattr(w4, "_is_device_tensor", lambda t: True)
    monkeypatch.setattr(w4, "_stream", lambda stream, device=None: ctypes.c_void_p(0))
    return f


def _v(p):
    return None if p is None else p.value


def _canon(N, K, G, zeros=True):
    q = torch.zeros((N, K // 8), dtype=torch.int32)
    s = torch.zeros((N, K // G), dtype=BF)
    z = torch.zeros((N, (K // G + 7) // 8), dtype=torch.int32) if zeros else None
    return q, s, z


def test_gemm_marshals_in_header_order(fake):
    M, N, K, G = 3, 48, 256, 64
    x = torch.zeros((M, K), dtype=BF)
    packed = torch.zeros(w4.repacked_bytes(N, K, G, False), dtype=torch.uint8)
    y = w4.gemm(x, packed, N, K, G, False)
    name, a = fake.calls[-1]
    assert name == "w4a16_gemm"
    assert _v(a[0]) == x.data_ptr() and _v(a[1]) == packed.data_ptr()
    assert a[2] is None and a[3] is None
    assert a[4:9] == (M, N, K, G, 0)
    assert _v(a[9]) == y.data_ptr() and tuple(y.shape) == (M, N) and y.dtype == BF


def test_gemm_rejects_short_buffers(fake):
    M, N, K, G = 3, 48, 256, 64
    x = torch.zeros((M, K), dtype=BF)
    need = w4.repacked_bytes(N, K, G, True)
    with pytest.raises(ValueError, match="packed holds"):
        w4.gemm(x, torch.zeros(need - 1, dtype=torch.uint8), N, K, G, True)
    packed = torch.zeros(need, dtype=torch.uint8)
    with pytest.raises(ValueError, match="out holds"):
        w4.gemm(x, packed, N, K, G, True, out=torch.zeros((M, N - 1), dtype=BF))
    with pytest.raises(ValueError, match="x must be"):
        w4.gemm(torch.zeros((M, K - 8), dtype=BF), packed, N, K, G, True)
    # a larger buffer is fine
    w4.gemm(x, torch.zeros(need + 512, dtype=torch.uint8), N, K, G, True)
    assert fake.calls[-1][0] == "w4a16_gemm"
    assert len(fake.calls) == 1


def test_argmax_index_buffer(fake):
    M, N, K, G = 4, 64, 128, 64
    x = torch.zeros((M, K), dtype=BF)
    packed = torch.zeros(w4.repacked_bytes(N, K, G, True), dtype=torch.uint8)
    with pytest.raises(TypeError, match="index_out"):
        w4.gemm_argmax(x, packed, N, K, G, True, index_out=torch.zeros(M, dtype=torch.int32))
    with pytest.raises(ValueError, match="index_out holds"):
        w4.gemm_argmax(x, packed, N, K, G, True, index_out=torch.zeros(M - 1, dtype=torch.int64))
    idx, y = w4.gemm_argmax(x, packed, N, K, G, True)
    assert y is None and idx.dtype == torch.int64 and idx.numel() == M
    name, a = fake.calls[-1]
    assert name == "w4a16_gemm_argmax" and a[7] is None and _v(a[8]) == idx.data_ptr()
    # M > 32 stores the logits
    x40 = torch.zeros((40, K), dtype=BF)
    idx, y = w4.gemm_argmax(x40, packed, N, K, G, True)
    assert tuple(y.shape) == (40, N)


def test_gateup_sizes(fake):
    M, N_each, K, G = 2, 100, 128, 64
    x = torch.zeros((M, K), dtype=BF)
    need = w4.gateup_repacked_bytes(N_each, K, G, True)
    assert need > w4.repacked_bytes(N_each, K, G, True)
    with pytest.raises(ValueError, match="packed holds"):
        w4.gateup_silu(x, torch.zeros(need - 256, dtype=torch.uint8), N_each, K, G, True)
    h = w4.gateup_silu(x, torch.zeros(need, dtype=torch.uint8), N_each, K, G, True)
    assert tuple(h.shape) == (M, N_each)
    q, s, z = _canon(N_each, K, G, zeros=False)
    w4.repack_gateup(q, s, None, q, s, None, N_each, K, G, True)
    with pytest.raises(ValueError, match="qw_up holds"):
        w4.repack_gateup(q, s, None, q[:-1], s, None, N_each, K, G, True)


def test_repack_canonical_sizes(fake):
    N, K, G = 40, 256, 64
    q, s, z = _canon(N, K, G)
    out = w4.repack(q, s, z, N, K, G, False)
    assert out.numel() == w4.repacked_bytes(N, K, G, False)
    name, a = fake.calls[-1]
    assert name == "w4a16_repack" and a[3:7] == (N, K, G, 0) and _v(a[7]) == out.data_ptr()
    w4.repack(q, s, None, N, K, G, True)  # symmetric: no zeros
    with pytest.raises(ValueError, match="qweight holds"):
        w4.repack(q[:-1], s, z, N, K, G, False)
    with pytest.raises(ValueError, match="scales holds"):
        w4.repack(q, s[:, :-1].contiguous(), z, N, K, G, False)
    with pytest.raises(ValueError, match="zeros holds"):
        w4.repack(q, s, z[:-1], N, K, G, False)
    with pytest.raises(ValueError, match="out holds"):
        w4.repack(q, s, z, N, K, G, False, out=torch.zeros(out.numel() - 1, dtype=torch.uint8))
    with pytest.raises(TypeError, match="scales"):
        w4.repack(q, s.float(), z, N, K, G, False)
    with pytest.raises(ValueError, match="contiguous"):
        w4.repack(q, torch.zeros((K // G, N), dtype=BF).t(), z, N, K, G, False)


def test_affine_sizes(fake):
    M, N, K, G = 40, 64, 256, 64
    q, s, _ = _canon(N, K, G, zeros=False)
    b = torch.zeros_like(s)
    w4.repack_affine(q, s, b, N, K, G)
    with pytest.raises(ValueError, match="biases holds"):
        w4.repack_affine(q, s, b[:-1], N, K, G)
    w4.repack_affine_gateup(q, s, b, q, s, b, N, K, G)
    with pytest.raises(ValueError, match="b_up holds"):
        w4.repack_affine_gateup(q, s, b, q, s, b[:-1], N, K, G)
    x = torch.zeros((M, K), dtype=BF)
    xs = w4.xsum(x, K, G)
    assert xs.numel() * 2 == w4.xsum_bytes(M, K, G)
    with pytest.raises(ValueError, match="out holds"):
        w4.xsum(x, K, G, out=torch.zeros(xs.numel() - 1, dtype=BF))
    packed = torch.zeros(w4.repacked_bytes(N, K, G, w4.AFFINE), dtype=torch.uint8)
    w4.gemm_affine(x, packed, N, K, G, xs)
    name, a = fake.calls[-1]
    assert name == "w4a16_gemm_affine" and _v(a[1]) == xs.data_ptr() and a[3:7] == (M, N, K, G)
    with pytest.raises(ValueError, match="xsum holds"):
        w4.gemm_affine(x, packed, N, K, G, xs[:-1])
    with pytest.raises(ValueError, match="packed holds"):
        w4.gemm_affine(x, packed[:-256], N, K, G, xs)
    # the zero-point layout of the same weight is smaller than the affine one
    with pytest.raises(ValueError, match="packed holds"):
        w4.gemm_affine(x, torch.zeros(w4.repacked_bytes(N, K, G, True), dtype=torch.uint8), N, K, G, xs)
    w4.gemm_affine(x[:8].contiguous(), packed, N, K, G)  # M <= 32: no table
    assert fake.calls[-1][1][1] is None
    w4.gemm_affine_noalloc(x, packed, N, K, G)
    assert fake.calls[-1][0] == "w4a16_gemm_affine_noalloc"
    pg = torch.zeros(w4.gateup_repacked_bytes(N, K, G, w4.AFFINE), dtype=torch.uint8)
    h = w4.gateup_silu_affine(x, pg, N, K, G, xs)
    assert tuple(h.shape) == (M, N)
    with pytest.raises(ValueError, match="packed holds"):
        w4.gateup_silu_affine(x, packed, N, K, G, xs)


def test_dequantize_size_and_devices(fake):
    N, K, G = 48, 128, 64
    packed = torch.zeros(w4.repacked_bytes(N, K, G, False), dtype=torch.uint8)
    w = w4.dequantize(packed, N, K, G, False)
    assert tuple(w.shape) == (N, K) and w.dtype == torch.float32
    with pytest.raises(ValueError, match="packed holds"):
        w4.dequantize(packed, N + 16, K, G, False)
    # every tensor of a call on the device of x
    x = torch.zeros((2, K), dtype=BF)
    with pytest.raises(ValueError, match="is on meta"):
        w4.gemm(x, torch.empty(packed.numel(), dtype=torch.uint8, device="meta"), N, K, G, False)


def test_stream_requires_current_device(monkeypatch):
    # checked when more than one device is visible (with one, every CUDA
    # tensor is on the current device)
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    monkeypatch.setattr(w4, "_device_count", lambda: 2)

    class S:
        cuda_stream = 1234

    assert w4._stream(S(), torch.device("cuda", 0)).value == 1234
    with pytest.raises(ValueError, match="current CUDA device"):
        w4._stream(S(), torch.device("cuda", 1))
