"""The Python binding's marshalling, on the host: every wrapper runs against a
stand-in for the library that records its calls, with CPU tensors in place
of device tensors (the CUDA-tensor check is lifted for this test only). This
checks which pointers, sizes and codes each wrapper passes, that outputs the
caller supplies are used, and that wrong ones are refused before any call."""

from __future__ import annotations

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


class FakeLib:
    """Records every call; workspace queries answer 1024 bytes; every call succeeds."""

    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        if not name.startswith("bitlinear_"):
            raise AttributeError(name)

        def fn(*args):
            self.calls.append((name, args))
            if name.endswith("_workspace_bytes"):
                return 1024
            if name in ("bitlinear_last_error", "bitlinear_strerror"):
                return b""
            return 0
        return fn


@pytest.fixture
def fake(monkeypatch):
    import importlib.util
    spec = importlib.util.spec_from_file_location("bl_build", os.path.join(ROOT, "bit_ternary_forward_b300", "build.py"))
    build = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(build)
    build.build()
    import torch
    import bit_ternary_forward_b300 as blt

    def cpu_ok(t, name, dtype=None):
        if dtype is not None and t.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        return t

    lib = FakeLib()
    monkeypatch.setattr(blt, "lib", lib)
    monkeypatch.setattr(blt, "_cuda", cpu_ok)
    monkeypatch.setattr(blt, "_stream", lambda device: 77)
    return blt, lib, torch


def last(lib, name):
    got = [a for n, a in lib.calls if n == name]
    assert got, f"{name} was not called"
    return got[-1]


def test_pack_weights_marshalling(fake):
    blt, lib, torch = fake
    w = torch.zeros(8, 16)
    p = blt.pack_weights(w)
    assert p.wp.shape == (8, 4) and p.wp.dtype == torch.uint8 and p.gamma.shape == (1,) and (p.n, p.k) == (8, 16)
    a = last(lib, "bitlinear_pack_weights")
    assert a[:5] == (w.data_ptr(), 8, 16, p.wp.data_ptr(), p.gamma.data_ptr())
    assert a[5] % 256 == 0 and a[6] == 1024 and a[7] == 77
    out = blt.PackedWeight(torch.empty(8, 4, dtype=torch.uint8), torch.empty(1), 8, 16)
    assert blt.pack_weights(w, out=out) is out
    blt.pack_weights(w, quantizer="threshold", factor=0.6)
    a = last(lib, "bitlinear_pack_weights_quantizer")
    assert a[3] == blt.QUANTIZERS["threshold"] and abs(a[4] - 0.6) < 1e-7
    with pytest.raises(ValueError):
        blt.pack_weights(w, out=blt.PackedWeight(torch.empty(8, 3, dtype=torch.uint8), torch.empty(1), 8, 16))
    with pytest.raises(TypeError):
        blt.pack_weights(w, out=blt.PackedWeight(torch.empty(8, 4, dtype=torch.uint8), torch.empty(1, dtype=torch.float64), 8, 16))
    with pytest.raises(ValueError):
        blt.pack_weights(w, quantizer="per_group")


def test_absmean_and_quantize_pack_marshalling(fake):
    blt, lib, torch = fake
    w = torch.zeros(8, 16)
    g = blt.absmean(w)
    assert last(lib, "bitlinear_absmean")[:4] == (w.data_ptr(), 8, 16, g.data_ptr())
    wp = blt.quantize_pack(w, g)
    assert last(lib, "bitlinear_quantize_pack") == (w.data_ptr(), 8, 16, g.data_ptr(), wp.data_ptr(), 77)
    with pytest.raises(ValueError):
        blt.quantize_pack(w, g, wp=torch.empty(4, 8, dtype=torch.uint8))
    with pytest.raises(ValueError):
        blt.absmean(w, gamma=torch.empty(2))


def test_quant_act_marshalling(fake):
    blt, lib, torch = fake
    x = torch.zeros(4, 16, dtype=torch.bfloat16)
    xq, s = blt.quant_act(x)
    assert last(lib, "bitlinear_quant_act") == (x.data_ptr(), blt.BL_BF16, 4, 16, xq.data_ptr(), s.data_ptr(), 77)
    xq2, s2 = torch.empty(4, 16, dtype=torch.int8), torch.empty(4)
    assert blt.quant_act(x.float(), xq=xq2, scale=s2)[0] is xq2
    assert last(lib, "bitlinear_quant_act")[1] == blt.BL_F32
    with pytest.raises(ValueError):
        blt.quant_act(x, scale=torch.empty(3))
    with pytest.raises(TypeError):
        blt.quant_act(x.half())


def test_forward_marshalling(fake):
    blt, lib, torch = fake
    packed = blt.PackedWeight(torch.zeros(8, 4, dtype=torch.uint8), torch.ones(1), 8, 16)
    x = torch.zeros(3, 16, dtype=torch.bfloat16)
    y = blt.forward(x, packed)
    a = last(lib, "bitlinear_forward")
    assert a[:8] == (x.data_ptr(), blt.BL_BF16, 3, packed.wp.data_ptr(), packed.gamma.data_ptr(), 8, 16, y.data_ptr())
    assert a[8] is None and a[9] is None and a[11] == 1024 and a[12] == 77
    y2, xq, s = blt.forward(x, packed, return_quant=True)
    a = last(lib, "bitlinear_forward")
    assert a[8] == xq.data_ptr() and a[9] == s.data_ptr() and xq.shape == (3, 16) and s.shape == (3,)
    mine = torch.empty(3, 8)
    assert blt.forward(x, packed, y=mine) is mine
    with pytest.raises(ValueError):
        blt.forward(x, packed, y=torch.empty(3, 7))
    with pytest.raises(ValueError):
        blt.forward(torch.zeros(3, 12, dtype=torch.bfloat16), packed)


def test_gemm_marshalling(fake):
    blt, lib, torch = fake
    packed = blt.PackedWeight(torch.zeros(8, 4, dtype=torch.uint8), torch.ones(1), 8, 16)
    xq, s = torch.zeros(3, 16, dtype=torch.int8), torch.ones(3)
    y = blt.gemm(xq, s, packed)
    a = last(lib, "bitlinear_gemm")
    assert a[:8] == (xq.data_ptr(), s.data_ptr(), 3, packed.wp.data_ptr(), packed.gamma.data_ptr(), 8, 16, y.data_ptr())
    with pytest.raises(ValueError):
        blt.gemm(xq, torch.ones(2), packed)
    acc = blt.gemm_i32(xq, packed.wp)
    a = last(lib, "bitlinear_gemm_i32")
    assert a[:6] == (xq.data_ptr(), packed.wp.data_ptr(), 3, 8, 16, acc.data_ptr()) and acc.dtype == torch.int32
    mine = torch.empty(3, 8, dtype=torch.int32)
    assert blt.gemm_i32(xq, packed.wp, acc=mine) is mine
    with pytest.raises(ValueError):
        blt.gemm_i32(xq, torch.zeros(8, 3, dtype=torch.uint8))
    with pytest.raises(TypeError):
        blt.gemm_i32(xq, packed.wp, acc=torch.empty(3, 8))


def test_grouped_marshalling(fake):
    blt, lib, torch = fake
    w = torch.zeros(8, 128)
    p = blt.pack_weights_grouped(w)
    assert p.wp.shape == (8, 32) and p.gammas.shape == (8, 2) and p.gammas.dtype == torch.float32
    a = last(lib, "bitlinear_pack_weights_grouped")
    assert a == (w.data_ptr(), 8, 128, p.wp.data_ptr(), p.gammas.data_ptr(), 77)
    out = blt.PackedGrouped(torch.empty(8, 32, dtype=torch.uint8), torch.empty(8, 2), 8, 128)
    assert blt.pack_weights_grouped(w, out=out) is out
    with pytest.raises(ValueError):
        blt.pack_weights_grouped(w, out=blt.PackedGrouped(out.wp, torch.empty(8, 3), 8, 128))
    x = torch.zeros(3, 128, dtype=torch.bfloat16)
    y, xq, s = blt.forward_grouped(x, p, return_quant=True)
    assert y.shape == (3, 8) and xq.shape == (3, 128) and s.shape == (3,)
    a = last(lib, "bitlinear_forward_grouped")
    assert a[:8] == (x.data_ptr(), blt.BL_BF16, 3, p.wp.data_ptr(), p.gammas.data_ptr(), 8, 128, y.data_ptr())
    assert a[8] == xq.data_ptr() and a[9] == s.data_ptr() and a[10] % 256 == 0 and a[11] == 1024 and a[12] == 77
    with pytest.raises(ValueError):
        blt.forward_grouped(torch.zeros(3, 64), p)


def test_forward_lut_marshalling(fake):
    blt, lib, torch = fake
    p = blt.PackedWeight(torch.empty(8, 32, dtype=torch.uint8), torch.empty(1), 8, 128)
    x = torch.zeros(1, 128)
    y = blt.forward_lut(x, p)
    assert y.shape == (1, 8)
    a = last(lib, "bitlinear_forward_lut")
    assert a == (x.data_ptr(), blt.BL_F32, 1, p.wp.data_ptr(), p.gamma.data_ptr(), 8, 128, y.data_ptr(), 77)
    with pytest.raises(ValueError):
        blt.forward_lut(torch.zeros(1, 64), p)
