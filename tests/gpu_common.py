"""Helpers for the GPU parity tests: run both sides on the same seeded inputs."""

from __future__ import annotations

import numpy as np
import torch

import oracle

F32 = np.float32


def x_to_oracle(x: torch.Tensor) -> np.ndarray:
    """The oracle's fp32 view of a CPU activation tensor (bf16 widened by the oracle)."""
    if x.dtype == torch.bfloat16:
        return oracle.bf16_bits_to_f32(x.view(torch.int16).numpy().view(np.uint16))
    return x.numpy().astype(np.float32)


def bits(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float32).view(np.uint32)


def oracle_weights(w: torch.Tensor):
    wn = w.numpy()
    g = oracle.absmean_gamma(wn)
    codes = oracle.ternary_codes(wn, g)
    return g, codes, oracle.pack_codes(codes)


def gpu_run(w: torch.Tensor, x: torch.Tensor, device="cuda"):
    import bit_ternary_forward_b300 as blt
    packed = blt.pack_weights(w.to(device))
    y, xq, s = blt.forward(x.to(device), packed, return_quant=True)
    acc = blt.gemm_i32(xq, packed.wp)
    torch.cuda.synchronize()
    return {"gamma": packed.gamma.cpu().numpy()[0], "packed": packed.wp.cpu().numpy(), "xq": xq.cpu().numpy(),
            "scale": s.cpu().numpy(), "acc": acc.cpu().numpy(), "y": y.cpu().numpy()}


def assert_y_close(y_gpu: np.ndarray, y_ref: np.ndarray, rel: float = 1e-6):
    """y within `rel` relative (absolute floor at the smallest normal)."""
    tol = rel * np.abs(y_ref).astype(np.float64) + 1.2e-38
    err = np.abs(y_gpu.astype(np.float64) - y_ref.astype(np.float64))
    bad = err > tol
    assert not bad.any(), f"{int(bad.sum())} outputs off by more than {rel} relative; max err {err.max()}"


def compare_full(w: torch.Tensor, x: torch.Tensor, g_run=None):
    """Every intermediate, bit for bit; y both bit-exact and within 1e-6 relative."""
    g_run = g_run or gpu_run(w, x)
    ref = oracle.bitlinear_forward(x_to_oracle(x), w.numpy())
    assert bits(g_run["gamma"]) == bits(ref["gamma"]), (g_run["gamma"], ref["gamma"])
    np.testing.assert_array_equal(g_run["packed"], ref["packed"])
    np.testing.assert_array_equal(g_run["xq"], ref["xq"])
    np.testing.assert_array_equal(bits(g_run["scale"]), bits(ref["scale"]))
    np.testing.assert_array_equal(g_run["acc"], ref["acc"])
    assert_y_close(g_run["y"], ref["y"])
    np.testing.assert_array_equal(bits(g_run["y"]), bits(ref["y"]))
    return ref


def compare_sampled_rows(w: torch.Tensor, x: torch.Tensor, rows, g_run=None):
    """Full weights/packing; activations, accumulators and outputs on sampled tokens."""
    g_run = g_run or gpu_run(w, x)
    gamma, codes, packed = oracle_weights(w)
    assert bits(g_run["gamma"]) == bits(gamma)
    np.testing.assert_array_equal(g_run["packed"], packed)
    xs = x_to_oracle(x)[rows]
    xq, s = oracle.quant_act(xs)
    np.testing.assert_array_equal(g_run["xq"][rows], xq)
    np.testing.assert_array_equal(bits(g_run["scale"][rows]), bits(s))
    acc = oracle.ternary_int8_matmul(xq, codes)
    np.testing.assert_array_equal(g_run["acc"][rows], acc)
    y = oracle.rescale(acc, gamma, s)
    assert_y_close(g_run["y"][rows], y)
    np.testing.assert_array_equal(bits(g_run["y"][rows]), bits(y))
