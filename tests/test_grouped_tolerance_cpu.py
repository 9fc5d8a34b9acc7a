"""The tolerance the per-group GPU parity tests use, checked on the host.

The per-group forward adds the exact products gamma[n][g] * acc[m][n][g] in
fp64 (eight partial sums over the groups g = w, w + 8, ..., added in order),
divides by s_m in fp64 and rounds to fp32. Against the oracle's exact value
rounded once, the difference is at most
    2^-23 |y_ref| + (K/64) 2^-52 sum_g |gamma * acc| / s + 2^-149.
This file replays that order of fp64 operations in numpy on oracle-derived
inputs, including sums that cancel and scales of very different size, and
checks the bound; it exercises no GPU code.
"""

from __future__ import annotations

import numpy as np
import pytest

import oracle

F32 = np.float32


def _fp64_order(acc, gam, s):
    """y as the contraction evaluates it: per (m, n), eight fp64 partials over
    g = w, w + 8, ... (exact products added with fma semantics: the product
    is exact in fp64), added in order, divided by s in fp64, rounded to fp32."""
    m_, n_, G = acc.shape
    y = np.empty((m_, n_), dtype=np.float32)
    for m in range(m_):
        for n in range(n_):
            parts = []
            for w in range(8):
                a = 0.0
                for g in range(w, G, 8):
                    a = a + float(gam[n, g]) * float(acc[m, n, g])   # product exact: 24 x 14 bits
                parts.append(a)
            v = 0.0
            for p in parts:
                v = v + p
            y[m, n] = np.float32(v / float(s[m]))
    return y


def _check(x, w):
    ref = oracle.bitlinear_forward_grouped(x, w)
    y = _fp64_order(ref["acc"], ref["gammas"], ref["scale"])
    bound = oracle.grouped_y_bound(ref["acc"], ref["gammas"], ref["scale"])
    k = w.shape[1]
    tol = 2.0 ** -23 * np.abs(ref["y"].astype(np.float64)) + (k // 64) * 2.0 ** -52 * bound + 2.0 ** -149
    err = np.abs(y.astype(np.float64) - ref["y"].astype(np.float64))
    assert (err <= tol).all(), float((err - tol).max())
    return err, tol


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_gaussian_within_bound(seed):
    rng = np.random.default_rng(900 + seed)
    w = (rng.standard_normal((6, 1024)) * 0.02).astype(np.float32)
    x = rng.standard_normal((3, 1024)).astype(np.float32)
    _check(x, w)


def test_cancellation_and_mixed_scales_within_bound():
    rng = np.random.default_rng(910)
    w = (rng.standard_normal((4, 2048)) * 0.02).astype(np.float32)
    w[0, :1024] = -w[0, 1024:]                 # the two halves of row 0 cancel for a symmetric x
    w[1, 64:128] *= F32(1e6)                   # one group far larger than the rest
    w[2, ::64] *= F32(1e-6)
    x = rng.standard_normal((2, 2048)).astype(np.float32)
    x[1, 1024:] = x[1, :1024]
    _check(x, w)
