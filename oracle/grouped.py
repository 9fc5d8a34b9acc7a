"""Per-group weight quantisation (group size 64) for the BitLinear forward.

TEST INFRASTRUCTURE ONLY -- like the rest of this package, nothing on the
product path may import this module.

Source: [HPFT] "BitNet 1-bit LLM 的混合精度微调技术：渐进量化策略"
(blog.hotdry.top), body text, which names per-group quantisation with a group
size of 64 as a way to keep the quantisation error local. The page gives no
axis and no formula beyond the group size; the readings taken here (each is
listed in the repository's design notes):

* A group is 64 consecutive input features k of one weight row n:
  W[n, 64g : 64g + 64]. This is the axis the dot product sums over, so one
  scale multiplies one partial sum.
* Each group's scale is the per-tensor rule applied to the group: gamma_{n,g}
  = the exact mean of |W| over its 64 values, rounded once to fp32 (ties to
  even); codes = clip(rint(fp32(W / fp32(gamma_{n,g} + 1e-5))), -1, 1).
* The packed codes keep the per-tensor layout; the scales are fp32
  [N][K / 64], row-major.
* The output is y[m][n] = sum_g gamma_{n,g} * acc_{m,n,g} / s_m, with
  acc_{m,n,g} = sum_{k in g} code * x_q, evaluated exactly and rounded once
  to fp32 (ties to even). A per-tensor scale factors out of the sum and the
  forward rounds twice (acc * gamma, then / s); with one scale per group the
  sum itself must be evaluated, and its exact value rounded once is the only
  reading that does not depend on a summation order.
"""

from __future__ import annotations

from fractions import Fraction

import numpy as np

from .bitlinear_oracle import (EPS_GAMMA, F32, absmean_gamma, quant_act, round_ratio_to_f32,
                               ternary_codes)

GROUP = 64


def group_gammas(w, group: int = GROUP) -> np.ndarray:
    """gamma_{n,g}: absmean_gamma (exact mean, one rounding) of each group of
    `group` consecutive k of each row; fp32 [N][K / group]."""
    w = np.asarray(w, dtype=np.float32)
    n, k = w.shape
    if k % group:
        raise ValueError("group_gammas: K must be a multiple of the group size")
    out = np.empty((n, k // group), dtype=np.float32)
    for r in range(n):
        for g in range(k // group):
            out[r, g] = absmean_gamma(w[r, g * group:(g + 1) * group])
    return out


def group_codes(w, gammas, eps=EPS_GAMMA, group: int = GROUP) -> np.ndarray:
    """clip(rint(W / fp32(gamma_{n,g} + eps)), -1, 1) per group, int8 [N][K]."""
    w = np.asarray(w, dtype=np.float32)
    n, k = w.shape
    codes = np.empty((n, k), dtype=np.int8)
    for g in range(k // group):
        sl = slice(g * group, (g + 1) * group)
        for r in range(n):
            codes[r, sl] = ternary_codes(w[r, sl], gammas[r, g], eps)
    return codes


def group_accumulators(xq, codes, group: int = GROUP) -> np.ndarray:
    """acc_{m,n,g} = sum over the group of code * x_q, exact; int64 [M][N][G]."""
    xq = np.asarray(xq, dtype=np.int64)
    codes = np.asarray(codes, dtype=np.int64)
    m, k = xq.shape
    n = codes.shape[0]
    g_count = k // group
    acc = np.empty((m, n, g_count), dtype=np.int64)
    for g in range(g_count):
        sl = slice(g * group, (g + 1) * group)
        acc[:, :, g] = xq[:, sl] @ codes[:, sl].T
    return acc


def _round_fraction_to_f32(v: Fraction) -> np.float32:
    """The fp32 value nearest to the rational v, ties to even (sign kept)."""
    if v == 0:
        return F32(0.0)
    mag = round_ratio_to_f32(abs(v.numerator), v.denominator)
    return F32(-mag) if v < 0 else mag


def grouped_rescale(acc, gammas, s) -> np.ndarray:
    """y[m][n] = fp32(exact(sum_g gamma_{n,g} * acc_{m,n,g}) / s_m): one rounding."""
    acc = np.asarray(acc, dtype=np.int64)
    m, n, _ = acc.shape
    gam = [[Fraction(float(v)) for v in row] for row in np.asarray(gammas, dtype=np.float32)]
    s = np.asarray(s, dtype=np.float32)
    y = np.empty((m, n), dtype=np.float32)
    for i in range(m):
        si = Fraction(float(s[i]))
        for j in range(n):
            t = sum((gam[j][g] * int(acc[i, j, g]) for g in range(acc.shape[2])), Fraction(0))
            y[i, j] = _round_fraction_to_f32(t / si)
    return y


def bitlinear_forward_grouped(x, w, group: int = GROUP):
    """All steps of the per-group forward; returns every intermediate."""
    gammas = group_gammas(w, group)
    codes = group_codes(w, gammas, group=group)
    xq, s = quant_act(x)
    acc = group_accumulators(xq, codes, group)
    y = grouped_rescale(acc, gammas, s)
    return {"gammas": gammas, "codes": codes, "xq": xq, "scale": s, "acc": acc, "y": y}


def grouped_y_bound(acc, gammas, s) -> np.ndarray:
    """sum_g |gamma_{n,g} * acc_{m,n,g}| / s_m in fp64: the magnitude against
    which a kernel's summation error is measured (cancellation can make y far
    smaller than its terms)."""
    acc = np.asarray(acc, dtype=np.float64)
    g = np.asarray(gammas, dtype=np.float64)
    return np.einsum("mng,ng->mn", np.abs(acc), np.abs(g)) / np.asarray(s, dtype=np.float64)[:, None]
