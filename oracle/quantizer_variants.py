"""Variant ternary weight quantisers from the pages -- TEST INFRASTRUCTURE ONLY.

Plain CPU definitions, like the rest of this package: only the tests may use
them. They are options of the weight packing, not the default rule (which is
`absmean_gamma` + `ternary_codes`).

Sources (web pages; cited by title and section):

* [STE] "BitNet 中使用直通估计器工程化三元权重训练" (blog.hotdry.top,
  2025-10-04), section "STE 机制在三元训练中的作用": the scale alpha is 0.7
  times mean(|W|) and the quantised weight is clip(round(W / alpha), -1, 1)
  times alpha; section "工程化训练流程与参数配置", item "缩放因子与阈值": the
  same alpha, and a threshold tau = 0.1 alpha for the zero decision.
* [TWO] "BitNet 三元权重阈值优化工程实践" (blog.hotdry.top, 2025-09-08), section
  "三元权重阈值优化的核心原理": the threshold delta is 0.7 times mean(|W|);
  weights below it map to 0, the others to their sign; the factor may be
  raised to 0.75 (attention) or lowered to 0.6 (FFN). Its threshold module
  scales the ternary weights by the mean over all elements of |W| times the
  mask |W| > delta.

Readings (each also listed with its reason in the design notes):

* mean(|W|) is the exact mean rounded once to fp32, as for the default rule.
* factor x mean is one fp32 multiplication (round to nearest even) of the
  fp32 factor and the fp32 mean.
* [STE]: codes = clip(rint(fp32(W / alpha)), -1, 1) with ties to even, and the
  forward's scale is alpha. The zero threshold tau = 0.1 alpha changes no code:
  |W| < tau means |W / alpha| < 0.1, which already rounds to 0. An all-zero W
  gives alpha = 0 and all codes 0.
* [TWO]: codes = sign(W) where |W| > delta (strictly), else 0; the scale is
  the exact sum of |W| over the kept weights divided by the number of all
  weights (the mean of |W| times the mask, as the module computes it),
  rounded once to fp32.
"""

from __future__ import annotations

from typing import Tuple

import numpy as np

from .bitlinear_oracle import F32, absmean_gamma, exact_abs_sum, round_ratio_to_f32

#: the factor both pages give (0.7 x mean(|W|))
DEFAULT_FACTOR = F32(0.7)


def scaled_mean(w, factor=DEFAULT_FACTOR) -> np.float32:
    """fp32(factor x gamma), gamma the exact mean of |W| rounded once to fp32."""
    return F32(F32(factor) * absmean_gamma(w))


def alpha_round_quantize(w, factor=DEFAULT_FACTOR) -> Tuple[np.ndarray, np.float32]:
    """[STE] alpha = fp32(factor x mean|W|); codes = clip(rint(fp32(W / alpha)), -1, 1).

    Returns (codes int8 [N][K], alpha): the forward rescales by alpha.
    """
    w = np.asarray(w, dtype=np.float32)
    alpha = scaled_mean(w, factor)
    if alpha == 0:
        return np.zeros(w.shape, dtype=np.int8), alpha
    with np.errstate(over="ignore"):
        q = np.rint(w / alpha)          # fp32 division (RN); overflow gives +-inf, clipped below
    return np.clip(q, -1, 1).astype(np.int8), alpha


def threshold_quantize(w, factor=DEFAULT_FACTOR) -> Tuple[np.ndarray, np.float32]:
    """[TWO] delta = fp32(factor x mean|W|); codes = sign(W) [|W| > delta];
    alpha = mean(|W| [|W| > delta]) over all elements, exact, rounded once.

    Returns (codes int8 [N][K], alpha): the forward rescales by alpha.
    """
    w = np.asarray(w, dtype=np.float32)
    delta = scaled_mean(w, factor)
    keep = np.abs(w) > delta
    codes = (np.sign(w) * keep).astype(np.int8)
    kept_sum = exact_abs_sum(np.where(keep, w, F32(0.0)))
    mean = kept_sum / w.size
    return codes, round_ratio_to_f32(mean.numerator, mean.denominator)
