"""Pins of the variant weight quantisers of the oracle (CPU only).

[STE] "BitNet 中使用直通估计器工程化三元权重训练", sections "STE 机制在三元训练中的作用"
and "工程化训练流程与参数配置" (alpha = 0.7 mean|W|, clip(round(W / alpha), -1, 1)).
[TWO] "BitNet 三元权重阈值优化工程实践", section "三元权重阈值优化的核心原理" and its
threshold module (delta = 0.7 mean|W|, sign(W) [|W| > delta], alpha = mean(|W| mask)).

Each pin takes the two quantisers as arguments; the planted-mistake cases at the
end run the same pins on broken copies and require every copy to fail one.
"""

from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
from pins import frac_f32, nearest_f32, rint_half_even

F32 = np.float32
SEVEN = Fraction(float(F32(0.7)))    # the fp32 factor 0.7, exactly


# ---------------------------------------------------------------- independent reference (rationals)
def _mean_abs(w) -> Fraction:
    return sum((abs(frac_f32(v)) for v in np.asarray(w, dtype=F32).ravel()), Fraction(0)) / w.size


def _ref_alpha_round(w, factor=SEVEN):
    alpha = nearest_f32(factor * frac_f32(nearest_f32(_mean_abs(w))))
    if alpha == 0:
        return np.zeros(w.shape, np.int8), alpha
    a = frac_f32(alpha)
    codes = [max(-1, min(1, rint_half_even(frac_f32(nearest_f32(frac_f32(v) / a))))) for v in w.ravel()]
    return np.array(codes, np.int8).reshape(w.shape), alpha


def _ref_threshold(w, factor=SEVEN):
    delta = frac_f32(nearest_f32(factor * frac_f32(nearest_f32(_mean_abs(w)))))
    codes, kept = [], Fraction(0)
    for v in w.ravel():
        fv = frac_f32(v)
        keep = abs(fv) > delta
        codes.append((1 if fv > 0 else -1) if keep else 0)
        kept += abs(fv) if keep else 0
    return np.array(codes, np.int8).reshape(w.shape), nearest_f32(kept / w.size)


# ---------------------------------------------------------------- pins
def pin_bruteforce_small(ar, th):
    rng = np.random.default_rng(7)
    for scale in (1.0, 0.02, 3e-20, 7e20):
        for shape in ((1, 4), (3, 8), (5, 12)):
            w = (rng.standard_normal(shape) * scale).astype(F32)
            c, a = ar(w)
            rc, ra = _ref_alpha_round(w)
            assert np.array_equal(c, rc) and F32(a) == ra, ("alpha-round", scale, shape)
            c, a = th(w)
            rc, ra = _ref_threshold(w)
            assert np.array_equal(c, rc) and F32(a) == ra, ("threshold", scale, shape)


def pin_closed_forms(ar, th):
    """Gaussian N(0, s^2): mean|W| = s sqrt(2/pi); [STE] zeroes |Z| <= 0.35 sqrt(2/pi),
    [TWO] zeroes |Z| <= c = 0.7 sqrt(2/pi) and its alpha is s E[|Z| 1{|Z| > c}] = 2 s phi(c)."""
    n = 1 << 22
    w = (np.random.default_rng(11).standard_normal((1024, n // 1024)) * 0.02).astype(F32)
    p6 = math.erf(0.35 * math.sqrt(2 / math.pi) / math.sqrt(2))        # 0.2200
    c = 0.7 * math.sqrt(2 / math.pi)
    p7 = math.erf(c / math.sqrt(2))                                     # 0.4235
    tol = lambda p: 6 * math.sqrt(p * (1 - p) / n)                      # noqa: E731
    codes, _ = ar(w)
    assert abs(float((codes == 0).mean()) - p6) < tol(p6)
    codes, alpha = th(w)
    assert abs(float((codes == 0).mean()) - p7) < tol(p7)
    want = 2 * math.exp(-c * c / 2) / math.sqrt(2 * math.pi) * 0.02       # 0.6827 s
    assert abs(float(alpha) - want) < 0.002 * want


def pin_ties(ar, th):
    """[STE]: an element exactly at alpha/2 rounds to 0 (half to even), one at
    3 alpha/2 rounds to 2 and clips to 1. [TWO]: an element equal to delta is
    below the strict threshold."""
    rng = np.random.default_rng(5)
    base = (rng.standard_normal((64, 64)) * 0.02).astype(F32)
    w = base.copy()
    for _ in range(4):                      # alpha barely moves when two elements change
        alpha = oracle.scaled_mean(w)
        w[0, 0], w[0, 1] = F32(alpha * F32(0.5)), F32(-alpha * F32(1.5))
    assert oracle.scaled_mean(w) == alpha
    c, a = ar(w)
    assert a == alpha and c[0, 0] == 0 and c[0, 1] == -1
    w = base.copy()
    for _ in range(4):
        delta = oracle.scaled_mean(w)
        w[1, 0], w[1, 1] = delta, np.nextafter(delta, F32(1))
    assert oracle.scaled_mean(w) == delta
    c, _ = th(w)
    assert c[1, 0] == 0 and c[1, 1] == 1


def pin_invariances(ar, th):
    """Powers of two scale alpha exactly and leave every code; negation flips codes."""
    w = (np.random.default_rng(3).standard_normal((32, 48)) * 0.02).astype(F32)
    for q in (ar, th):
        c0, a0 = q(w)
        for j in (-9, 6):
            c, a = q((w * F32(2.0 ** j)).astype(F32))
            assert np.array_equal(c, c0) and F32(a) == F32(a0 * F32(2.0 ** j))
        c, a = q(-w)
        assert np.array_equal(c, -c0) and a == a0
        assert set(np.unique(c0)) <= {-1, 0, 1}


def pin_zero_tensor(ar, th):
    z = np.zeros((4, 8), F32)
    for q in (ar, th):
        c, a = q(z)
        assert a == 0 and not c.any()


def pin_worked_example(ar, th):
    """By hand, with dyadic weights so every step is exact:
    W = [[0.25, -0.375, 1, -2], [0, 0.75, -1.125, 2.5]]; sum |W| = 8 over 8
    elements, mean = 1, so alpha = delta = fp32(0.7) = 0.699999988079071.
    [STE] W / alpha = 0.357, -0.536, 1.43, -2.86, 0, 1.07, -1.61, 3.57 round to
    0, -1, 1, -3, 0, 1, -2, 4 and clip to 0, -1, 1, -1, 0, 1, -1, 1; scale 0.7.
    [TWO] kept (|w| > 0.69999999): 1, 2, 0.75, 1.125, 2.5; codes 0, 0, 1, -1,
    0, 1, -1, 1; scale (1 + 2 + 0.75 + 1.125 + 2.5) / 8 = 7.375 / 8 = 0.921875."""
    w = np.array([[0.25, -0.375, 1.0, -2.0], [0.0, 0.75, -1.125, 2.5]], F32)
    c, a = ar(w)
    assert a == F32(0.7)
    assert c.tolist() == [[0, -1, 1, -1], [0, 1, -1, 1]]
    c, a = th(w)
    assert c.tolist() == [[0, 0, 1, -1], [0, 1, -1, 1]]
    assert a == F32(0.921875)


PINS = [pin_bruteforce_small, pin_closed_forms, pin_ties, pin_invariances, pin_zero_tensor, pin_worked_example]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_variant_pin(pin):
    pin(oracle.alpha_round_quantize, oracle.threshold_quantize)


# ---------------------------------------------------------------- planted mistakes
def _m_ar_half_up(w, factor=oracle.DEFAULT_FACTOR):
    w = np.asarray(w, F32)
    alpha = oracle.scaled_mean(w, factor)
    if alpha == 0:
        return np.zeros(w.shape, np.int8), alpha
    q = np.sign(w) * np.floor(np.abs(w / alpha) + F32(0.5))
    return np.clip(q, -1, 1).astype(np.int8), alpha


def _m_ar_gamma_scale(w, factor=oracle.DEFAULT_FACTOR):
    c, _ = oracle.alpha_round_quantize(w, factor)
    return c, oracle.absmean_gamma(w)                  # rescale by mean|W| instead of alpha


def _m_th_mean_over_kept(w, factor=oracle.DEFAULT_FACTOR):
    c, _ = oracle.threshold_quantize(w, factor)
    w = np.asarray(w, F32)
    kept = np.abs(w)[c != 0].astype(np.float64)
    return c, F32(kept.mean()) if kept.size else F32(0)


def _m_th_ge(w, factor=oracle.DEFAULT_FACTOR):
    w = np.asarray(w, F32)
    delta = oracle.scaled_mean(w, factor)
    keep = np.abs(w) >= delta
    c = (np.sign(w) * keep).astype(np.int8)
    s = oracle.exact_abs_sum(np.where(keep, w, F32(0))) / w.size
    return c, oracle.round_ratio_to_f32(s.numerator, s.denominator)


def _m_th_signed_mask(w, factor=oracle.DEFAULT_FACTOR):
    w = np.asarray(w, F32)
    delta = oracle.scaled_mean(w, factor)
    keep = w > delta                                   # drops every negative weight
    c = (np.sign(w) * keep).astype(np.int8)
    s = oracle.exact_abs_sum(np.where(keep, w, F32(0))) / w.size
    return c, oracle.round_ratio_to_f32(s.numerator, s.denominator)


def _m_th_alpha_fp32_sum(w, factor=oracle.DEFAULT_FACTOR):
    c, _ = oracle.threshold_quantize(w, factor)
    w = np.asarray(w, F32)
    return c, F32(np.sum(np.abs(w) * (c != 0), dtype=F32) / F32(w.size))


MUTANTS = {
    "alpha_round_half_up": (_m_ar_half_up, oracle.threshold_quantize),
    "alpha_round_rescale_by_mean": (_m_ar_gamma_scale, oracle.threshold_quantize),
    "threshold_mean_over_kept": (oracle.alpha_round_quantize, _m_th_mean_over_kept),
    "threshold_ge": (oracle.alpha_round_quantize, _m_th_ge),
    "threshold_signed_mask": (oracle.alpha_round_quantize, _m_th_signed_mask),
    "threshold_fp32_sum": (oracle.alpha_round_quantize, _m_th_alpha_fp32_sum),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_variant_mutant_is_caught(name):
    ar, th = MUTANTS[name]
    failed = []
    for pin in PINS:
        try:
            pin(ar, th)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"planted mistake {name} passed every pin"


# ---------------------------------------------------------------- generated inputs
def test_variants_match_rationals_on_generated_tensors():
    """Both rules against the rational references on generated tiny tensors over
    every finite fp32 value (subnormals, the largest normals, signed zeros).
    |w| <= N K mean|W|, so w / alpha stays finite."""
    from hypothesis import given, settings
    from hypothesis import strategies as st

    finite32 = st.floats(width=32, allow_nan=False, allow_infinity=False)
    values = st.one_of(finite32, st.floats(min_value=-1.0, max_value=1.0, width=32))

    @settings(max_examples=300, deadline=None)
    @given(st.integers(1, 3), st.sampled_from([4, 8]), st.data())
    def check(n, k, data):
        w = np.array(data.draw(st.lists(values, min_size=n * k, max_size=n * k)), F32).reshape(n, k)
        c, a = oracle.alpha_round_quantize(w)
        rc, ra = _ref_alpha_round(w)
        assert np.array_equal(c, rc) and F32(a).view(np.uint32) == F32(ra).view(np.uint32)
        c, a = oracle.threshold_quantize(w)
        rc, ra = _ref_threshold(w)
        assert np.array_equal(c, rc) and F32(a).view(np.uint32) == F32(ra).view(np.uint32)

    check()
