"""Pins of the per-group (64) oracle, and planted mistakes that must fail them.

The per-group rule ([HPFT] body: per-group quantisation, group size 64) is
checked against facts fixed outside the oracle:

* brute force in exact rationals on tiny inputs (scales, codes, partial sums
  and y, with the fp32 rounding found by neighbour search);
* structure: changing one group moves only that group's scale and codes; a
  power of two on one group scales only its gamma (codes unchanged, eps = 0);
  when every group holds the same 64 values the rule is the per-tensor rule;
* the rescale is the exact sum rounded once: ties between two fp32 values go
  to the even one, and sums that cancel keep their exact value;
* the zero fraction of Gaussian weights, derived here for groups of 64: a
  weight is part of its own group's mean, so it is zero when |w| <= (|w| + S)
  / 128 with S the sum of the other 63 |w|, which moves the fraction from
  0.3101 (per tensor) to about 0.3077.
"""

from __future__ import annotations

import math
import types
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import grouped as og
from pins import frac_f32, nearest_f32, rint_half_even

F32 = np.float32


# ------------------------------------------------------------------ namespace of the grouped oracle (mutable copies)
def _ns(**overrides):
    ns = types.SimpleNamespace(group_gammas=og.group_gammas, group_codes=og.group_codes,
                               group_accumulators=og.group_accumulators, grouped_rescale=og.grouped_rescale,
                               quant_act=oracle.quant_act)
    for k, v in overrides.items():
        setattr(ns, k, v)

    def forward(x, w):
        g = ns.group_gammas(w)
        c = ns.group_codes(w, g)
        xq, s = ns.quant_act(x)
        acc = ns.group_accumulators(xq, c)
        return {"gammas": g, "codes": c, "xq": xq, "scale": s, "acc": acc, "y": ns.grouped_rescale(acc, g, s)}
    ns.forward = forward
    return ns


def _bits(a):
    return np.asarray(a, dtype=np.float32).view(np.uint32)


# ------------------------------------------------------------------ pins
def pin_bruteforce(o):
    rng = np.random.default_rng(41)
    w = (rng.standard_normal((3, 128)) * 0.02).astype(np.float32)
    w[1, 64:] *= F32(1e3)                                   # groups of very different scale
    w[2, :8] = 0.0
    x = rng.standard_normal((2, 128)).astype(np.float32)
    r = o.forward(x, w)
    for n in range(3):
        for g in range(2):
            vals = w[n, 64 * g:64 * g + 64]
            gam = nearest_f32(sum(Fraction(float(v)) for v in np.abs(vals)) / 64)
            assert r["gammas"][n, g].view(np.uint32) == gam.view(np.uint32), (n, g)
            d = nearest_f32(frac_f32(gam) + frac_f32(F32(1e-5)))
            for k, v in enumerate(vals):
                q = nearest_f32(frac_f32(v) / frac_f32(d))
                assert r["codes"][n, 64 * g + k] == max(-1, min(1, rint_half_even(Fraction(float(q))))), (n, g, k)
    for m in range(2):
        a = max(max(abs(Fraction(float(v))) for v in x[m]), Fraction(float(F32(1e-5))))
        s = nearest_f32(Fraction(127) / a)
        assert r["scale"][m].view(np.uint32) == s.view(np.uint32)
        xq = [max(-128, min(127, rint_half_even(Fraction(float(nearest_f32(frac_f32(v) * frac_f32(s))))))) for v in x[m]]
        for n in range(3):
            total = Fraction(0)
            for g in range(2):
                acc = sum(int(r["codes"][n, k]) * xq[k] for k in range(64 * g, 64 * g + 64))
                assert r["acc"][m, n, g] == acc
                total += frac_f32(r["gammas"][n, g]) * acc
            y = nearest_f32(total / frac_f32(s))
            assert r["y"][m, n].view(np.uint32) == y.view(np.uint32), (m, n)


def pin_group_independence(o):
    rng = np.random.default_rng(42)
    w = (rng.standard_normal((4, 256)) * 0.02).astype(np.float32)
    g0 = o.group_gammas(w)
    c0 = o.group_codes(w, g0)
    w2 = w.copy()
    w2[2, 128:192] = (rng.standard_normal(64) * 0.5).astype(np.float32)   # row 2, group 2 only
    g1 = o.group_gammas(w2)
    c1 = o.group_codes(w2, g1)
    changed = g1 != g0
    assert changed[2, 2] and changed.sum() == 1
    mask = np.ones_like(c0, dtype=bool)
    mask[2, 128:192] = False
    np.testing.assert_array_equal(c1[mask], c0[mask])


def pin_group_scale_invariance(o):
    rng = np.random.default_rng(43)
    w = (rng.standard_normal((3, 192)) * 0.02).astype(np.float32)
    g0 = o.group_gammas(w)
    c0 = o.group_codes(w, g0, eps=F32(0.0))
    for j in (-9, 4):
        w2 = w.copy()
        w2[1, 64:128] = np.ldexp(w2[1, 64:128], j).astype(np.float32)
        g1 = o.group_gammas(w2)
        assert g1[1, 1] == F32(np.ldexp(g0[1, 1], j))
        np.testing.assert_array_equal(np.delete(g1.ravel(), 4), np.delete(g0.ravel(), 4))
        np.testing.assert_array_equal(o.group_codes(w2, g1, eps=F32(0.0)), c0)


def pin_identical_groups_are_per_tensor(o):
    rng = np.random.default_rng(44)
    pattern = (rng.standard_normal(64) * 0.02).astype(np.float32)
    w = np.tile(pattern, (5, 4))                              # every group holds the same 64 values
    gam = o.group_gammas(w)
    g = oracle.absmean_gamma(w)
    assert (gam == g).all()
    np.testing.assert_array_equal(o.group_codes(w, gam), oracle.ternary_codes(w, g))
    x = rng.standard_normal((3, 256)).astype(np.float32)
    r = o.forward(x, w)
    acc = oracle.ternary_int8_matmul(r["xq"], r["codes"])
    for m in range(3):
        for n in range(5):
            want = nearest_f32(frac_f32(g) * int(acc[m, n]) / frac_f32(r["scale"][m]))
            assert r["y"][m, n].view(np.uint32) == want.view(np.uint32)


def pin_rescale_exact(o):
    # one rounding of the exact sum: ties to even, cancellation kept exactly
    one = F32(1.0)
    ulp = F32(np.ldexp(1.0, -23))
    # sum = 1 + 2^-24 (halfway between 1 and 1 + 2^-23): even -> 1
    acc = np.array([[[1, 1]]], dtype=np.int64)
    gam = np.array([[one, F32(np.ldexp(1.0, -24))]], dtype=np.float32)
    assert o.grouped_rescale(acc, gam, np.array([1.0], np.float32))[0, 0] == one
    # sum = 1 + 3 * 2^-24: halfway between 1 + 2^-23 and 1 + 2^-22 -> 1 + 2^-22
    acc = np.array([[[1, 3]]], dtype=np.int64)
    assert o.grouped_rescale(acc, gam, np.array([1.0], np.float32))[0, 0] == F32(one + 2 * ulp)
    # cancellation: 2^30 - 2^30 + 3 * 2^-20 keeps the small term exactly
    acc = np.array([[[1, -1, 3]]], dtype=np.int64)
    gam = np.array([[F32(2.0 ** 30), F32(2.0 ** 30), F32(2.0 ** -20)]], dtype=np.float32)
    assert o.grouped_rescale(acc, gam, np.array([1.0], np.float32))[0, 0] == F32(3 * 2.0 ** -20)
    # random cases against rationals, division by s included
    rng = np.random.default_rng(45)
    acc = rng.integers(-8128, 8129, size=(3, 4, 6))
    gam = (rng.uniform(0.001, 0.05, size=(4, 6))).astype(np.float32)
    s = rng.uniform(1.0, 200.0, size=3).astype(np.float32)
    y = o.grouped_rescale(acc, gam, s)
    for m in range(3):
        for n in range(4):
            t = sum(frac_f32(gam[n, g]) * int(acc[m, n, g]) for g in range(6))
            assert y[m, n].view(np.uint32) == nearest_f32(t / frac_f32(s[m])).view(np.uint32)


def _expected_zero_fraction(group=64, eps_over_sigma=1e-5 / 0.02):
    """E over S of P(|Z| <= (|Z| + S) / (2 group) + eps / 2), |Z| half-normal,
    S the sum of the other group - 1 half-normals (normal by the central limit
    theorem): |Z| (2 group - 1) / (2 group) <= S / (2 group) + eps / 2."""
    from scipy import integrate, special
    mu = math.sqrt(2 / math.pi)
    var = 1 - 2 / math.pi
    mean_s, sd_s = (group - 1) * mu, math.sqrt((group - 1) * var)
    c = (2 * group - 1) / (2 * group)

    def integrand(z):
        s = mean_s + sd_s * z
        t = (s / (2 * group) + eps_over_sigma / 2) / c
        return special.erf(t / math.sqrt(2)) * math.exp(-z * z / 2) / math.sqrt(2 * math.pi)
    return integrate.quad(integrand, -8, 8)[0]


def pin_gaussian_zero_fraction(o):
    want = _expected_zero_fraction()
    assert abs(want - 0.3077) < 0.0005                    # the derivation above, per tensor it is 0.3101
    rng = np.random.default_rng(46)
    w = (rng.standard_normal((512, 4096)) * 0.02).astype(np.float32)   # 2 M weights, sd of the fraction 3e-4
    gam = o.group_gammas(w)
    f = float((o.group_codes(w, gam) == 0).mean())
    assert abs(f - want) < 0.0015, (f, want)


def group_tie_weights():
    """Weights [2][128] whose second group of row 0 holds +-t with t == d/2
    exactly, d = fp32(gamma_{0,1} + 1e-5); gamma depends on t, so t is
    refined to a fixed point t_{i+1} = d(t_i) / 2 (found by rationals here)."""
    rng = np.random.default_rng(47)
    w = (rng.standard_normal((2, 128)) * 0.02).astype(np.float32)
    t = F32(0.008)
    for _ in range(60):
        w[0, 126], w[0, 127] = t, -t
        grp = w[0, 64:128]
        gam = nearest_f32(sum(Fraction(float(v)) for v in np.abs(grp)) / 64)
        d = nearest_f32(frac_f32(gam) + frac_f32(F32(1e-5)))
        nt = F32(np.ldexp(d, -1))
        if nt == t:
            return w, gam, t
        t = nt
    raise AssertionError("tie construction did not converge")


def pin_group_code_tie(o):
    w, gam, t = group_tie_weights()
    g = o.group_gammas(w)
    assert g[0, 1] == gam
    c = o.group_codes(w, g)
    # t / d is exactly 0.5: half to even gives 0 (half up would give +1 / -1)
    assert c[0, 126] == 0 and c[0, 127] == 0


PINS = [pin_bruteforce, pin_group_code_tie, pin_group_independence, pin_group_scale_invariance, pin_identical_groups_are_per_tensor,
        pin_rescale_exact, pin_gaussian_zero_fraction]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_grouped_oracle_pins(pin):
    pin(_ns())


# ------------------------------------------------------------------ planted mistakes
def m_gammas_per_tensor(w, group=og.GROUP):
    w = np.asarray(w, np.float32)
    return np.full((w.shape[0], w.shape[1] // group), oracle.absmean_gamma(w), np.float32)


def m_gammas_along_rows(w, group=og.GROUP):
    # groups of 64 rows within a column instead of 64 k within a row (as many as fit)
    w = np.asarray(w, np.float32)
    n, k = w.shape
    out = np.empty((n, k // group), np.float32)
    for c in range(k // group):
        col = w[:, c * group:(c + 1) * group]
        out[:, c] = oracle.absmean_gamma(col.T.ravel()[:min(n, group) * group].reshape(-1, group))
    return out


def m_gammas_group32(w, group=og.GROUP):
    w = np.asarray(w, np.float32)
    g32 = og.group_gammas(w, 32)
    return g32[:, ::2].copy()


def m_gammas_fp32_sum(w, group=og.GROUP):
    w = np.asarray(w, np.float32)
    n, k = w.shape
    return np.abs(w).reshape(n, k // group, group).mean(axis=2, dtype=np.float32)


def m_codes_half_up(w, gammas, eps=og.EPS_GAMMA, group=og.GROUP):
    w = np.asarray(w, np.float32)
    d = (np.asarray(gammas, np.float32) + F32(eps)).astype(np.float32)
    dd = np.repeat(d, group, axis=1)
    return np.clip(np.floor(w / dd + F32(0.5)), -1, 1).astype(np.int8)


def m_rescale_fp32_sequential(acc, gammas, s):
    acc = np.asarray(acc, np.int64)
    m, n, g = acc.shape
    t = np.zeros((m, n), np.float32)
    for j in range(g):
        t = (t + acc[:, :, j].astype(np.float32) * np.asarray(gammas, np.float32)[None, :, j]).astype(np.float32)
    return (t / np.asarray(s, np.float32)[:, None]).astype(np.float32)


def m_rescale_eps_in_gamma(acc, gammas, s):
    return og.grouped_rescale(acc, (np.asarray(gammas, np.float32) + F32(1e-5)).astype(np.float32), s)


def m_acc_drops_last_k(xq, codes, group=og.GROUP):
    codes = np.asarray(codes).copy()
    codes[:, -1] = 0
    return og.group_accumulators(xq, codes, group)


MUTANTS = {
    "gammas_per_tensor": {"group_gammas": m_gammas_per_tensor},
    "gammas_along_rows": {"group_gammas": m_gammas_along_rows},
    "gammas_group32": {"group_gammas": m_gammas_group32},
    "gammas_fp32_sum": {"group_gammas": m_gammas_fp32_sum},
    "codes_half_up": {"group_codes": m_codes_half_up},
    "rescale_fp32_sequential": {"grouped_rescale": m_rescale_fp32_sequential},
    "rescale_eps_in_gamma": {"grouped_rescale": m_rescale_eps_in_gamma},
    "acc_drops_last_k": {"group_accumulators": m_acc_drops_last_k},
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(name):
    ns = _ns(**MUTANTS[name])
    failed = []
    for pin in PINS:
        try:
            pin(ns)
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
