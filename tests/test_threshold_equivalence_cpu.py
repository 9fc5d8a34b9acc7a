"""The comparison the packing kernels use in place of a division.

The kernels take code = 0 when |w| <= d/2, else the sign of w, where the
pages' rule is clip(rint(fp32(w / d)), -1, 1) with round-half-even. The two
agree for every finite fp32 w and every normal fp32 d (d/2 is then exact):
if |w| <= d/2 the quotient rounds to at most 0.5 in magnitude, which rint
takes to 0; if |w| > d/2 then |w| is at least the fp32 successor of d/2, so
the exact quotient exceeds 0.5 by more than half an ulp of 0.5 (d/2 has a
significand below 2), the fp32 quotient is at least the successor of 0.5, and
rint gives at least 1 in magnitude, which the clip takes to 1.

This test checks that claim with IEEE fp32 arithmetic (numpy) at the values
where it could fail: w at, just below and just above d/2 and 3d/2,
subnormal and huge w, and d across the normal range, including the
alpha-round rule's d = fp32(0.7 * gamma) down to 2^-125 (below which the
kernel divides instead).
"""

import numpy as np
import pytest

F32 = np.float32


def rule_by_division(w, d):
    with np.errstate(over="ignore", under="ignore"):
        q = np.rint(w / d)
    return np.clip(q, -1, 1).astype(np.int8)


def rule_by_comparison(w, d):
    h = F32(d) * F32(0.5)
    return np.where(np.abs(w) <= h, 0, np.sign(w)).astype(np.int8)


def boundary_weights(d):
    """Finite fp32 weights at and next to d/2, 3d/2 and d, plus extremes."""
    d = F32(d)
    with np.errstate(over="ignore"):
        h = F32(d * F32(0.5))
        pts = [h, F32(d * F32(1.5)), d, F32(0.0), F32(-0.0)]
        out = []
        for p in pts:
            for v in (p, np.nextafter(p, F32(np.inf)), np.nextafter(p, F32(0)),
                      np.nextafter(np.nextafter(p, F32(np.inf)), F32(np.inf))):
                out += [v, -v]
    out += [F32(1e-45), F32(-1e-45), F32(1.1754942e-38), F32(3.4028235e38), F32(-3.4028235e38)]
    w = np.array(out, dtype=F32)
    return w[np.isfinite(w)]


@pytest.mark.parametrize("seed", range(4))
def test_comparison_equals_division_at_the_boundaries(seed):
    rng = np.random.default_rng(seed)
    exps = rng.integers(-125, 127, size=400)
    mants = rng.uniform(1.0, 2.0, size=400)
    ds = (mants * 2.0 ** exps).astype(F32)
    ds = np.concatenate([ds, np.array([2.0 ** -125, 2.0 ** -126 * 1.5, 1e-5, 0.02, 1.0, 3.0e38], F32)])
    for d in ds:
        if not np.isfinite(d) or d < np.finfo(F32).tiny * 2:
            continue                        # d/2 must be a normal number, so exact
        w = boundary_weights(d)
        assert np.array_equal(rule_by_comparison(w, d), rule_by_division(w, d)), d


def test_comparison_equals_division_on_random_weights():
    rng = np.random.default_rng(7)
    w = (rng.standard_normal(1 << 20) * 0.02).astype(F32)
    for gamma in (F32(0.016), F32(0.01595), F32(1e-20), F32(7e20)):
        d = F32(gamma + F32(1e-5))               # the absmean rule's divisor
        assert np.array_equal(rule_by_comparison(w * (gamma / F32(0.016)), d),
                              rule_by_division(w * (gamma / F32(0.016)), d))
        alpha = F32(F32(0.7) * gamma)              # the alpha-round rule's divisor
        assert np.array_equal(rule_by_comparison(w, alpha), rule_by_division(w, alpha))


def test_half_tie_rounds_to_zero_not_away():
    # the tie w = d/2 is where half-up rounding would give 1: both rules give 0
    d = F32(0.0200100001)
    w = np.array([d * F32(0.5), -d * F32(0.5)], F32)
    assert rule_by_division(w, d).tolist() == [0, 0]
    assert rule_by_comparison(w, d).tolist() == [0, 0]
