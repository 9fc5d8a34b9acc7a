"""Property-based pins of the oracle: generated tiny inputs over every finite
fp32 value (subnormals, the largest normals, signed zeros) against an
evaluation of the definitions in exact rationals that shares nothing with
the oracle (the helpers of tests/pins.py: fp32 rounding by neighbour search,
round-half-even on rationals). Half of the generated tokens hold near-ties of
the activation rounding. Exact ties of the weight rounding need a fixed-point
construction and are pinned in tests/pins.py instead.

Definitions (the oracle's header cites the passages): gamma = mean|W| exact,
rounded once; d = fp32(gamma + 1e-5f); code = clip(rint(fp32(w / d)), -1, 1);
s = fp32(127 / max(max|x|, 1e-5f)); x_q = clip(rint(fp32(x s)), -128, 127);
acc = sum code x_q; y = fp32(fp32(acc gamma) / s).
"""

from __future__ import annotations

from fractions import Fraction

import numpy as np
from hypothesis import HealthCheck, given, settings
from hypothesis import strategies as st

import oracle
from pins import frac_f32, nearest_f32, rint_half_even

F32 = np.float32
EPS = F32(1e-5)

finite32 = st.floats(width=32, allow_nan=False, allow_infinity=False)
# weights and activations of a plausible scale, mixed with arbitrary finite values
scaled32 = st.one_of(finite32, st.floats(min_value=-4.0, max_value=4.0, width=32))


def _sign(v: np.float32) -> int:
    return 1 if v > 0 else (-1 if v < 0 else 0)


def reference(w: np.ndarray, x: np.ndarray):
    """Every output of the forward, evaluated from the definitions in rationals."""
    n, k = w.shape
    total = sum(abs(frac_f32(v)) for v in w.ravel())
    gamma = nearest_f32(total / (n * k))
    d = nearest_f32(frac_f32(gamma) + frac_f32(EPS))
    codes = np.zeros(w.shape, np.int8)
    for idx, v in np.ndenumerate(w):
        q = nearest_f32(frac_f32(v) / frac_f32(d))
        codes[idx] = _sign(q) if not np.isfinite(q) else max(-1, min(1, rint_half_even(frac_f32(q))))
    m = x.shape[0]
    xq = np.zeros(x.shape, np.int8)
    s = np.zeros(m, np.float32)
    for i in range(m):
        a = max(max(abs(frac_f32(v)) for v in x[i]), frac_f32(EPS))
        s[i] = nearest_f32(Fraction(127) / a)
        for j in range(k):
            p = nearest_f32(frac_f32(x[i, j]) * frac_f32(s[i]))
            xq[i, j] = max(-128, min(127, rint_half_even(frac_f32(p))))
    acc = codes.astype(np.int64) @ xq.astype(np.int64).T          # [N][M]
    y = np.zeros((m, n), np.float32)
    for i in range(m):
        for j in range(n):
            t = nearest_f32(Fraction(int(acc[j, i])) * frac_f32(gamma))
            y[i, j] = t if not np.isfinite(t) else nearest_f32(frac_f32(t) / frac_f32(s[i]))
    packed = np.zeros((n, k // 4), np.uint8)
    for r in range(n):
        for b in range(k // 4):
            packed[r, b] = sum((int(codes[r, 4 * b + i]) + 1) << (2 * i) for i in range(4))
    return {"gamma": gamma, "codes": codes, "packed": packed, "xq": xq, "scale": s, "acc": acc.T, "y": y}


def bits(a):
    return np.asarray(a, np.float32).view(np.uint32)


@st.composite
def near_tie_token(draw, k):
    """A token whose products x s sit within an ulp of j + 1/2: x_j = fp32((j + 1/2) / s)
    next to its absmax a (so that s = fp32(127 / a)); these separate round-half-even
    from half-up and 127 / a from a / 127."""
    a = draw(st.floats(min_value=0.0009765625, max_value=1024.0, width=32))
    sc = nearest_f32(Fraction(127) / frac_f32(a))
    js = draw(st.lists(st.integers(-126, 125), min_size=k - 1, max_size=k - 1))
    row = [F32(float(a) if draw(st.booleans()) else -float(a))]
    row += [nearest_f32((Fraction(j) + Fraction(1, 2)) / frac_f32(sc)) for j in js]
    return row


@st.composite
def problems(draw):
    n = draw(st.integers(1, 3))
    k = draw(st.sampled_from([4, 8]))
    m = draw(st.integers(1, 2))
    w = np.array(draw(st.lists(scaled32, min_size=n * k, max_size=n * k)), np.float32).reshape(n, k)
    rows = [draw(st.one_of(st.lists(scaled32, min_size=k, max_size=k), near_tie_token(k))) for _ in range(m)]
    x = np.array(rows, np.float32).reshape(m, k)
    return w, x


@settings(max_examples=300, deadline=None, suppress_health_check=[HealthCheck.too_slow])
@given(problems())
def test_oracle_matches_the_definitions_on_generated_inputs(prob):
    w, x = prob
    with np.errstate(over="ignore"):        # extreme inputs may overflow y to +-inf
        got = oracle.bitlinear_forward(x, w)
    want = reference(w, x)
    assert bits(got["gamma"]) == bits(want["gamma"])
    assert np.array_equal(got["codes"], want["codes"])
    assert np.array_equal(got["packed"], want["packed"])
    assert np.array_equal(got["xq"], want["xq"])
    assert np.array_equal(bits(got["scale"]), bits(want["scale"]))
    assert np.array_equal(np.asarray(got["acc"], np.int64), want["acc"])
    assert np.array_equal(bits(got["y"]), bits(want["y"]))


@settings(max_examples=200, deadline=None)
@given(st.lists(finite32, min_size=1, max_size=16))
def test_gamma_is_the_exact_mean_rounded_once(vals):
    w = np.array(vals, np.float32).reshape(1, -1)
    exact = sum(abs(frac_f32(v)) for v in w.ravel()) / w.size
    assert bits(oracle.absmean_gamma(w)) == bits(nearest_f32(exact))


@settings(max_examples=200, deadline=None)
@given(st.lists(finite32, min_size=4, max_size=16).filter(lambda v: len(v) % 4 == 0))
def test_codes_survive_packing(vals):
    w = np.array(vals, np.float32).reshape(1, -1)
    c = oracle.ternary_codes(w, oracle.absmean_gamma(w))
    p = oracle.pack_codes(c)
    fields = np.stack([(p >> (2 * i)) & 3 for i in range(4)])
    assert p.shape == (1, w.size // 4) and not np.any(fields == 3)
    assert np.array_equal(oracle.unpack_codes(p), c)
