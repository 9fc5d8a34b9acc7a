"""Pins: checks that tie the oracle to facts fixed outside itself.

Each ``pin_*`` function takes an oracle namespace ``o`` (the real
``oracle`` package, or a copy with one function replaced by a planted
mistake) and raises AssertionError when the oracle disagrees with

* a hand-derived worked example (``tests/golden/worked_example.json``),
* brute force with exact rationals on tiny inputs,
* closed forms (the Gaussian / Student-t zero fractions implied by absmean),
* invariants (scale, permutation, round trip), or
* tie cases that separate round-half-to-even from round-half-up.

The helpers here are written independently of the oracle: the fp32 rounding
of a rational is found by a neighbour search, not by the oracle's routine.
"""

from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np

F32 = np.float32
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ------------------------------------------------------------------ helpers
def nearest_f32(v: Fraction) -> np.float32:
    """fp32 nearest to the rational v (ties to even), by neighbour search."""
    v = Fraction(v)
    # IEEE overflow: at or above the midpoint between the largest finite fp32
    # (2^128 - 2^104) and 2^128, round-to-nearest gives infinity
    if abs(v) >= Fraction(2 ** 128 - 2 ** 103):
        return F32(np.inf) if v > 0 else F32(-np.inf)
    c = F32(min(float(v), 3.4028234663852886e38)) if v > 0 else F32(max(float(v), -3.4028234663852886e38))
    best = None
    for cand in (np.nextafter(c, F32(-np.inf)), c, np.nextafter(c, F32(np.inf))):
        cand = F32(cand)
        if not np.isfinite(cand):
            continue
        dist = abs(Fraction(float(cand)) - v)
        if best is None or dist < best[0]:
            best = (dist, cand)
        elif dist == best[0]:
            # tie: even significand (lowest bit of the encoding clear)
            if int(cand.view(np.uint32)) & 1 == 0:
                best = (dist, cand)
    return F32(best[1])


def frac_f32(x) -> Fraction:
    return Fraction(float(F32(x)))


def rint_half_even(v: Fraction) -> int:
    # Python's round() on a Fraction rounds half to even
    return int(round(Fraction(v)))


def load_golden(name="worked_example.json"):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ gamma
def pin_round_ratio_neighbour_search(o):
    rng = np.random.default_rng(7)
    cases = [(1, 3), (2, 3), (1, 10), (7, 1), (10 ** 40, 3), (1, 2 ** 150), (3, 2 ** 150), (1, 2 ** 151),
             (2 ** 24 + 1, 2), (2 ** 25 + 3, 4), (123456789, 1000)]
    for _ in range(300):
        num = int(rng.integers(1, 2 ** 62))
        den = int(rng.integers(1, 2 ** 62))
        sh = int(rng.integers(-160, 100))
        if sh >= 0:
            num <<= sh
        else:
            den <<= -sh
        cases.append((num, den))
    for num, den in cases:
        got = o.round_ratio_to_f32(num, den)
        want = nearest_f32(Fraction(num, den))
        assert got.view(np.uint32) == want.view(np.uint32), (num, den, got, want)


def pin_gamma_bruteforce_small(o):
    rng = np.random.default_rng(11)
    arrays = [
        rng.standard_normal((3, 8)).astype(np.float32) * F32(0.02),
        rng.standard_normal((5, 4)).astype(np.float32) * F32(1e3),
        np.array([[2.0 ** 24, 1.0, 1.0, 1.0]], dtype=np.float32),                 # fp32 naive sum would drop the 1s
        np.array([[1e-45, 3e-45, 0.0, -1e-45]], dtype=np.float32),                 # subnormals
        np.array([[3.0e38, -3.0e38, 3.0e38, 1.0]], dtype=np.float32),             # sum overflows fp32
        rng.standard_normal((7, 12)).astype(np.float32) * np.logspace(-30, 30, 12, dtype=np.float32),
    ]
    for w in arrays:
        exact = sum(Fraction(float(v)) for v in np.abs(w).ravel())
        want = nearest_f32(exact / w.size)
        got = o.absmean_gamma(w)
        assert got.view(np.uint32) == want.view(np.uint32), (w, got, want)


def pin_gamma_fsum(o):
    rng = np.random.default_rng(12)
    w = (rng.standard_normal((512, 768)) * 0.02).astype(np.float32)
    s = math.fsum(np.abs(w).astype(np.float64).ravel())
    want = F32(s / w.size)
    assert o.absmean_gamma(w) == want


def pin_gamma_closed_forms(o):
    # constant tensor: the mean is the value
    assert o.absmean_gamma(np.full((4, 8), -0.375, np.float32)) == F32(0.375)
    # 1..n: mean (n+1)/2
    n = 4096
    w = np.arange(1, n + 1, dtype=np.float32).reshape(64, 64)
    assert o.absmean_gamma(w) == F32((n + 1) / 2)
    # ties to even: mean 1 + 2^-24 lies halfway between 1 and 1 + 2^-23 -> 1
    one = F32(1.0)
    up1 = np.nextafter(one, F32(2))
    up2 = np.nextafter(up1, F32(2))
    assert o.absmean_gamma(np.array([[one, up1]], np.float32)) == one
    # mean halfway between 1+2^-23 (odd) and 1+2^-22 (even) -> the even one
    assert o.absmean_gamma(np.array([[up1, up2]], np.float32)) == up2
    # subnormal ties
    tiny = F32(np.ldexp(1.0, -149))
    assert o.absmean_gamma(np.array([[tiny, 0.0]], np.float32)) == F32(0.0)
    assert o.absmean_gamma(np.array([[3 * tiny, 0.0]], np.float32)) == F32(np.ldexp(1.0, -148))


def pin_gamma_invariances(o):
    rng = np.random.default_rng(13)
    w = (rng.standard_normal((64, 96)) * 0.02).astype(np.float32)
    g = o.absmean_gamma(w)
    assert o.absmean_gamma(-w) == g
    perm = rng.permutation(w.size)
    assert o.absmean_gamma(w.ravel()[perm].reshape(96, 64)) == g
    for j in (-7, 3, 20):
        assert o.absmean_gamma(np.ldexp(w, j).astype(np.float32)) == F32(np.ldexp(g, j))


# ------------------------------------------------------------------ codes
def pin_codes_bruteforce(o):
    rng = np.random.default_rng(21)
    w = (rng.standard_normal((6, 16)) * 0.02).astype(np.float32)
    g = o.absmean_gamma(w)
    d = F32(F32(g) + F32(1e-5))
    codes = o.ternary_codes(w, g)
    for (i, j), v in np.ndenumerate(w):
        q = nearest_f32(frac_f32(v) / frac_f32(d))        # fp32 division, RN
        c = max(-1, min(1, rint_half_even(Fraction(float(q)))))
        assert codes[i, j] == c, (v, d, codes[i, j], c)


def _tie_tensor():
    """A tensor holding +-t with t == d/2 exactly, where d = fp32(gamma + 1e-5).

    gamma depends on t, so t is refined to a fixed point: t_{i+1} = d(t_i)/2.
    """
    rng = np.random.default_rng(22)
    base = (rng.standard_normal(1022) * 0.02).astype(np.float32)
    t = F32(0.008)
    for _ in range(60):
        w = np.concatenate([base, np.array([t, -t], np.float32)]).reshape(2, 512)
        exact = sum(Fraction(float(v)) for v in np.abs(w).ravel())
        g = nearest_f32(exact / w.size)
        d = nearest_f32(frac_f32(g) + frac_f32(F32(1e-5)))
        nt = F32(np.ldexp(d, -1))
        if nt == t:
            return w, g, t
        t = nt
    raise AssertionError("tie construction did not converge")


def pin_codes_half_tie(o):
    w, g, t = _tie_tensor()
    assert o.absmean_gamma(w) == g
    c = o.ternary_codes(w, g).ravel()
    # t/d is exactly 0.5: half-to-even gives 0 (half-up would give +1 / -1)
    assert c[-2] == 0 and c[-1] == 0, c[-2:]
    # the next fp32 above t quantises to +1
    t_up = np.nextafter(t, F32(1))
    assert o.ternary_codes(np.array([[t_up, -t_up, 0, 0]], np.float32), g).tolist() == [[1, -1, 0, 0]]


def pin_codes_scale_invariance(o):
    rng = np.random.default_rng(23)
    w = (rng.standard_normal((64, 64)) * 0.02).astype(np.float32)
    g = o.absmean_gamma(w)
    c0 = o.ternary_codes(w, g, eps=F32(0.0))
    for j in (-5, 4, 30):
        ws = np.ldexp(w, j).astype(np.float32)
        cj = o.ternary_codes(ws, o.absmean_gamma(ws), eps=F32(0.0))
        assert np.array_equal(c0, cj), j
    # with the 1e-5 epsilon the codes move only where |W| sits near d/2
    c1 = o.ternary_codes(w, g)
    ws = np.ldexp(w, 3).astype(np.float32)
    c2 = o.ternary_codes(ws, o.absmean_gamma(ws))
    assert np.mean(c1 != c2) <= 1e-3


def pin_codes_values(o):
    rng = np.random.default_rng(24)
    w = (rng.standard_normal((32, 128)) * 3).astype(np.float32)
    c = o.ternary_codes(w, o.absmean_gamma(w))
    assert c.dtype == np.int8 and set(np.unique(c).tolist()) <= {-1, 0, 1}
    # a code never has the opposite sign of its weight
    assert np.all(c.astype(np.int32) * np.sign(w).astype(np.int32) >= 0)


def pin_gaussian_zero_fraction(o):
    # |W| <= d/2 with d ~ sigma*sqrt(2/pi): P = erf(sqrt(2/pi)/2/sqrt(2)) = 0.310064
    from workloads import gaussian_weights
    w = gaussian_weights(1024, 1024, seed=101).numpy()
    c = o.ternary_codes(w, o.absmean_gamma(w))
    p0 = math.erf(math.sqrt(2 / math.pi) / 2 / math.sqrt(2))
    f0 = float(np.mean(c == 0))
    assert abs(f0 - p0) < 0.003, f0                     # sd at 2^20 samples ~ 4.5e-4
    assert abs(float(np.mean(c == 1)) - (1 - p0) / 2) < 0.003
    assert abs(float(np.mean(c == -1)) - (1 - p0) / 2) < 0.003


def pin_student_t_zero_fraction(o):
    # 0.02 * T_4: E|T_4| = 1, zero fraction = 2F(0.5)-1 with the closed-form t4 CDF
    from workloads import student_t_weights
    w = student_t_weights(1024, 1024, seed=102).numpy()
    c = o.ternary_codes(w, o.absmean_gamma(w))
    t = 0.5
    cdf = 0.5 + t * (t * t + 6) / (2 * (t * t + 4) ** 1.5)
    p0 = 2 * cdf - 1
    assert abs(float(np.mean(c == 0)) - p0) < 0.004, float(np.mean(c == 0))


# ------------------------------------------------------------------ packing
def pin_pack_layout(o):
    c = np.array([[-1, 0, 1, -1, 1, 1, 1, 1], [0, 0, 0, 0, -1, -1, -1, -1]], np.int8)
    p = o.pack_codes(c)
    # field = code + 1, least significant first: [0,1,2,0] -> 0 + 4 + 32 + 0 = 0x24
    assert p.tolist() == [[0x24, 0xAA], [0x55, 0x00]], p
    assert np.array_equal(o.unpack_codes(p), c)


def pin_pack_roundtrip(o):
    rng = np.random.default_rng(31)
    c = rng.integers(-1, 2, size=(17, 64)).astype(np.int8)
    p = o.pack_codes(c)
    assert p.shape == (17, 16) and p.dtype == np.uint8
    assert np.array_equal(o.unpack_codes(p), c)
    fields = np.stack([(p >> (2 * i)) & 3 for i in range(4)])
    assert not np.any(fields == 3)
    # every byte value with no field equal to 3 unpacks and repacks to itself
    ok = [b for b in range(256) if all(((b >> (2 * i)) & 3) != 3 for i in range(4))]
    assert len(ok) == 81
    pb = np.array(ok, np.uint8).reshape(81, 1)
    assert np.array_equal(o.pack_codes(o.unpack_codes(pb)), pb)


# ------------------------------------------------------------------ activations
def pin_act_ties(o):
    x = np.array([[2.5, 3.5, -0.5, 126.5, 127.0, -1.5]], np.float32)
    q, s = o.quant_act(x)
    assert s.tolist() == [1.0]
    assert q.tolist() == [[2, 4, 0, 126, 127, -2]]


def pin_act_bruteforce(o):
    rng = np.random.default_rng(41)
    x = rng.standard_normal((5, 24)).astype(np.float32) * np.array([1, 1e-3, 50, 1e-7, 3], np.float32)[:, None]
    q, s = o.quant_act(x)
    for m in range(x.shape[0]):
        a = max(max(abs(frac_f32(v)) for v in x[m]), frac_f32(F32(1e-5)))
        sm = nearest_f32(Fraction(127) / a)
        assert s[m] == sm, (m, s[m], sm)
        for k in range(x.shape[1]):
            p = nearest_f32(frac_f32(x[m, k]) * frac_f32(sm))
            want = max(-128, min(127, rint_half_even(Fraction(float(p)))))
            assert q[m, k] == want, (m, k, q[m, k], want)


def pin_act_product_emulation(o):
    """x_q = rint(RN32(x*s)) on many near-tie products.

    The product of two fp32 values is exact in fp64 (48 significant bits), so
    converting the fp64 product to fp32 is a single correct rounding: an
    independent vectorised emulation of the fp32 multiply.
    """
    rng = np.random.default_rng(43)
    m, k = 32, 2048
    x = rng.standard_normal((m, k)).astype(np.float32)
    x *= np.exp2(rng.integers(-20, 20, size=(m, 1))).astype(np.float32) * rng.uniform(1, 2, size=(m, 1)).astype(np.float32)
    a = np.max(np.abs(x), axis=1)
    x[:, 0] = -a                       # the absmax sits at an even column the planting keeps
    s = np.array([nearest_f32(Fraction(127) / max(frac_f32(v), frac_f32(F32(1e-5)))) for v in a], np.float32)
    # plant near-ties: x = RN32((j + 1/2) / s) so that x*s sits within an ulp of j + 1/2
    j = rng.integers(-126, 126, size=(m, k // 2))
    x[:, 1::2] = ((j + 0.5) / s[:, None].astype(np.float64)).astype(np.float32)
    q, s_o = o.quant_act(x)
    assert np.array_equal(s_o, s)
    prod = (x.astype(np.float64) * s.astype(np.float64)[:, None]).astype(np.float32)
    want = np.clip(np.rint(prod), -128, 127).astype(np.int8)
    assert np.array_equal(q, want), int(np.sum(q != want))


def pin_act_invariants(o):
    rng = np.random.default_rng(42)
    x = rng.standard_normal((8, 300)).astype(np.float32)
    q, s = o.quant_act(x)
    # the absmax element of each token maps to +-127
    am = np.argmax(np.abs(x), axis=1)
    assert np.all(np.abs(q[np.arange(8), am]) == 127)
    assert np.all(np.abs(q.astype(np.int32)) <= 127)
    # exact invariance of x_q under x -> 2^j x (epsilon floor inactive)
    for j in (-10, 7):
        qj, sj = o.quant_act(np.ldexp(x, j).astype(np.float32))
        assert np.array_equal(q, qj)
        assert np.array_equal(sj, np.ldexp(s, -j).astype(np.float32))
    # an all-zero token: a = 1e-5, every code 0
    qz, sz = o.quant_act(np.zeros((1, 16), np.float32))
    assert np.all(qz == 0) and sz[0] == nearest_f32(Fraction(127) / frac_f32(F32(1e-5)))


def pin_bf16_widening(o):
    bits = np.array([0x3F80, 0xBF80, 0x0000, 0x8000, 0x4049, 0x7F7F, 0x0001], np.uint16)
    f = o.bf16_bits_to_f32(bits)
    assert f[0] == 1.0 and f[1] == -1.0 and f[2] == 0.0 and np.signbit(f[3])
    assert f[4] == F32(3.140625)                          # 0x4049 = 1.5703125 * 2
    assert f[5] == F32(np.ldexp(255 / 128, 127))          # largest finite bf16
    assert f[6] == F32(np.ldexp(1.0, -133))               # smallest bf16 subnormal


# ------------------------------------------------------------------ matmul / rescale
def pin_matmul_bruteforce(o):
    rng = np.random.default_rng(51)
    xq = rng.integers(-127, 128, size=(3, 12)).astype(np.int8)
    c = rng.integers(-1, 2, size=(5, 12)).astype(np.int8)
    acc = o.ternary_int8_matmul(xq, c)
    assert acc.shape == (3, 5) and acc.dtype == np.int32
    for m in range(3):
        for n in range(5):
            assert acc[m, n] == sum(int(c[n, k]) * int(xq[m, k]) for k in range(12))


def pin_matmul_exhaustive_codes(o):
    # all 3^8 code rows against one fixed token
    import itertools
    xq = np.array([[127, -128 + 1, 5, -3, 64, 0, -77, 1]], np.int8)
    rows = np.array(list(itertools.product((-1, 0, 1), repeat=8)), np.int8)
    acc = o.ternary_int8_matmul(xq, rows)
    want = rows.astype(np.int64) @ xq[0].astype(np.int64)
    assert np.array_equal(acc[0], want)
    ones = np.ones((1, 8), np.int8)
    assert o.ternary_int8_matmul(xq, ones)[0, 0] == int(xq.astype(np.int64).sum())


def pin_rescale_exact(o):
    rng = np.random.default_rng(61)
    acc = rng.integers(-1_400_000, 1_400_000, size=(4, 40)).astype(np.int32)
    acc[0, :3] = [0, 1, -1]
    gamma = F32(0.0159734)
    s = np.array([31.75, 12700000.0, 0.0423, 1.0], np.float32)
    y = o.rescale(acc, gamma, s)
    for m in range(4):
        for n in range(40):
            t = nearest_f32(Fraction(int(acc[m, n])) * frac_f32(gamma))
            want = nearest_f32(Fraction(float(t)) / frac_f32(s[m]))
            assert y[m, n].view(np.uint32) == want.view(np.uint32), (m, n)


def pin_worked_example(o):
    g = load_golden()
    w = np.array(g["W"], np.float32)
    x = np.array(g["x"], np.float32)
    r = o.bitlinear_forward(x, w)
    assert Fraction(float(r["gamma"])) == Fraction(g["gamma"])
    assert Fraction(float(F32(r["gamma"]) + F32(1e-5))) == Fraction(g["divisor"])
    assert r["codes"].tolist() == g["codes"]
    assert r["packed"].ravel().tolist() == g["packed"]
    assert r["xq"].tolist() == g["xq"]
    assert [Fraction(float(v)) for v in r["scale"]] == [Fraction(v) for v in g["scale"]]
    assert r["acc"].tolist() == g["acc"]
    want_y = [[nearest_f32(Fraction(v)) for v in row] for row in g["y_exact_before_final_rounding"]]
    assert [[F32(v) for v in row] for row in r["y"]] == want_y


def pin_forward_vs_dequantised_fp64(o):
    """y equals the fp64 product of the dequantised operands to fp32 rounding."""
    rng = np.random.default_rng(71)
    w = (rng.standard_normal((48, 256)) * 0.02).astype(np.float32)
    x = rng.standard_normal((6, 256)).astype(np.float32)
    r = o.bitlinear_forward(x, w)
    xd = r["xq"].astype(np.float64) / r["scale"].astype(np.float64)[:, None]
    wd = r["codes"].astype(np.float64) * float(r["gamma"])
    ref = xd @ wd.T
    err = np.abs(r["y"].astype(np.float64) - ref)
    assert np.all(err <= 2.5e-7 * np.abs(ref) + 1e-30)
    # and it is a sane approximation of the unquantised product (ternary error is large but bounded)
    full = x.astype(np.float64) @ w.astype(np.float64).T
    cos = float(np.sum(full * ref) / np.sqrt(np.sum(full ** 2) * np.sum(ref ** 2)))
    assert cos > 0.75, cos


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
