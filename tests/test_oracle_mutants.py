"""Plant plausible mistakes in copies of the oracle and check that a pin fails.

The mistakes are planted on the CPU, in a namespace copy of the oracle; the
real oracle is untouched. Each mutant must be rejected by at least one pin,
which shows that the pins constrain every step of the method.
"""

import types

import numpy as np
import pytest

import oracle
from oracle import bitlinear_oracle as ob
from pins import ALL_PINS

F32 = np.float32


def _copy(**overrides):
    ns = types.SimpleNamespace(**{k: getattr(oracle, k) for k in oracle.__all__ if hasattr(oracle, k)}
                               if hasattr(oracle, "__all__") else
                               {k: getattr(oracle, k) for k in dir(oracle) if not k.startswith("_")})
    for k, v in overrides.items():
        setattr(ns, k, v)

    # bitlinear_forward must compose the namespace's (possibly mutated) steps
    def forward(x, w):
        g = ns.absmean_gamma(w)
        c = ns.ternary_codes(w, g)
        p = ns.pack_codes(c)
        xq, s = ns.quant_act(x)
        acc = ns.ternary_int8_matmul(xq, c)
        return {"gamma": g, "codes": c, "packed": p, "xq": xq, "scale": s, "acc": acc,
                "y": ns.rescale(acc, g, s)}
    if "bitlinear_forward" not in overrides:
        ns.bitlinear_forward = forward
    return ns


def m_codes_half_up(w, gamma, eps=ob.EPS_GAMMA):
    d = F32(F32(gamma) + F32(eps))
    q = np.floor(np.asarray(w, np.float32) / d + F32(0.5))
    return np.clip(q, -1, 1).astype(np.int8)


def m_codes_no_eps(w, gamma, eps=ob.EPS_GAMMA):
    return ob.ternary_codes(w, gamma, eps=F32(0.0))


def m_gamma_fp32_mean(w):
    return F32(np.mean(np.abs(np.asarray(w, np.float32)), dtype=np.float32))


def m_gamma_double_rounding(w):
    w = np.asarray(w, np.float32)
    s = ob.exact_abs_sum(w)
    return F32(float(F32(float(s))) / w.size)


def m_gamma_max(w):
    return F32(np.max(np.abs(np.asarray(w, np.float32))))


def m_pack_msb_first(c):
    c = np.asarray(c, np.int8)
    n, k = c.shape
    f = (c.astype(np.int16) + 1).astype(np.uint8).reshape(n, k // 4, 4)
    return (f[..., 3] | (f[..., 2] << 2) | (f[..., 1] << 4) | (f[..., 0] << 6)).astype(np.uint8)


def m_pack_raw_codes(c):
    c = np.asarray(c, np.int8)
    n, k = c.shape
    f = (c.astype(np.int16) & 3).astype(np.uint8).reshape(n, k // 4, 4)
    return (f[..., 0] | (f[..., 1] << 2) | (f[..., 2] << 4) | (f[..., 3] << 6)).astype(np.uint8)


def m_act_divide(x):
    xf = np.asarray(x, np.float32)
    a = np.maximum(np.max(np.abs(xf), axis=1), ob.EPS_ABSMAX)
    s = (F32(127.0) / a).astype(np.float32)
    q = np.clip(np.rint(xf / (a / F32(127.0))[:, None]), -128, 127).astype(np.int8)
    return q, s


def m_act_no_floor(x):
    xf = np.asarray(x, np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        a = np.max(np.abs(xf), axis=1)
        s = (F32(127.0) / a).astype(np.float32)
        q = np.clip(np.nan_to_num(np.rint(xf * s[:, None])), -128, 127).astype(np.int8)
    return q, s


def m_act_half_up(x):
    xf = np.asarray(x, np.float32)
    a = np.maximum(np.max(np.abs(xf), axis=1), ob.EPS_ABSMAX)
    s = (F32(127.0) / a).astype(np.float32)
    v = xf * s[:, None]
    q = np.clip(np.sign(v) * np.floor(np.abs(v) + F32(0.5)), -128, 127).astype(np.int8)
    return q, s


def m_act_per_tensor(x):
    xf = np.asarray(x, np.float32)
    a = np.maximum(np.max(np.abs(xf)), ob.EPS_ABSMAX)
    s = np.full(xf.shape[0], F32(127.0) / a, np.float32)
    return np.clip(np.rint(xf * s[:, None]), -128, 127).astype(np.int8), s


def m_matmul_drop_last_k(xq, codes):
    return ob.ternary_int8_matmul(np.asarray(xq)[:, :-1], np.asarray(codes)[:, :-1])


def m_matmul_sign_flip(xq, codes):
    return ob.ternary_int8_matmul(xq, -np.asarray(codes, np.int8))


def m_matmul_reversed_k(xq, codes):
    return ob.ternary_int8_matmul(xq, np.asarray(codes)[:, ::-1])


def m_rescale_gamma_eps(acc, gamma, s):
    return ob.rescale(acc, F32(F32(gamma) + ob.EPS_GAMMA), s)


def m_rescale_combined_factor(acc, gamma, s):
    s = np.asarray(s, np.float32)
    return np.asarray(acc, np.int32).astype(np.float32) * (F32(gamma) / s)[:, None]


def m_rescale_multiply_s(acc, gamma, s):
    return (np.asarray(acc, np.int32).astype(np.float32) * F32(gamma)) * np.asarray(s, np.float32)[:, None]


def m_round_ratio_truncate(num, den):
    v = ob.round_ratio_to_f32(num, den)
    # truncation toward zero instead of nearest
    from fractions import Fraction
    if Fraction(float(v)) > Fraction(num, den):
        v = np.nextafter(v, F32(0))
    return F32(v)


MUTANTS = {
    "codes_half_up": dict(ternary_codes=m_codes_half_up),
    "codes_no_eps": dict(ternary_codes=m_codes_no_eps),
    "gamma_fp32_mean": dict(absmean_gamma=m_gamma_fp32_mean),
    "gamma_double_rounding": dict(absmean_gamma=m_gamma_double_rounding),
    "gamma_max": dict(absmean_gamma=m_gamma_max),
    "pack_msb_first": dict(pack_codes=m_pack_msb_first),
    "pack_raw_codes": dict(pack_codes=m_pack_raw_codes),
    "act_divide_by_a_over_127": dict(quant_act=m_act_divide),
    "act_no_eps_floor": dict(quant_act=m_act_no_floor),
    "act_half_up": dict(quant_act=m_act_half_up),
    "act_per_tensor": dict(quant_act=m_act_per_tensor),
    "matmul_drop_last_k": dict(ternary_int8_matmul=m_matmul_drop_last_k),
    "matmul_sign_flip": dict(ternary_int8_matmul=m_matmul_sign_flip),
    "matmul_reversed_k": dict(ternary_int8_matmul=m_matmul_reversed_k),
    "rescale_gamma_plus_eps": dict(rescale=m_rescale_gamma_eps),
    "rescale_combined_factor": dict(rescale=m_rescale_combined_factor),
    "rescale_multiply_by_s": dict(rescale=m_rescale_multiply_s),
    "round_ratio_truncate": dict(round_ratio_to_f32=m_round_ratio_truncate),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    ns = _copy(**MUTANTS[name])
    failed = []
    for pin in ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(ns)
        except (AssertionError, ValueError, OverflowError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"no pin rejects the planted mistake {name}"


def test_unmutated_copy_passes_every_pin():
    ns = _copy()
    for pin in ALL_PINS:
        pin(ns)
