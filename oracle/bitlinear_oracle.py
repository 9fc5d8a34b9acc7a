"""Plain, slow, obviously-correct CPU oracle of the BitLinear W1.58A8 forward.

TEST INFRASTRUCTURE ONLY -- see the package docstring. Nothing on the product
path may import this module.

Sources (web pages; cited by title and section):

* [HPFT] "BitNet 1-bit LLM 的混合精度微调技术：渐进量化策略" (blog.hotdry.top,
  2025-10-07), body text, the paragraph listing the quantisation functions
  ("量化函数": weight absmean = mean(|W|), activation absmax = max(|X|, eps=1e-5))
  and the sentence on the forward pass (weights divided by the absmean factor,
  rounded, limited to [-1, 1], multiplied back by the factor; activations
  absmax-quantised per token to 8 bits).
* [2B4T] "穿越1比特的奇幻旅程：高效语言模型的未来之谜" (beiduofen.top; a summary of
  the BitNet b1.58 2B4T Technical Report), section "架构创新：量化魔法的背后"
  (absmean weight quantisation to {-1, 0, +1}; per-token absmax INT8
  activations; no bias terms) and section "GPU端：CUDA内核的定制魔法" (W1.58A8
  matmul, four ternary weights packed into one 8-bit value).
* [STE] "BitNet 中使用直通估计器工程化三元权重训练" (blog.hotdry.top, 2025-10-04),
  section "STE 机制在三元训练中的作用" (round(clamp(.)) uses torch.round, i.e.
  round-half-to-even) and "工程化训练流程与参数配置" (8-bit per-token absmax).

Readings where the pages are silent or disagree (each one is listed with its
reason in the design notes of the repository):

* gamma is per tensor and is the exact mean of |W| rounded once to fp32
  (round-to-nearest-even). The pages give "mean(|W|)" without precision or
  summation order; the exact mean is the only order-free reading.
* The quantisation divisor is d = fp32(gamma + 1e-5); the rescale uses gamma.
* Every rounding is round-half-to-even (torch.round semantics).
* The activation scale is s = 127 / max(max|x|, 1e-5) in fp32; x_q =
  clip(rint(fp32(x * s)), -128, 127).
* Packing: field = code + 1 (0 -> -1, 1 -> 0, 2 -> +1) in 2-bit fields, four
  consecutive k per byte, least-significant field first, row-major [N][K/4].
* acc = sum_k code[n][k] * x_q[m][k] in exact integers; y = fp32(fp32(acc *
  gamma) / s[m]), evaluated left to right.
"""

from __future__ import annotations

import math
from fractions import Fraction
from typing import Dict

import numpy as np

F32 = np.float32

#: epsilon added to gamma in the weight-quantisation divisor
EPS_GAMMA = F32(1e-5)
#: floor on the per-token absmax ([HPFT] "absmax = max(|X|, eps=1e-5)")
EPS_ABSMAX = F32(1e-5)


# --------------------------------------------------------------------------
# exact rounding of a non-negative rational to fp32
# --------------------------------------------------------------------------
def round_ratio_to_f32(num: int, den: int) -> np.float32:
    """The fp32 value nearest to num/den (num >= 0, den > 0), ties to even.

    Written from the IEEE-754 definition: find the binade 2^e <= v < 2^(e+1),
    the spacing of fp32 values there (2^(e-23), or 2^-149 below the normal
    range), the integer number of spacings below v, and round by comparing the
    remainder with half a spacing.
    """
    num = int(num)
    den = int(den)
    if den <= 0 or num < 0:
        raise ValueError("round_ratio_to_f32 needs num >= 0 and den > 0")
    if num == 0:
        return F32(0.0)
    e = num.bit_length() - den.bit_length()
    # now num/den lies in [2^(e-1), 2^(e+1)); pick the binade
    ge = (num >= (den << e)) if e >= 0 else ((num << -e) >= den)
    if not ge:
        e -= 1
    q_exp = max(e, -126) - 23
    if q_exp >= 0:
        n2, d2 = num, den << q_exp
    else:
        n2, d2 = num << -q_exp, den
    q, r = divmod(n2, d2)
    if 2 * r > d2 or (2 * r == d2 and (q & 1)):
        q += 1
    if q * (2.0 ** q_exp) >= 2.0 ** 128:
        return F32(np.inf)
    return F32(math.ldexp(q, q_exp))


# --------------------------------------------------------------------------
# (a) weight absmean and ternary codes   [HPFT] quantisation functions; [2B4T] 架构创新
# --------------------------------------------------------------------------
def exact_abs_sum(w) -> Fraction:
    """Exact sum of |W| as a rational number.

    By the IEEE-754 binary32 definition, a value with biased exponent field
    e and fraction field f is (2^23 + f) * 2^(e - 150) when e >= 1 and
    f * 2^-149 when e = 0, so |W| summed over all elements is a finite sum of
    integers times powers of two. The integer significands are summed per
    exponent field; each is split into two 12-bit halves so that every
    per-exponent sum stays below 2^53 (up to 2^41 elements) and is therefore
    exact in the fp64 accumulator of bincount. The 256 per-exponent sums are
    then combined as Python rationals.
    """
    b = np.ascontiguousarray(np.asarray(w, dtype=np.float32)).ravel().view(np.uint32)
    e = ((b >> 23) & 0xFF).astype(np.int64)
    if np.any(e == 0xFF):
        raise ValueError("exact_abs_sum: non-finite input")
    if b.size >= 2 ** 41:
        raise ValueError("exact_abs_sum: too many elements for exact per-exponent sums")
    frac = b & 0x7FFFFF
    sig = np.where(e > 0, frac | 0x800000, frac)             # integer significand
    hi = np.bincount(e, weights=(sig >> 12).astype(np.float64), minlength=256)
    lo = np.bincount(e, weights=(sig & 0xFFF).astype(np.float64), minlength=256)
    total = Fraction(0)
    for ex in np.nonzero((hi != 0) | (lo != 0))[0]:
        s = int(hi[ex]) * 4096 + int(lo[ex])
        total += Fraction(s) * Fraction(2) ** (max(int(ex), 1) - 150)
    return total


def absmean_gamma(w) -> np.float32:
    """gamma = mean(|W|) over the whole tensor, rounded once to fp32 (RNE)."""
    w = np.asarray(w, dtype=np.float32)
    if w.size == 0:
        raise ValueError("absmean_gamma: empty weight tensor")
    mean = exact_abs_sum(w) / w.size
    return round_ratio_to_f32(mean.numerator, mean.denominator)


def ternary_codes(w, gamma, eps=EPS_GAMMA) -> np.ndarray:
    """code = clip(rint(W / (gamma + eps)), -1, 1) in fp32, int8 result.

    [HPFT] forward-pass sentence: divide by the absmean factor, round, limit to
    [-1, 1]. The divisor and the quotient are fp32 (IEEE division, RN) and the
    rounding to an integer is half-to-even.
    """
    w = np.asarray(w, dtype=np.float32)
    d = F32(F32(gamma) + F32(eps))
    q = np.rint(w / d)
    return np.clip(q, -1, 1).astype(np.int8)


# --------------------------------------------------------------------------
# (b) packing   [2B4T] GPU端：四个三值权重被打包进一个int8
# --------------------------------------------------------------------------
def pack_codes(codes) -> np.ndarray:
    """Four ternary codes per byte: field_i = code[4j+i] + 1 at bits 2i..2i+1."""
    c = np.asarray(codes, dtype=np.int8)
    n, k = c.shape
    if k % 4:
        raise ValueError("pack_codes: K must be a multiple of 4")
    f = (c.astype(np.int16) + 1).astype(np.uint8).reshape(n, k // 4, 4)
    out = f[..., 0] | (f[..., 1] << 2) | (f[..., 2] << 4) | (f[..., 3] << 6)
    return out.astype(np.uint8)


def unpack_codes(packed) -> np.ndarray:
    """Inverse of pack_codes; raises if a field holds the unused value 3."""
    p = np.asarray(packed, dtype=np.uint8)
    n, kb = p.shape
    f = np.stack([(p >> (2 * i)) & 3 for i in range(4)], axis=-1).reshape(n, kb * 4)
    if np.any(f == 3):
        raise ValueError("unpack_codes: field value 3 is not a ternary code")
    return (f.astype(np.int16) - 1).astype(np.int8)


# --------------------------------------------------------------------------
# (c) per-token absmax int8 activations   [HPFT] absmax per token; [2B4T] INT8 absmax
# --------------------------------------------------------------------------
def bf16_bits_to_f32(bits) -> np.ndarray:
    """bf16 is the top half of an fp32 word: widen by a 16-bit shift."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def quant_act(x):
    """Per-token absmax quantisation to int8.

    a_m = max(max_k |x[m][k]|, 1e-5);  s_m = 127 / a_m;
    x_q = clip(rint(x * s_m), -128, 127).  All fp32, RN, ties to even.
    Returns (x_q int8 [M][K], s fp32 [M]).
    """
    xf = np.asarray(x, dtype=np.float32)
    if xf.ndim != 2 or xf.shape[1] == 0:
        raise ValueError("quant_act: x must be [M][K] with K > 0")
    a = np.maximum(np.max(np.abs(xf), axis=1), EPS_ABSMAX).astype(np.float32)
    s = (F32(127.0) / a).astype(np.float32)
    q = np.clip(np.rint(xf * s[:, None]), -128, 127).astype(np.int8)
    return q, s


# --------------------------------------------------------------------------
# (d) ternary x int8 matmul and rescale   [2B4T] W1.58A8 matmul; [HPFT] multiply back
# --------------------------------------------------------------------------
def ternary_int8_matmul(xq, codes) -> np.ndarray:
    """acc[m][n] = sum_k codes[n][k] * xq[m][k], exact integers, int32 result."""
    acc = np.asarray(xq, dtype=np.int64) @ np.asarray(codes, dtype=np.int64).T
    if acc.size and np.abs(acc).max() >= 2 ** 31:
        raise OverflowError("accumulator exceeds int32")
    return acc.astype(np.int32)


def rescale(acc, gamma, s) -> np.ndarray:
    """y = (fp32(acc) * gamma) / s_m, two fp32 operations in this order."""
    acc = np.asarray(acc, dtype=np.int32)
    if acc.size and np.abs(acc).max() >= 2 ** 24:
        raise OverflowError("acc not exactly representable in fp32")
    s = np.asarray(s, dtype=np.float32)
    return (acc.astype(np.float32) * F32(gamma)) / s[:, None]


def bitlinear_forward(x, w) -> Dict[str, np.ndarray]:
    """All steps of the forward in the pages' order; returns every intermediate."""
    gamma = absmean_gamma(w)
    codes = ternary_codes(w, gamma)
    packed = pack_codes(codes)
    xq, s = quant_act(x)
    acc = ternary_int8_matmul(xq, codes)
    y = rescale(acc, gamma, s)
    return {"gamma": gamma, "codes": codes, "packed": packed, "xq": xq, "scale": s,
            "acc": acc, "y": y}
