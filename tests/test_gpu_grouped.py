"""GPU parity of the per-group (64) packing and forward against the oracle.

Passage: "BitNet 1-bit LLM 的混合精度微调技术：渐进量化策略", body: per-group
quantisation with a group size of 64 (groups of 64 consecutive k of a row).

The scales, packed codes, activation codes and token scales are compared bit
for bit. y is a floating-point sum over groups with a different scale each:
the library adds the exact products gamma * acc in fp64, so it is compared
with the oracle's once-rounded exact value within
    |y - y_ref| <= 2^-23 |y_ref| + (K/64) 2^-52 bound + 2^-149,
bound = sum_g |gamma * acc| / s (the fp64 summation error plus one fp32
rounding of each side).
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_common import bits, x_to_oracle
from workloads import gaussian_activations, gaussian_weights
from workloads.synth import student_t_weights

pytestmark = pytest.mark.gpu

import bit_ternary_forward_b300 as blt  # noqa: E402  (fails loudly if the library is missing)


def _run(w: torch.Tensor, x: torch.Tensor):
    packed = blt.pack_weights_grouped(w.cuda())
    y, xq, s = blt.forward_grouped(x.cuda(), packed, return_quant=True)
    torch.cuda.synchronize()
    assert blt.device_error() == 0
    return {"gammas": packed.gammas.cpu().numpy(), "packed": packed.wp.cpu().numpy(), "xq": xq.cpu().numpy(),
            "scale": s.cpu().numpy(), "y": y.cpu().numpy()}


def _assert_y(y, ref, k):
    bound = oracle.grouped_y_bound(ref["acc"], ref["gammas"], ref["scale"])
    tol = 2.0 ** -23 * np.abs(ref["y"].astype(np.float64)) + (k // 64) * 2.0 ** -52 * bound + 2.0 ** -149
    err = np.abs(y.astype(np.float64) - ref["y"].astype(np.float64))
    both_inf = np.isinf(y) & np.isinf(ref["y"]) & (np.sign(y) == np.sign(ref["y"]))
    bad = (err > tol) & ~both_inf
    assert not bad.any(), f"{int(bad.sum())} outputs outside the bound; worst {err[bad].max()} vs {tol[bad].min()}"


def _compare(w: torch.Tensor, x: torch.Tensor):
    g = _run(w, x)
    ref = oracle.bitlinear_forward_grouped(x_to_oracle(x), w.numpy())
    np.testing.assert_array_equal(bits(g["gammas"]), bits(ref["gammas"]))
    np.testing.assert_array_equal(g["packed"], oracle.pack_codes(ref["codes"]))
    np.testing.assert_array_equal(g["xq"], ref["xq"])
    np.testing.assert_array_equal(bits(g["scale"]), bits(ref["scale"]))
    _assert_y(g["y"], ref, w.shape[1])
    return g, ref


@pytest.mark.parametrize("m,k,n,xdt", [(1, 2560, 300, torch.bfloat16), (4, 256, 96, torch.float32),
                                       (3, 1024, 257, torch.bfloat16), (2, 128, 5, torch.float32),
                                       (1, 64, 1, torch.bfloat16), (24, 512, 130, torch.bfloat16),
                                       (7, 6912, 33, torch.float32)])
def test_grouped_shapes(m, k, n, xdt):
    w = gaussian_weights(n, k, seed=700 + n)
    x = gaussian_activations(m, k, seed=710 + m, dtype=xdt)
    _compare(w, x)


def test_grouped_student_t_and_scaled_groups():
    # groups of very different scale in one row, heavy tails, an all-zero group
    w = student_t_weights(40, 1024, seed=720)
    w[3, 64:128] *= 1e3
    w[3, 128:192] *= 1e-3
    w[5, 256:320] = 0.0
    w[7, ::64] *= 50.0
    x = gaussian_activations(3, 1024, seed=721, dtype=torch.float32)
    _compare(w, x)


def test_grouped_exact_sum_far_spread_and_subnormals():
    # groups whose weights span more than 2^33 (the one-lane exact sum),
    # subnormal weights, and huge and tiny groups
    rng = np.random.default_rng(722)
    w = (rng.standard_normal((12, 512)) * 0.02).astype(np.float32)
    w[0, 0], w[0, 1] = 1e30, 1e-30
    w[1, 64:128] = rng.standard_normal(64).astype(np.float32) * np.float32(1e-40)   # subnormal group
    w[2, 128:192] = rng.standard_normal(64).astype(np.float32) * np.float32(3e37)
    w[3, 192] = 3e38
    w[3, 193] = -1e-45
    w[4, 256:320] = np.ldexp(1.0, -126)
    w[5, 320:384:2] = 1e20
    w[5, 321:384:2] = 1e-20
    x = gaussian_activations(2, 512, seed=723, dtype=torch.bfloat16)
    _compare(torch.from_numpy(w), x)


def test_grouped_code_tie():
    from test_grouped_oracle_cpu import group_tie_weights
    w, gam, t = group_tie_weights()
    g = _run(torch.from_numpy(w), gaussian_activations(1, w.shape[1], seed=724))
    assert bits(g["gammas"][0, 1]) == bits(gam)
    codes = oracle.unpack_codes(g["packed"])
    assert codes[0, 126] == 0 and codes[0, 127] == 0
    np.testing.assert_array_equal(bits(g["gammas"]), bits(oracle.group_gammas(w)))


def test_grouped_decode_2b_full_size_sampled():
    # the 2B up projection at full size: every scale and packed byte of sampled
    # rows, and y on those rows, against the oracle on the rows alone
    n, k = 6912, 2560
    w = gaussian_weights(n, k, seed=725)
    x = gaussian_activations(1, k, seed=726)
    g = _run(w, x)
    rows = np.random.default_rng(727).choice(n, size=24, replace=False)
    wr = w.numpy()[rows]
    ref = oracle.bitlinear_forward_grouped(x_to_oracle(x), wr)
    np.testing.assert_array_equal(bits(g["gammas"][rows]), bits(ref["gammas"]))
    np.testing.assert_array_equal(g["packed"][rows], oracle.pack_codes(ref["codes"]))
    np.testing.assert_array_equal(g["xq"], ref["xq"])
    _assert_y(g["y"][:, rows], ref, k)


def test_grouped_per_tensor_limit():
    # every group holds the same 64 values: the scales equal the per-tensor gamma
    # and y agrees with the per-tensor forward within the bound
    pattern = gaussian_weights(1, 64, seed=728)
    w = pattern.repeat(50, 16)
    x = gaussian_activations(2, 1024, seed=729, dtype=torch.float32)
    g, ref = _compare(w, x)
    gamma = oracle.absmean_gamma(w.numpy())
    assert (bits(g["gammas"]) == bits(np.float32(gamma))).all()


def test_grouped_errors():
    w = gaussian_weights(8, 96, seed=730).cuda()
    with pytest.raises(blt.BitLinearError):
        blt.pack_weights_grouped(w)          # K % 64 != 0
