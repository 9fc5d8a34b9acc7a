"""GPU parity of the lookup-table decode GEMV (the table idea of bitnet.cpp's
TL1 kernel; "部署 BitNet 1-bit LLM：三元权重边缘推理优化", kernel types) against
the oracle: y bit for bit, and bit for bit equal to the dp4a path's y."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_common import bits, x_to_oracle
from workloads import gaussian_activations, gaussian_weights, make_projection_inputs, WORKLOADS
from workloads.synth import student_t_weights

pytestmark = pytest.mark.gpu

import bit_ternary_forward_b300 as blt  # noqa: E402  (fails loudly if the library is missing)


def _check(w: torch.Tensor, x: torch.Tensor):
    packed = blt.pack_weights(w.cuda())
    y_lut = blt.forward_lut(x.cuda(), packed)
    y_dp4a = blt.forward(x.cuda(), packed)
    torch.cuda.synchronize()
    ref = oracle.bitlinear_forward(x_to_oracle(x), w.numpy())
    np.testing.assert_array_equal(bits(y_lut.cpu().numpy()), bits(ref["y"]))
    np.testing.assert_array_equal(bits(y_lut.cpu().numpy()), bits(y_dp4a.cpu().numpy()))


@pytest.mark.parametrize("idx", [0, 1])
def test_lut_decode_2b_every_output(idx):
    p = WORKLOADS["decode_2b"].projections[idx]
    w, x = make_projection_inputs(p)
    _check(w, x)


@pytest.mark.parametrize("n,k,xdt", [(1, 64, torch.float32), (37, 128, torch.bfloat16), (300, 1088, torch.float32),
                                     (1000, 4096, torch.bfloat16), (257, 11008, torch.bfloat16),
                                     (64, 16384, torch.float32)])
def test_lut_shapes(n, k, xdt):
    _check(gaussian_weights(n, k, seed=800 + n), gaussian_activations(1, k, seed=810 + k, dtype=xdt))


def test_lut_heavy_tails_zero_token_and_extremes():
    w = student_t_weights(96, 2560, seed=820)
    _check(w, gaussian_activations(1, 2560, seed=821))
    _check(w, torch.zeros(1, 2560))
    x = gaussian_activations(1, 2560, seed=822, dtype=torch.float32) * 1e30
    _check(w, x)
    x = gaussian_activations(1, 2560, seed=823, dtype=torch.float32) * 1e-30
    _check(w, x)


def test_lut_errors():
    packed = blt.pack_weights(gaussian_weights(8, 128, seed=830).cuda())
    with pytest.raises(blt.BitLinearError):
        blt.forward_lut(gaussian_activations(2, 128, seed=831).cuda(), packed)      # M != 1
    big = blt.pack_weights(gaussian_weights(2, 32768, seed=832).cuda())
    with pytest.raises(blt.BitLinearError):
        blt.forward_lut(gaussian_activations(1, 32768, seed=833).cuda(), big)       # K > 16384
