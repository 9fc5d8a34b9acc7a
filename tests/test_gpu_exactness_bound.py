"""GPU parity at the tensor-core path's exactness bound.

The tensor-core contraction (M >= 17, K % 64 == 0) runs as an fp16 MMA with an
fp32 accumulator and is exact only because every partial sum it forms is an
integer multiple of 2^-24 no larger than 2 * 128 * K * 2^-24, which is 1 at
K = 65536, the largest K the library accepts. These tests drive that sum to
the bound and compare with the oracle bit for bit:

* K = 65536, on split tiles (M = 17 and 64: every tile's k-stages spread over
  all SMs, partial sums meeting through fp32 atomics in the workspace) and on
  whole tiles (M = 300 and 1024, ragged token tiles);
* tokens of all +127, all -127 and all -128 (the int8 extreme, reachable
  through bitlinear_gemm_i32) against weight rows of all +1 (field 2), so
  |sum field * x_q| reaches 2 * 127 * 65536 and 2^24; tokens whose running
  sum climbs to half the bound and comes back; a long run of +127 followed by
  small terms of the opposite sign; random tokens;
* the int32 accumulator (bitlinear_gemm_i32), y from bitlinear_gemm with
  given scales, and the bf16 forward (activation pass included), with the
  oracle's matmul evaluated on the distinct weight rows and broadcast.

A last group checks the rescale where the reciprocal-and-correction division
would overflow or underflow: huge activations with large gamma (y = +-inf in
IEEE arithmetic) and tiny quotients, on the dp4a GEMV (M <= 4) and on the
tensor-core path.

Passage: "穿越1比特的奇幻旅程" (2B4T summary), section "GPU端：CUDA内核的定制魔法"
(the W1.58A8 matmul); "BitNet 1-bit LLM 的混合精度微调技术", the forward-pass
sentence (rescale by the factors).
"""

import numpy as np
import pytest
import torch

import oracle
from gpu_common import assert_y_close, bits, x_to_oracle

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU runs deselect -m gpu
    pytest.skip("needs a CUDA device", allow_module_level=True)

import bit_ternary_forward_b300 as blt  # noqa: E402

K = 65536
N_ROW_TYPES = 8


def _unique_code_rows(seed: int) -> np.ndarray:
    """The distinct weight rows: all +1, all -1, all 0, +1 then -1, four random."""
    rng = np.random.default_rng(seed)
    u = np.empty((N_ROW_TYPES, K), dtype=np.int8)
    u[0] = 1
    u[1] = -1
    u[2] = 0
    u[3, :K // 2] = 1
    u[3, K // 2:] = -1
    u[4:] = rng.integers(-1, 2, size=(N_ROW_TYPES - 4, K))
    return u


def _tokens_i8(m: int, seed: int) -> np.ndarray:
    """Token m has pattern m % 6: +127; -128; -127; +127 then -127; a long run
    of +127 then -1s; uniform random int8."""
    rng = np.random.default_rng(seed)
    xq = np.empty((m, K), dtype=np.int8)
    for i in range(m):
        t = i % 6
        if t == 0:
            xq[i] = 127
        elif t == 1:
            xq[i] = -128
        elif t == 2:
            xq[i] = -127
        elif t == 3:
            xq[i, :K // 2] = 127
            xq[i, K // 2:] = -127
        elif t == 4:
            xq[i, :65000] = 127
            xq[i, 65000:] = -1
        else:
            xq[i] = rng.integers(-128, 128, size=K)
    return xq


def _weights(n: int, seed: int):
    """(unique code rows, row type of each of n rows, packed [n][K/4])."""
    u = _unique_code_rows(seed)
    row_type = np.arange(n) % N_ROW_TYPES
    packed = oracle.pack_codes(u)[row_type]
    return u, row_type, np.ascontiguousarray(packed)


def _plan_kind(m: int, n: int):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    p, _ = blt.tc_schedule(m, n, K, sms)
    return "split" if p.sk_tiles and not p.dp_tiles else ("whole" if not p.sk_tiles else "mixed")


@pytest.mark.parametrize("m,n,kind", [(17, 1024, "split"), (64, 1024, "split"),
                                      (300, 2048, "whole"), (1024, 1024, "whole")])
def test_accumulator_and_y_at_the_bound(m, n, kind):
    assert _plan_kind(m, n) == kind
    u, row_type, packed = _weights(n, seed=m)
    xq = _tokens_i8(m, seed=m + 1)
    # the oracle on the distinct rows, broadcast to every row of that type
    acc_u = oracle.ternary_int8_matmul(xq, u)
    acc_ref = acc_u[:, row_type]
    # the bound is reached: |sum field * x_q| = 2^24 for the -128 tokens on +1 rows
    field_sum = acc_ref[:, row_type == 0].astype(np.int64) + xq.astype(np.int64).sum(axis=1)[:, None]
    assert np.abs(field_sum).max() == 2 ** 24

    wp = torch.from_numpy(packed).cuda()
    xq_d = torch.from_numpy(xq).cuda()
    acc = blt.gemm_i32(xq_d, wp)
    rng = np.random.default_rng(m + 2)
    s = (10.0 ** rng.uniform(-3, 3, size=m)).astype(np.float32)
    gamma = np.float32(0.0137)
    y = blt.gemm(xq_d, torch.from_numpy(s).cuda(),
                 blt.PackedWeight(wp, torch.tensor([gamma], dtype=torch.float32).cuda(), n, K))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(acc.cpu().numpy(), acc_ref)
    y_ref = oracle.rescale(acc_ref, gamma, s)
    np.testing.assert_array_equal(bits(y.cpu().numpy()), bits(y_ref))


@pytest.mark.parametrize("m,n", [(17, 1024), (300, 2048)])
def test_bf16_forward_at_the_bound(m, n):
    """The whole forward (activation pass on the device) with tokens of +-1.0,
    half and half, a long run and small opposite terms, and Gaussian tokens."""
    u, row_type, packed = _weights(n, seed=10 + m)
    g = torch.Generator().manual_seed(20 + m)
    x = torch.randn((m, K), generator=g)
    for i in range(m):
        t = i % 5
        if t == 0:
            x[i] = 1.0
        elif t == 1:
            x[i] = -1.0
        elif t == 2:
            x[i, :K // 2] = 1.0
            x[i, K // 2:] = -1.0
        elif t == 3:
            x[i, :65000] = 1.0
            x[i, 65000:] = -1.0 / 127.0
    x = x.to(torch.bfloat16)
    gamma = np.float32(0.0211)
    packed_w = blt.PackedWeight(torch.from_numpy(packed).cuda(), torch.tensor([gamma]).cuda(), n, K)
    y, xq, s = blt.forward(x.cuda(), packed_w, return_quant=True)
    torch.cuda.synchronize()
    xq_ref, s_ref = oracle.quant_act(x_to_oracle(x))
    np.testing.assert_array_equal(xq.cpu().numpy(), xq_ref)
    np.testing.assert_array_equal(bits(s.cpu().numpy()), bits(s_ref))
    acc_ref = oracle.ternary_int8_matmul(xq_ref, u)[:, row_type]
    y_ref = oracle.rescale(acc_ref, gamma, s_ref)
    assert_y_close(y.cpu().numpy(), y_ref)
    np.testing.assert_array_equal(bits(y.cpu().numpy()), bits(y_ref))


def test_gaussian_forward_k65536_tensor_core():
    """Ordinary data at K = 65536 on the tensor-core path, weights packed on the device."""
    from workloads import gaussian_activations, gaussian_weights
    n, m = 256, 40
    w = gaussian_weights(n, K, seed=77)
    x = gaussian_activations(m, K, seed=78)
    packed = blt.pack_weights(w.cuda())
    y, xq, s = blt.forward(x.cuda(), packed, return_quant=True)
    torch.cuda.synchronize()
    ref = oracle.bitlinear_forward(x_to_oracle(x), w.numpy())
    assert bits(packed.gamma.cpu().numpy()[0]) == bits(ref["gamma"])
    np.testing.assert_array_equal(packed.wp.cpu().numpy(), ref["packed"])
    np.testing.assert_array_equal(xq.cpu().numpy(), ref["xq"])
    np.testing.assert_array_equal(bits(y.cpu().numpy()), bits(ref["y"]))


# ------------------------------------------------------------------ rescale outside the fast division's range
@pytest.mark.parametrize("m", [1, 4, 24])
def test_rescale_overflow_and_underflow(m):
    """y = fp32(fp32(acc * gamma) / s) where the quotient overflows to +-inf
    (activations near 1e30, gamma 1e9) or lands far below the normal
    range (tiny gamma, tiny activations' reciprocal scale), through the
    forward's own epilogue: M = 1 and 4 on the dp4a GEMV, M = 24 on the
    tensor-core path."""
    k, n = 256, 96
    rng = np.random.default_rng(300 + m)
    codes = rng.integers(-1, 2, size=(n, k)).astype(np.int8)
    wp = torch.from_numpy(oracle.pack_codes(codes)).cuda()
    cases = []
    # huge activations (s ~ 4e-29, inside the fast division's scale range)
    # with gamma 1e9: t / s overflows to +-inf for most outputs
    xa = (rng.standard_normal((m, k)) * 1e30).astype(np.float32)
    cases.append((xa, np.float32(1.0e9)))
    # tiny gamma with unit activations: t / s far below 2^-100 (subnormal or zero)
    xb = rng.standard_normal((m, k)).astype(np.float32)
    cases.append((xb, np.float32(1.0e-38)))
    # gamma that takes t near the top of the range, activations of magnitude 1
    cases.append((xb, np.float32(3.0e34)))
    for x, gamma in cases:
        packed = blt.PackedWeight(wp, torch.tensor([gamma]).cuda(), n, k)
        y, xq, s = blt.forward(torch.from_numpy(x).cuda(), packed, return_quant=True)
        torch.cuda.synchronize()
        xq_ref, s_ref = oracle.quant_act(x)
        np.testing.assert_array_equal(xq.cpu().numpy(), xq_ref)
        acc_ref = oracle.ternary_int8_matmul(xq_ref, codes)
        with np.errstate(over="ignore", under="ignore"):
            y_ref = oracle.rescale(acc_ref, gamma, s_ref)
        np.testing.assert_array_equal(bits(y.cpu().numpy()), bits(y_ref))


def test_rescale_overflow_reaches_infinity():
    """The overflow case above really produces infinities in the oracle (so
    the comparison covers the branch that used to return NaN)."""
    rng = np.random.default_rng(5)
    k, n, m = 256, 32, 2
    codes = rng.integers(-1, 2, size=(n, k)).astype(np.int8)
    x = (rng.standard_normal((m, k)) * 1e30).astype(np.float32)
    xq_ref, s_ref = oracle.quant_act(x)
    with np.errstate(over="ignore"):
        y_ref = oracle.rescale(oracle.ternary_int8_matmul(xq_ref, codes), np.float32(1.0e9), s_ref)
    assert np.isinf(y_ref).sum() > 0
    packed = blt.PackedWeight(torch.from_numpy(oracle.pack_codes(codes)).cuda(),
                              torch.tensor([np.float32(1.0e9)]).cuda(), n, k)
    y = blt.forward(torch.from_numpy(x).cuda(), packed)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(y.cpu().numpy()), bits(y_ref))
