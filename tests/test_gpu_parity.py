"""GPU parity: the CUDA path (through the C ABI) against the oracle.

Bit-exact on gamma, packed bytes, x_q, per-token scales and the int32
accumulators; y is checked both within 1e-6 relative (the stated tolerance)
and bit for bit (the kernels evaluate the rescale in the oracle's order).
"""

import numpy as np
import pytest
import torch

import oracle
from gpu_common import bits, compare_full, compare_sampled_rows, gpu_run, oracle_weights, x_to_oracle
from workloads import WORKLOADS, gaussian_activations, gaussian_weights, make_projection_inputs
from workloads.synth import student_t_weights

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU runs deselect -m gpu
    pytest.skip("needs a CUDA device", allow_module_level=True)

import bit_ternary_forward_b300 as blt  # noqa: E402  (fails loudly if the library is missing)


# ------------------------------------------------------------------ the five workloads
def test_cpu_small_every_output():
    p = WORKLOADS["cpu_small"].projections[0]
    w, x = make_projection_inputs(p)
    compare_full(w, x)


@pytest.mark.parametrize("idx", [0, 1])
def test_decode_2b_every_output(idx):
    p = WORKLOADS["decode_2b"].projections[idx]
    w, x = make_projection_inputs(p)
    compare_full(w, x)


@pytest.mark.parametrize("idx", range(6))
def test_skinny_2b_outliers_every_output(idx):
    p = WORKLOADS["skinny_2b"].projections[idx]
    w, x = make_projection_inputs(p)
    compare_full(w, x)


@pytest.mark.parametrize("idx", [0, 1])
def test_prefill_2b_sampled_tokens(idx):
    p = WORKLOADS["prefill_2b"].projections[idx]
    w, x = make_projection_inputs(p)
    rows = np.sort(np.random.default_rng(idx).choice(p.m, 48, replace=False))
    rows = np.concatenate([[0, p.m - 1], rows])
    compare_sampled_rows(w, x, rows)


@pytest.mark.parametrize("proj", range(4))
def test_stack_7b_layer0_decode_every_output(proj):
    p = WORKLOADS["stack_7b_decode"].projections[proj]
    w, x = make_projection_inputs(p)
    compare_full(w, x)


@pytest.mark.parametrize("proj", [1, 3])
def test_stack_7b_last_layer_prefill_sampled(proj):
    p = WORKLOADS["stack_7b_prefill"].projections[31 * 4 + proj]
    w, x = make_projection_inputs(p)
    rows = np.array([0, 1, 777, 1500, 2047])
    compare_sampled_rows(w, x, rows)


# ------------------------------------------------------------------ chained calls (dependent launch)
@pytest.mark.parametrize("m", [1, 3, 8, 24])
def test_chained_forwards_against_the_oracle_chain(m):
    """Forwards back to back on one stream, each reading the fp32 output of
    the one before as its input, with every weight packed on the same stream
    just before its forward (so a forward's weights are written by the kernel
    it follows). Every kernel is a programmatic dependent launch; the chain
    must match the oracle's chain output by output, bit for bit."""
    dims = [2560, 6912, 2560, 4096, 1088, 256]
    ws = [gaussian_weights(dims[i + 1], dims[i], seed=700 + i) for i in range(len(dims) - 1)]
    x0 = gaussian_activations(m, dims[0], seed=800 + m, dtype=torch.float32)
    s = torch.cuda.Stream()
    outs = []
    with torch.cuda.stream(s):
        wd = [w.cuda() for w in ws]
        x = x0.cuda()
        for w in wd:
            packed = blt.pack_weights(w)
            x = blt.forward(x, packed)
            outs.append(x)
    s.synchronize()
    ref = x_to_oracle(x0)
    for i, (w, y) in enumerate(zip(ws, outs)):
        r = oracle.bitlinear_forward(ref, w.numpy())
        np.testing.assert_array_equal(bits(y.cpu().numpy()), bits(r["y"]), err_msg=f"projection {i}")
        ref = r["y"]


# ------------------------------------------------------------------ shapes and tails
@pytest.mark.parametrize("m,n,k", [
    (1, 1, 4), (1, 3, 8), (2, 5, 12), (3, 7, 100), (5, 9, 64), (4, 33, 192), (2, 17, 1028),
    (7, 65, 320), (9, 31, 4096), (1, 130, 65536), (4, 64, 65536), (17, 129, 960), (64, 300, 2560),
    (3, 200, 16384), (2, 77, 32768), (1, 4096, 11008), (2, 1000, 64),
    (65, 257, 128), (129, 96, 1088), (33, 70, 100), (17, 9, 1028),
])
@pytest.mark.parametrize("xdt", [torch.bfloat16, torch.float32])
def test_shapes(m, n, k, xdt):
    w = gaussian_weights(n, k, seed=1000 + n + k)
    x = gaussian_activations(m, k, seed=2000 + m + k, dtype=xdt)
    compare_full(w, x)


@pytest.mark.parametrize("m,n,k", [(100, 300, 1024), (700, 500, 2048), (512, 896, 4096), (512, 19200, 256)])
def test_split_tile_contraction(m, n, k):
    """Tensor-core shapes whose tiles are split by k-stages over several CTAs
    (partial sums meet in the fp32 buffer): a few tiles with ragged M and N,
    runs that cross tile boundaries, and whole tiles followed by a split
    remainder."""
    w = gaussian_weights(n, k, seed=3000 + n + k)
    x = gaussian_activations(m, k, seed=4000 + m + k)
    compare_full(w, x)


# Shapes that select each token-tile width of the tensor-core contraction, whole
# and split by k-stages, on a 148-SM B300: two accumulators with weight stages
# beside them (32-224 tokens) and the one-accumulator 256-token tile.
TILE_CASES = [
    # (width, split, M, N, K)
    (32, False, 33, 1024, 512), (32, True, 17, 2560, 2560),
    (64, False, 65, 1024, 512), (64, True, 33, 2560, 2560),
    (128, False, 65, 2560, 2560), (128, True, 17, 1024, 512),
    (160, False, 1000, 2560, 512), (160, True, 129, 1024, 1024),
    (192, True, 161, 1024, 1024), (224, False, 1500, 2560, 512),
    (256, False, 193, 2560, 2560), (256, True, 2048, 2560, 2560),
]


@pytest.mark.parametrize("bn,split,m,n,k", TILE_CASES)
def test_every_tile_width_and_split(bn, split, m, n, k):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan, _ = blt.tc_schedule(m, n, k, sms)
    if sms == 148:
        assert (plan.bn, plan.sk_tiles > 0) == (bn, split), plan
    w = gaussian_weights(n, k, seed=6000 + bn + n)
    x = gaussian_activations(m, k, seed=6100 + m + k)
    if m * n * k <= 300_000_000:
        compare_full(w, x)
    else:
        rows = np.sort(np.random.default_rng(bn).choice(m, 40, replace=False))
        compare_sampled_rows(w, x, np.concatenate([[0, m - 1], rows]))


# ------------------------------------------------------------------ degenerate and special values
def test_zero_token_and_zero_weights():
    w = gaussian_weights(64, 256, seed=5)
    x = gaussian_activations(6, 256, seed=6)
    x[2] = 0
    x[4, :] = 0
    compare_full(w, x)
    compare_full(torch.zeros(32, 128), gaussian_activations(3, 128, seed=7))


def test_gamma_tie_element():
    from pins import _tie_tensor
    wt, g, t = _tie_tensor()                    # contains +-t with t == (gamma + 1e-5)/2 exactly
    w = torch.from_numpy(wt.copy())
    r = gpu_run(w, gaussian_activations(2, w.shape[1], seed=8))
    assert bits(r["gamma"]) == bits(g)
    codes = oracle.unpack_codes(r["packed"]).ravel()
    assert codes[-2] == 0 and codes[-1] == 0


@pytest.mark.parametrize("scale", [1e-30, 1e-3, 1.0, 1e4, 1e30])
def test_weight_magnitudes(scale):
    w = gaussian_weights(48, 512, seed=9) * scale
    compare_full(w.to(torch.float32), gaussian_activations(3, 512, seed=10))


def test_subnormal_and_mixed_exponent_weights():
    g = torch.Generator().manual_seed(11)
    w = torch.randn(40, 256, generator=g) * torch.exp2(torch.randint(-140, 60, (40, 256), generator=g).float())
    w[0, :8] = torch.tensor([1e-45, -3e-45, 0.0, -0.0, 2e-44, 1e-40, 3e38, -3e38])
    compare_full(w.to(torch.float32), gaussian_activations(2, 256, seed=12))


def test_student_t_weights_and_outlier_tokens():
    w = student_t_weights(96, 1024, seed=13)
    x = gaussian_activations(8, 1024, seed=14)
    x[:, ::97] *= 50
    compare_full(w, x.to(torch.bfloat16))


def test_activation_ties_on_device():
    # a = 127 exactly, so s = 1 and x*s = x: halves must go to the even integer
    x = torch.tensor([[2.5, 3.5, -0.5, 126.5, 127.0, -1.5, 0.5, -2.5]], dtype=torch.float32)
    xq, s = blt.quant_act(x.cuda())
    assert s.cpu().tolist() == [1.0]
    assert xq.cpu().tolist() == [[2, 4, 0, 126, 127, -2, 0, -2]]


# ------------------------------------------------------------------ the stand-alone packing calls
@pytest.mark.parametrize("n,k", [(1, 4), (3, 12), (7, 1028), (256, 1024), (1000, 1028), (2048, 2052)])
def test_absmean_then_quantize_pack_match_pack_weights(n, k):
    """bitlinear_absmean + bitlinear_quantize_pack (gamma read from memory) and
    bitlinear_pack_weights (gamma combined inside the packing kernel) both
    give the oracle's gamma and bytes: one-byte and one-word outputs, tails
    of 1..3 bytes, and grids with several ring stages per CTA."""
    w = gaussian_weights(n, k, seed=n + k)
    g_ref, _, wp_ref = oracle_weights(w)
    wd = w.cuda()
    gamma = blt.absmean(wd)
    wp = blt.quantize_pack(wd, gamma)
    packed = blt.pack_weights(wd)
    torch.cuda.synchronize()
    assert bits(gamma.cpu().numpy()[0]) == bits(g_ref)
    assert bits(packed.gamma.cpu().numpy()[0]) == bits(g_ref)
    np.testing.assert_array_equal(wp.cpu().numpy(), wp_ref)
    np.testing.assert_array_equal(packed.wp.cpu().numpy(), wp_ref)


# ------------------------------------------------------------------ the pages' variant quantisers
_VARIANT = {"alpha_round": oracle.alpha_round_quantize, "threshold": oracle.threshold_quantize}


def _check_variant(w, quantizer, factor, x=None):
    """Codes (packed bytes) and scale bit-exact; with x, the forward with that scale too."""
    codes, scale = _VARIANT[quantizer](w.numpy(), np.float32(factor))
    packed = blt.pack_weights(w.cuda(), quantizer=quantizer, factor=factor)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(packed.wp.cpu().numpy(), oracle.pack_codes(codes))
    assert bits(packed.gamma.cpu().numpy()[0]) == bits(scale), (quantizer, factor)
    if x is not None:
        y, xq, s = blt.forward(x.cuda(), packed, return_quant=True)
        torch.cuda.synchronize()
        xq_ref, s_ref = oracle.quant_act(x_to_oracle(x))
        y_ref = oracle.rescale(oracle.ternary_int8_matmul(xq_ref, codes), scale, s_ref)
        np.testing.assert_array_equal(xq.cpu().numpy(), xq_ref)
        np.testing.assert_array_equal(bits(y.cpu().numpy()), bits(y_ref))


@pytest.mark.parametrize("quantizer", ["alpha_round", "threshold"])
@pytest.mark.parametrize("factor", [0.7, 0.6, 0.75])
@pytest.mark.parametrize("n,k", [(3, 12), (257, 1028), (2048, 2560)])
def test_variant_quantizers_match_oracle(quantizer, factor, n, k):
    w = gaussian_weights(n, k, seed=n * 7 + k)
    x = gaussian_activations(3, k, seed=k) if n * k <= 300_000 else None
    _check_variant(w, quantizer, factor, x)


@pytest.mark.parametrize("quantizer", ["alpha_round", "threshold"])
def test_variant_quantizers_special_weights(quantizer):
    # Student-t weights and an outlier token through the tensor-core forward
    _check_variant(student_t_weights(96, 1024, seed=21), quantizer, 0.7,
                   gaussian_activations(80, 1024, seed=22).to(torch.bfloat16))
    # tiny weights: alpha below 2^-125, where the codes come from the exact quotient
    _check_variant((gaussian_weights(16, 256, seed=23) * 1e-36).to(torch.float32), quantizer, 0.7)
    # an all-zero tensor: scale 0, all codes 0
    _check_variant(torch.zeros(8, 64), quantizer, 0.7)
    # elements exactly at the thresholds (alpha / 2 and delta), found on the host
    w = gaussian_weights(64, 256, seed=24).numpy()
    for _ in range(4):
        t = oracle.scaled_mean(w)
        w[0, 0] = np.float32(t * np.float32(0.5)) if quantizer == "alpha_round" else t
        w[0, 1] = -w[0, 0]
    assert oracle.scaled_mean(w) == t
    _check_variant(torch.from_numpy(w.copy()), quantizer, 0.7)


# ------------------------------------------------------------------ invariants of the device path
def test_pack_is_deterministic_and_order_free():
    w = gaussian_weights(512, 1024, seed=15)
    a = blt.pack_weights(w.cuda())
    b = blt.pack_weights(w.cuda())
    perm = torch.randperm(w.numel(), generator=torch.Generator().manual_seed(16))
    c = blt.pack_weights(w.flatten()[perm].reshape(1024, 512).contiguous().cuda())
    torch.cuda.synchronize()
    assert torch.equal(a.wp, b.wp) and torch.equal(a.gamma, b.gamma)
    assert torch.equal(a.gamma, c.gamma)


def test_non_default_stream_and_reuse():
    w = gaussian_weights(256, 512, seed=17)
    x = gaussian_activations(3, 512, seed=18)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        packed = blt.pack_weights(w.cuda())
        y1 = blt.forward(x.cuda(), packed)
        y2 = blt.forward(x.cuda(), packed)
    s.synchronize()
    assert torch.equal(y1, y2)
    ref = oracle.bitlinear_forward(x_to_oracle(x), w.numpy())
    np.testing.assert_array_equal(bits(y1.cpu().numpy()), bits(ref["y"]))


def test_errors_raise_not_fallback():
    w = gaussian_weights(8, 64, seed=19).cuda()
    with pytest.raises(blt.BitLinearError):
        blt.pack_weights(w[:, :62].contiguous())          # K % 4 != 0
    packed = blt.pack_weights(w)
    with pytest.raises(ValueError):
        blt.forward(torch.zeros(2, 60, device="cuda", dtype=torch.bfloat16), packed)


@pytest.mark.parametrize("gexp", [-40, -8, 0, 20])
def test_tensor_core_rescale_bit_exact_over_scale_range(gexp):
    # the tensor-core epilogue divides with a reciprocal and one correction
    # step inside 2^-96..2^96 and with IEEE division outside; both must give
    # fp32(fp32(acc * gamma) / s) bit for bit over every scale 127/max(|x|,
    # 1e-5) can take (about 3.7e-37 .. 1.27e7)
    rng = np.random.default_rng(200 + gexp)
    m, n, k = 2048, 256, 128
    xq = rng.integers(-127, 128, size=(m, k)).astype(np.int8)
    codes = rng.integers(-1, 2, size=(n, k)).astype(np.int8)
    s = (10.0 ** rng.uniform(-36.4, 7.1, size=m)).astype(np.float32)
    gamma = np.float32(rng.uniform(1.0, 2.0) * 2.0 ** gexp)
    packed = blt.PackedWeight(torch.from_numpy(oracle.pack_codes(codes)).cuda(),
                              torch.tensor([gamma], dtype=torch.float32).cuda(), n, k)
    y = blt.gemm(torch.from_numpy(xq).cuda(), torch.from_numpy(s).cuda(), packed)
    acc = blt.gemm_i32(torch.from_numpy(xq).cuda(), packed.wp)
    torch.cuda.synchronize()
    acc_ref = oracle.ternary_int8_matmul(xq, codes)
    np.testing.assert_array_equal(acc.cpu().numpy(), acc_ref)
    y_ref = oracle.rescale(acc_ref, gamma, s)
    np.testing.assert_array_equal(bits(y.cpu().numpy()), bits(y_ref))


def test_no_bounded_wait_gave_up():
    # every kernel above finished its waits for its own copies in time
    torch.cuda.synchronize()
    assert blt.device_error() == 0
