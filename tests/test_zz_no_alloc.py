"""The packing entry point that allocates nothing, against the ordinary one.

bitlinear_pack_weights_noalloc is for callers that cannot allocate device
memory and so cannot hand the library a workspace: a plugin inside another
framework whose caching allocator owns the GPU, or a runtime that reserved
all device memory up front. It keeps the scratch of the exact absmean in a
static device array inside the library instead.

Each test calls it through the C ABI twice in a row, on different weights,
and checks both calls against bitlinear_pack_weights given a workspace:
packed bytes and gamma bit for bit, the tolerance the parity tests use for
integer outputs and scales. Both calls are also compared with the oracle
(gamma and packed bytes, bit for bit). The second call runs on whatever the
first one left in the shared array, so it shows that nothing needs clearing.

This file is collected last on purpose, and passes alone in a fresh process
(where its first call also sets up the array's address) or after the rest.
"""

import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU runs deselect -m gpu
    pytest.skip("needs a CUDA device", allow_module_level=True)

import numpy as np  # noqa: E402

import bit_ternary_forward_b300 as blt  # noqa: E402
import oracle  # noqa: E402
from workloads import gaussian_weights, student_t_weights  # noqa: E402


def _pack_noalloc(w: torch.Tensor):
    n, k = w.shape
    wp = torch.full((n, k // 4), 0xFF, dtype=torch.uint8, device=w.device)
    gamma = torch.full((1,), float("nan"), dtype=torch.float32, device=w.device)
    st = blt.lib.bitlinear_pack_weights_noalloc(w.data_ptr(), n, k, wp.data_ptr(), gamma.data_ptr(),
                                                torch.cuda.current_stream(w.device).cuda_stream)
    assert st == blt.BL_OK, blt.lib.bitlinear_last_error().decode()
    return wp, gamma


def _check_pair(weights):
    outs = [_pack_noalloc(w) for w in weights]          # two calls back to back on one stream
    torch.cuda.synchronize()
    for w, (wp, gamma) in zip(weights, outs):
        ref = blt.pack_weights(w)                        # the ordinary entry, with a workspace
        torch.cuda.synchronize()
        assert torch.equal(wp, ref.wp)
        assert torch.equal(gamma.view(torch.int32), ref.gamma.view(torch.int32))
        wn = w.cpu().numpy()
        g_ref = oracle.absmean_gamma(wn)
        assert gamma.cpu().numpy().view(np.uint32)[0] == np.float32(g_ref).view(np.uint32)
        np.testing.assert_array_equal(wp.cpu().numpy(), oracle.pack_codes(oracle.ternary_codes(wn, g_ref)))


def test_noalloc_matches_pack_weights_decode_shapes():
    _check_pair([gaussian_weights(6912, 2560, seed=10).cuda(),
                 gaussian_weights(2560, 6912, seed=11).cuda()])


def test_noalloc_matches_pack_weights_ragged_and_heavy_tailed():
    _check_pair([student_t_weights(4096, 4096, seed=1001).cuda(),
                 (gaussian_weights(37, 1028, seed=3) * 1e-3).cuda()])
