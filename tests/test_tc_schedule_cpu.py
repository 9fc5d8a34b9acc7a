"""The tensor-core contraction's launch plan and work lists, on the host.

bitlinear_tc_schedule runs the kernel's own schedule code (the same
host/device functions the persistent kernel calls) without a GPU. These tests
check, for the bench shapes, skinny and ragged shapes and several SM counts,
that the plan is consistent and that the CTAs' work items cover every output
tile's k-stages exactly once, in the order the kernel relies on.
"""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

TILE_WIDTHS = {256, 224, 192, 160, 128, 64, 32}

SHAPES = [
    # (M, N, K): 2B-class prefill, 7B-class prefill, skinny batches, ragged cases
    (2048, 6912, 2560), (2048, 2560, 6912),
    (2048, 12288, 4096), (2048, 4096, 4096), (2048, 11008, 4096), (2048, 4096, 11008),
    (17, 2560, 2560), (32, 6912, 2560), (64, 2560, 2560), (64, 12288, 4096),
    (33, 70, 128), (96, 256, 256), (100, 1000, 640), (300, 129, 1024), (1000, 4099, 192),
    (17, 1, 64), (32, 256, 64), (64, 6912, 64), (2049, 6913, 2560),
]
SMS = [148, 132, 7, 1]


@pytest.fixture(scope="module")
def blt():
    import importlib.util
    spec = importlib.util.spec_from_file_location("bl_build", os.path.join(ROOT, "bit_ternary_forward_b300", "build.py"))
    build = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(build)
    build.build()
    import bit_ternary_forward_b300 as b
    return b


def ceil_div(a, b):
    return -(-a // b)


@pytest.mark.parametrize("sms", SMS)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_schedule_covers_every_stage_once(blt, shape, sms):
    M, N, K = shape
    p, items = blt.tc_schedule(M, N, K, sms)

    # the plan
    assert p.bn in TILE_WIDTHS
    assert p.row_tiles == ceil_div(N, 128)
    assert p.k_iters == K // 64
    assert p.token_tiles == ceil_div(M, p.bn)
    assert (p.token_tiles - 1) * p.bn < M            # no empty token tile
    tiles = p.row_tiles * p.token_tiles
    assert p.dp_tiles + p.sk_tiles == tiles
    assert 1 <= p.grid <= sms and len(items) == p.grid
    assert p.dp_tiles % sms == 0 or p.sk_tiles == 0   # split tiles only after whole rounds
    if p.sk_tiles:
        assert 1 <= p.sk_ctas <= p.grid
        assert p.sk_bytes >= p.sk_tiles * p.bn * 128 * 4 + p.sk_tiles * 4
    else:
        assert p.sk_ctas == 0

    # coverage: whole tiles once, split tiles by disjoint ranges that fill [0, k_iters)
    seen = {}
    for b, work in enumerate(items):
        for tile, k0, k1 in work:
            assert 0 <= tile < tiles and 0 <= k0 < k1 <= p.k_iters
            seen.setdefault(tile, []).append((k0, k1, b))
    assert sorted(seen) == list(range(tiles))
    for tile, parts in seen.items():
        if tile < p.dp_tiles:
            assert parts == [(0, p.k_iters, tile % p.grid)]      # round-robin, whole
        else:
            parts.sort()
            assert parts[0][0] == 0 and parts[-1][1] == p.k_iters
            for (a0, a1, _), (b0, b1, _) in zip(parts, parts[1:]):
                assert a1 == b0                                  # no gap, no overlap

    # order and balance: a CTA's split run first, in tile order, then its whole tiles
    runs = []
    for b, work in enumerate(items):
        split = [w for w in work if w[0] >= p.dp_tiles]
        whole = [w for w in work if w[0] < p.dp_tiles]
        assert work == split + whole
        assert [w[0] for w in split] == sorted(w[0] for w in split)
        assert [w[0] for w in whole] == list(range(b, p.dp_tiles, p.grid))
        if split:
            assert b < p.sk_ctas
            # a run is contiguous in the split tiles' stage order
            flat = [(t - p.dp_tiles) * p.k_iters + k for t, k0, k1 in split for k in range(k0, k1)]
            assert flat == list(range(flat[0], flat[-1] + 1))
            runs.append(len(flat))
    if p.sk_tiles:
        assert len(runs) == p.sk_ctas
        assert max(runs) - min(runs) <= 1                         # equal runs to within one stage


def test_plans_of_the_measured_shapes(blt):
    """The plans the profiles were measured with on 148 SMs."""
    p, _ = blt.tc_schedule(2048, 6912, 2560, 148)     # up projection: three rounds of whole tiles
    assert (p.bn, p.dp_tiles, p.sk_tiles, p.grid) == (256, 432, 0, 148)
    p, items = blt.tc_schedule(2048, 2560, 6912, 148)  # down: 12 tiles split over all CTAs first
    assert (p.bn, p.dp_tiles, p.sk_tiles, p.sk_ctas) == (256, 148, 12, 148)
    assert items[0] == [(148, 0, 8), (0, 0, 108)]
    p, _ = blt.tc_schedule(64, 6912, 2560, 148)       # skinny: one 64-token tile, every tile split
    assert (p.bn, p.token_tiles, p.dp_tiles, p.sk_tiles) == (64, 1, 0, 54)


def test_workspace_size_includes_the_split_buffer(blt):
    # no GPU here, so the library plans for 148 SMs
    for M, N, K in [(2048, 2560, 6912), (64, 6912, 2560), (96, 256, 256)]:
        p, _ = blt.tc_schedule(M, N, K, 148)
        align = lambda v: -(-v // 256) * 256                    # noqa: E731
        want = align(M * K * 2) + 2 * align(M * 4) + p.sk_bytes
        assert blt.lib.bitlinear_forward_workspace_bytes(M, N, K) == want


def test_schedule_rejects_bad_arguments(blt):
    import ctypes
    plan = (ctypes.c_int32 * 9)()
    f = blt.lib.bitlinear_tc_schedule
    assert f(2048, 256, 100, 148, plan, None, None, 0) == blt.BL_ERR_INVALID_ARG   # K % 64
    assert f(0, 256, 256, 148, plan, None, None, 0) == blt.BL_ERR_INVALID_ARG
    assert f(64, 256, 256, 0, plan, None, None, 0) == blt.BL_ERR_INVALID_ARG
    assert f(64, 256, 256, 148, None, None, None, 0) == blt.BL_ERR_INVALID_ARG
    counts = (ctypes.c_int32 * 148)()
    items = (ctypes.c_int32 * (148 * 1 * 3))()
    # the down projection's CTAs have two or three items: one slot is too few
    assert f(2048, 2560, 6912, 148, plan, counts, items, 1) == blt.BL_ERR_INVALID_ARG
    assert max(counts) >= 2
    assert b"max_items" in blt.lib.bitlinear_last_error()
