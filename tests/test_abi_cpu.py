"""The C-ABI library without a GPU: it loads, exports every declared symbol,
reports its constants, and rejects bad arguments on the host before any CUDA
call is made."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bitlinear.h")


@pytest.fixture(scope="module")
def blt():
    import importlib.util
    spec = importlib.util.spec_from_file_location("bl_build", os.path.join(ROOT, "bit_ternary_forward_b300", "build.py"))
    build = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(build)
    build.build()
    import bit_ternary_forward_b300 as b
    return b


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(bitlinear_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("bitlinear_pack_weights", "bitlinear_quant_act", "bitlinear_forward", "bitlinear_gemm_i32"):
        assert must in names


def test_library_exports_every_declared_symbol(blt):
    lib = ctypes.CDLL(blt.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_library_exports_nothing_else(blt):
    # the C ABI is the only public surface (kernels and helpers are hidden)
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", blt.LIB_PATH], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    ours = {n for n in exported if n.startswith("bitlinear_")}
    assert ours == set(declared_functions())


def test_constants(blt):
    lib = blt.lib
    assert lib.bitlinear_version() == 1
    assert lib.bitlinear_strerror(0) == b"ok"
    assert b"invalid" in lib.bitlinear_strerror(1)
    assert lib.bitlinear_pack_workspace_bytes(6912, 2560) >= 64 * 148
    # the one-kernel decode GEMV (M <= 4, K % 64 == 0) needs no workspace; the
    # two-kernel forms keep the codes there
    assert lib.bitlinear_forward_workspace_bytes(4, 256, 256) == 0
    assert lib.bitlinear_forward_workspace_bytes(4, 256, 260) >= 4 * 260
    assert lib.bitlinear_forward_workspace_bytes(8, 256, 256) >= 8 * 256
    assert lib.bitlinear_forward_workspace_bytes(0, 256, 256) == 0


@pytest.mark.parametrize("n,k", [(0, 256), (8, 0), (8, 6), (8, 70000), (1 << 20, 1 << 12)])
def test_pack_rejects_bad_dims_on_host(blt, n, k):
    lib = blt.lib
    st = lib.bitlinear_pack_weights(16, n, k, 16, 16, 256, 1 << 20, None)
    assert st in (blt.BL_ERR_INVALID_ARG, blt.BL_ERR_UNSUPPORTED)
    assert lib.bitlinear_last_error()


def test_pack_rejects_null_misaligned_and_workspace(blt):
    lib = blt.lib
    ws = lib.bitlinear_pack_workspace_bytes(64, 64)
    assert lib.bitlinear_pack_weights(None, 64, 64, 16, 16, 256, ws, None) == blt.BL_ERR_INVALID_ARG
    assert lib.bitlinear_pack_weights(8, 64, 64, 16, 16, 256, ws, None) == blt.BL_ERR_INVALID_ARG      # W misaligned
    assert lib.bitlinear_pack_weights(16, 64, 64, 16, 16, None, ws, None) == blt.BL_ERR_WORKSPACE
    assert lib.bitlinear_pack_weights(16, 64, 64, 16, 16, 128, ws, None) == blt.BL_ERR_WORKSPACE       # not 256-aligned
    assert lib.bitlinear_pack_weights(16, 64, 64, 16, 16, 256, ws - 1, None) == blt.BL_ERR_WORKSPACE


def test_pack_quantizer_rejects_bad_args_on_host(blt):
    lib = blt.lib
    ws = lib.bitlinear_pack_workspace_bytes(64, 64)
    f = lib.bitlinear_pack_weights_quantizer
    assert f(16, 64, 64, 3, 0.7, 16, 16, 256, ws, None) == blt.BL_ERR_INVALID_ARG        # unknown quantizer
    assert f(16, 64, 64, -1, 0.7, 16, 16, 256, ws, None) == blt.BL_ERR_INVALID_ARG
    for bad in (0.0, -0.7, float("inf"), float("nan")):
        assert f(16, 64, 64, 1, bad, 16, 16, 256, ws, None) == blt.BL_ERR_INVALID_ARG     # factor
        assert f(16, 64, 64, 2, bad, 16, 16, 256, ws, None) == blt.BL_ERR_INVALID_ARG
    assert f(16, 64, 64, 2, 0.7, None, 16, 256, ws, None) == blt.BL_ERR_INVALID_ARG       # Wp
    assert f(16, 64, 64, 2, 0.7, 16, None, 256, ws, None) == blt.BL_ERR_INVALID_ARG       # scale
    assert f(16, 64, 62, 2, 0.7, 16, 16, 256, ws, None) == blt.BL_ERR_INVALID_ARG         # K % 4
    assert f(16, 64, 64, 2, 0.7, 16, 16, 256, ws - 1, None) == blt.BL_ERR_WORKSPACE
    assert blt.QUANTIZERS == {"absmean": 0, "alpha_round": 1, "threshold": 2}


def test_forward_and_quant_reject_bad_args_on_host(blt):
    lib = blt.lib
    ws = lib.bitlinear_forward_workspace_bytes(4, 64, 64)
    assert lib.bitlinear_forward(16, 7, 4, 16, 16, 64, 64, 16, None, None, 256, ws, None) == blt.BL_ERR_INVALID_ARG
    assert lib.bitlinear_forward(16, 1, 0, 16, 16, 64, 64, 16, None, None, 256, ws, None) == blt.BL_ERR_INVALID_ARG
    assert lib.bitlinear_forward(16, 1, 4, 16, 16, 64, 62, 16, None, None, 256, ws, None) == blt.BL_ERR_INVALID_ARG
    assert lib.bitlinear_forward(16, 1, 4, 16, 16, 64, 64, 24, None, None, 256, ws, None) == blt.BL_ERR_INVALID_ARG
    assert lib.bitlinear_forward(16, 1, 4, 16, 16, 64, 64, 16, 8, None, 256, ws, None) == blt.BL_ERR_INVALID_ARG
    ws68 = lib.bitlinear_forward_workspace_bytes(4, 64, 68)     # K % 64 != 0: the two-kernel path keeps codes there
    assert ws68 > 0
    assert lib.bitlinear_forward(16, 1, 4, 16, 16, 64, 68, 16, None, None, None, ws68, None) == blt.BL_ERR_WORKSPACE
    assert lib.bitlinear_quant_act(16, 1, 4, 6, 16, 16, None) == blt.BL_ERR_INVALID_ARG
    assert lib.bitlinear_quant_act(None, 1, 4, 8, 16, 16, None) == blt.BL_ERR_INVALID_ARG
    assert lib.bitlinear_gemm_i32(16, 16, 4, 4, 6, 16, None, 0, None) == blt.BL_ERR_INVALID_ARG
    assert lib.bitlinear_gemm_i32(16, 16, 4, 4, 8, 20, None, 0, None) == blt.BL_ERR_INVALID_ARG


def test_python_binding_rejects_cpu_tensors(blt):
    import torch
    with pytest.raises(TypeError):
        blt.pack_weights(torch.zeros(4, 4))
    with pytest.raises(TypeError):
        blt.quant_act(torch.zeros(4, 4))


def test_python_binding_checks_caller_outputs(blt):
    # the binding checks every caller-provided output before the library
    # writes into it (the checks use no CUDA call, so CPU tensors show them)
    import torch
    cpu = torch.device("cpu")
    ok = torch.empty((4, 8), dtype=torch.float32)
    assert blt._out(ok, "y", torch.float32, (4, 8), cpu) is ok
    with pytest.raises(TypeError):
        blt._out(ok, "y", torch.int32, (4, 8), cpu)                       # dtype
    with pytest.raises(ValueError):
        blt._out(ok, "y", torch.float32, (4, 9), cpu)                     # shape
    with pytest.raises(ValueError):
        blt._out(ok.t(), "y", torch.float32, (8, 4), cpu)                 # not contiguous
    with pytest.raises(ValueError):
        blt._out(ok, "y", torch.float32, (4, 8), torch.device("cuda", 0))  # another device
    with pytest.raises(TypeError):
        blt._out(None, "y", torch.float32, (4, 8), cpu)


def test_python_binding_checks_the_workspace(blt):
    import torch
    cpu = torch.device("cpu")
    assert blt._workspace(0, cpu, None) == (None, 0, 0)
    ws = torch.empty(1024 + 256, dtype=torch.uint8)
    hold, base, n = blt._workspace(1024, cpu, ws)
    assert hold is ws and base % 256 == 0 and n == 1024
    assert base + n <= ws.data_ptr() + ws.numel()
    wide = torch.empty(320, dtype=torch.float32)                         # 1280 bytes
    assert blt._workspace(1024, cpu, wide)[2] == 1024
    with pytest.raises(ValueError):
        blt._workspace(4096, cpu, ws)                                    # too small
    with pytest.raises(ValueError):
        blt._workspace(1024, torch.device("cuda", 0), ws)               # another device
