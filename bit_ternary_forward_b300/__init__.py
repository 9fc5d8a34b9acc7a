"""B300-native BitLinear W1.58A8 forward.

A thin ctypes binding over ``libbitlinear.so`` (the C ABI declared in
``include/bitlinear.h``). Every step of the computation runs in the library's
CUDA kernels; this module only checks tensor types and passes pointers,
sizes and the current CUDA stream. PyTorch provides device memory and streams.

    packed = pack_weights(W)            # W: fp32 [N][K] on the GPU
    y = forward(x, packed)              # x: bf16 or fp32 [M][K] -> fp32 [M][N]

There is no CPU fallback: importing this package fails if the library has
not been built (``python bit_ternary_forward_b300/build.py``).
"""

from __future__ import annotations

import ctypes
import os
from typing import NamedTuple, Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbitlinear.so")

BL_OK, BL_ERR_INVALID_ARG, BL_ERR_UNSUPPORTED, BL_ERR_CUDA, BL_ERR_WORKSPACE = range(5)
BL_F32, BL_BF16 = 0, 1
#: weight quantisers of bitlinear_pack_weights_quantizer (bl_quantizer)
QUANTIZERS = {"absmean": 0, "alpha_round": 1, "threshold": 2}


class BitLinearError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed with status {status}: {msg}")
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python bit_ternary_forward_b300/build.py`")
    lib = ctypes.CDLL(LIB_PATH)
    i64, vp, sz = ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
    st = ctypes.c_int
    sig = {
        "bitlinear_pack_workspace_bytes": (sz, [i64, i64]),
        "bitlinear_pack_weights": (st, [vp, i64, i64, vp, vp, vp, sz, vp]),
        "bitlinear_pack_weights_noalloc": (st, [vp, i64, i64, vp, vp, vp]),
        "bitlinear_pack_weights_quantizer": (st, [vp, i64, i64, ctypes.c_int, ctypes.c_float, vp, vp, vp, sz, vp]),
        "bitlinear_absmean": (st, [vp, i64, i64, vp, vp, sz, vp]),
        "bitlinear_quantize_pack": (st, [vp, i64, i64, vp, vp, vp]),
        "bitlinear_gemm_workspace_bytes": (sz, [i64, i64, i64]),
        "bitlinear_gemm": (st, [vp, vp, i64, vp, vp, i64, i64, vp, vp, sz, vp]),
        "bitlinear_quant_act": (st, [vp, ctypes.c_int, i64, i64, vp, vp, vp]),
        "bitlinear_forward_workspace_bytes": (sz, [i64, i64, i64]),
        "bitlinear_forward": (st, [vp, ctypes.c_int, i64, vp, vp, i64, i64, vp, vp, vp, vp, sz, vp]),
        "bitlinear_gemm_i32_workspace_bytes": (sz, [i64, i64, i64]),
        "bitlinear_gemm_i32": (st, [vp, vp, i64, i64, i64, vp, vp, sz, vp]),
        "bitlinear_strerror": (ctypes.c_char_p, [st]),
        "bitlinear_last_error": (ctypes.c_char_p, []),
        "bitlinear_version": (ctypes.c_int, []),
        "bitlinear_device_error": (st, [ctypes.POINTER(ctypes.c_int)]),
        "bitlinear_tc_schedule": (st, [i64, i64, i64, ctypes.c_int, vp, vp, vp, ctypes.c_int]),
        "bitlinear_forward_lut": (st, [vp, ctypes.c_int, i64, vp, vp, i64, i64, vp, vp]),
        "bitlinear_pack_weights_grouped": (st, [vp, i64, i64, vp, vp, vp]),
        "bitlinear_forward_grouped_workspace_bytes": (sz, [i64, i64, i64]),
        "bitlinear_forward_grouped": (st, [vp, ctypes.c_int, i64, vp, vp, i64, i64, vp, vp, vp, vp, sz, vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


lib = _load()


def _check(fn: str, status: int) -> None:
    if status != BL_OK:
        detail = lib.bitlinear_last_error().decode() or lib.bitlinear_strerror(status).decode()
        raise BitLinearError(fn, status, detail)


def _stream(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _cuda(t: torch.Tensor, name: str, dtype=None) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _same_device(t: torch.Tensor, name: str, device: torch.device) -> torch.Tensor:
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    return t


def _out(t: torch.Tensor, name: str, dtype, shape, device: torch.device) -> torch.Tensor:
    """A caller-provided output: checked before the library writes shape-many elements into it."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return _same_device(t, name, device)


def _workspace(nbytes: int, device, ws: Optional[torch.Tensor]):
    """(holder, base, nbytes): a 256-byte aligned region; keep `holder` alive across the call."""
    if nbytes == 0:
        return None, 0, 0
    if ws is None:
        # 256 extra bytes so the base can be rounded up to a 256-byte boundary
        ws = torch.empty(nbytes + 256, dtype=torch.uint8, device=device)
    elif ws.device != torch.device(device) or not ws.is_contiguous():
        raise ValueError(f"workspace must be a contiguous tensor on {device}")
    p = ws.data_ptr()
    base = (p + 255) // 256 * 256
    if base + nbytes > p + ws.numel() * ws.element_size():
        raise ValueError("workspace tensor too small")
    return ws, base, nbytes


class PackedWeight(NamedTuple):
    """Packed ternary weights: wp uint8 [N][K/4] and gamma fp32 [1], on the GPU."""

    wp: torch.Tensor
    gamma: torch.Tensor
    n: int
    k: int


def pack_workspace_bytes(n: int, k: int) -> int:
    return int(lib.bitlinear_pack_workspace_bytes(n, k))


def forward_workspace_bytes(m: int, n: int, k: int) -> int:
    return int(lib.bitlinear_forward_workspace_bytes(m, n, k))


def pack_weights(w: torch.Tensor, out: Optional[PackedWeight] = None,
                 workspace: Optional[torch.Tensor] = None, quantizer: str = "absmean",
                 factor: float = 0.7) -> PackedWeight:
    """Ternary quantisation and 2-bit packing of fp32 weights [N][K].

    quantizer: "absmean" (the default rule; factor unused), "alpha_round" or
    "threshold" (bitlinear_pack_weights_quantizer); the returned scale (the
    PackedWeight's gamma) is what the forward multiplies by.
    """
    _cuda(w, "W", torch.float32)
    if w.dim() != 2:
        raise ValueError("W must be 2-D [N][K]")
    if quantizer not in QUANTIZERS:
        raise ValueError(f"unknown quantizer {quantizer!r}; expected one of {sorted(QUANTIZERS)}")
    n, k = w.shape
    if out is None:
        out = PackedWeight(torch.empty((n, k // 4), dtype=torch.uint8, device=w.device),
                           torch.empty(1, dtype=torch.float32, device=w.device), n, k)
    else:
        _out(out.wp, "out.wp", torch.uint8, (n, k // 4), w.device)
        _out(out.gamma, "out.gamma", torch.float32, (1,), w.device)
    hold, ws, wsn = _workspace(pack_workspace_bytes(n, k), w.device, workspace)
    if quantizer == "absmean":
        _check("bitlinear_pack_weights",
               lib.bitlinear_pack_weights(w.data_ptr(), n, k, out.wp.data_ptr(), out.gamma.data_ptr(),
                                          ws, wsn, _stream(w.device)))
    else:
        _check("bitlinear_pack_weights_quantizer",
               lib.bitlinear_pack_weights_quantizer(w.data_ptr(), n, k, QUANTIZERS[quantizer], float(factor),
                                                    out.wp.data_ptr(), out.gamma.data_ptr(), ws, wsn,
                                                    _stream(w.device)))
    return out


def absmean(w: torch.Tensor, gamma: Optional[torch.Tensor] = None,
            workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """gamma = mean(|W|) as fp32 [1] (exact sum, one rounding)."""
    _cuda(w, "W", torch.float32)
    n, k = w.shape
    if gamma is None:
        gamma = torch.empty(1, dtype=torch.float32, device=w.device)
    else:
        _out(gamma, "gamma", torch.float32, (1,), w.device)
    hold, ws, wsn = _workspace(pack_workspace_bytes(n, k), w.device, workspace)
    _check("bitlinear_absmean", lib.bitlinear_absmean(w.data_ptr(), n, k, gamma.data_ptr(), ws, wsn,
                                                      _stream(w.device)))
    return gamma


def quantize_pack(w: torch.Tensor, gamma: torch.Tensor, wp: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Ternary codes of W against a given gamma, packed four per byte: uint8 [N][K/4]."""
    _cuda(w, "W", torch.float32)
    _same_device(_cuda(gamma, "gamma", torch.float32), "gamma", w.device)
    n, k = w.shape
    if wp is None:
        wp = torch.empty((n, k // 4), dtype=torch.uint8, device=w.device)
    else:
        _out(wp, "wp", torch.uint8, (n, k // 4), w.device)
    _check("bitlinear_quantize_pack", lib.bitlinear_quantize_pack(w.data_ptr(), n, k, gamma.data_ptr(),
                                                                  wp.data_ptr(), _stream(w.device)))
    return wp


def gemm(xq: torch.Tensor, scale: torch.Tensor, packed: PackedWeight, y: Optional[torch.Tensor] = None,
         workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """y = (x_q . codes^T) * gamma / s on already-quantised activations."""
    _cuda(xq, "xq", torch.int8)
    m, k = xq.shape
    if k != packed.k:
        raise ValueError(f"xq must be [M][{packed.k}]")
    n = packed.n
    _out(_cuda(scale, "scale", torch.float32), "scale", torch.float32, (m,), xq.device)
    _same_device(packed.wp, "packed.wp", xq.device)
    _same_device(packed.gamma, "packed.gamma", xq.device)
    if y is None:
        y = torch.empty((m, n), dtype=torch.float32, device=xq.device)
    else:
        _out(y, "y", torch.float32, (m, n), xq.device)
    hold, ws, wsn = _workspace(int(lib.bitlinear_gemm_workspace_bytes(m, n, k)), xq.device, workspace)
    _check("bitlinear_gemm", lib.bitlinear_gemm(xq.data_ptr(), scale.data_ptr(), m, packed.wp.data_ptr(),
                                                packed.gamma.data_ptr(), n, k, y.data_ptr(), ws, wsn,
                                                _stream(xq.device)))
    return y


def _dtype_code(x: torch.Tensor) -> int:
    if x.dtype == torch.bfloat16:
        return BL_BF16
    if x.dtype == torch.float32:
        return BL_F32
    raise TypeError(f"activations must be bf16 or fp32, got {x.dtype}")


def quant_act(x: torch.Tensor, xq: Optional[torch.Tensor] = None,
              scale: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Per-token absmax int8 quantisation; returns (x_q int8 [M][K], s fp32 [M])."""
    _cuda(x, "x")
    m, k = x.shape
    if xq is None:
        xq = torch.empty((m, k), dtype=torch.int8, device=x.device)
    else:
        _out(xq, "xq", torch.int8, (m, k), x.device)
    if scale is None:
        scale = torch.empty(m, dtype=torch.float32, device=x.device)
    else:
        _out(scale, "scale", torch.float32, (m,), x.device)
    _check("bitlinear_quant_act",
           lib.bitlinear_quant_act(x.data_ptr(), _dtype_code(x), m, k, xq.data_ptr(), scale.data_ptr(),
                                   _stream(x.device)))
    return xq, scale


def forward(x: torch.Tensor, packed: PackedWeight, y: Optional[torch.Tensor] = None,
            return_quant: bool = False, workspace: Optional[torch.Tensor] = None):
    """y = BitLinear(x) = (x_q . codes^T) * gamma / s; fp32 [M][N]."""
    _cuda(x, "x")
    if x.dim() != 2 or x.shape[1] != packed.k:
        raise ValueError(f"x must be [M][{packed.k}]")
    m, k = x.shape
    n = packed.n
    _same_device(packed.wp, "packed.wp", x.device)
    _same_device(packed.gamma, "packed.gamma", x.device)
    if y is None:
        y = torch.empty((m, n), dtype=torch.float32, device=x.device)
    else:
        _out(y, "y", torch.float32, (m, n), x.device)
    xq = scale = None
    if return_quant:
        xq = torch.empty((m, k), dtype=torch.int8, device=x.device)
        scale = torch.empty(m, dtype=torch.float32, device=x.device)
    hold, ws, wsn = _workspace(forward_workspace_bytes(m, n, k), x.device, workspace)
    _check("bitlinear_forward",
           lib.bitlinear_forward(x.data_ptr(), _dtype_code(x), m, packed.wp.data_ptr(), packed.gamma.data_ptr(),
                                 n, k, y.data_ptr(), xq.data_ptr() if xq is not None else None,
                                 scale.data_ptr() if scale is not None else None, ws, wsn, _stream(x.device)))
    return (y, xq, scale) if return_quant else y


def forward_lut(x: torch.Tensor, packed: PackedWeight, y: Optional[torch.Tensor] = None) -> torch.Tensor:
    """The one-token forward by table lookup (bitlinear_forward_lut); same y as forward, bit for bit."""
    _cuda(x, "x")
    if x.dim() != 2 or x.shape[1] != packed.k:
        raise ValueError(f"x must be [1][{packed.k}]")
    m, k = x.shape
    n = packed.n
    _same_device(packed.wp, "packed.wp", x.device)
    _same_device(packed.gamma, "packed.gamma", x.device)
    if y is None:
        y = torch.empty((m, n), dtype=torch.float32, device=x.device)
    else:
        _out(y, "y", torch.float32, (m, n), x.device)
    _check("bitlinear_forward_lut",
           lib.bitlinear_forward_lut(x.data_ptr(), _dtype_code(x), m, packed.wp.data_ptr(), packed.gamma.data_ptr(),
                                     n, k, y.data_ptr(), _stream(x.device)))
    return y


class PackedGrouped(NamedTuple):
    """Per-group (64) packed ternary weights: wp uint8 [N][K/4] and gammas fp32 [N][K/64]."""

    wp: torch.Tensor
    gammas: torch.Tensor
    n: int
    k: int


def pack_weights_grouped(w: torch.Tensor, out: Optional[PackedGrouped] = None) -> PackedGrouped:
    """Per-group absmean quantisation (groups of 64 consecutive k of a row) and 2-bit packing."""
    _cuda(w, "W", torch.float32)
    if w.dim() != 2:
        raise ValueError("W must be 2-D [N][K]")
    n, k = w.shape
    if out is None:
        out = PackedGrouped(torch.empty((n, k // 4), dtype=torch.uint8, device=w.device),
                            torch.empty((n, k // 64), dtype=torch.float32, device=w.device), n, k)
    else:
        _out(out.wp, "out.wp", torch.uint8, (n, k // 4), w.device)
        _out(out.gammas, "out.gammas", torch.float32, (n, k // 64), w.device)
    _check("bitlinear_pack_weights_grouped",
           lib.bitlinear_pack_weights_grouped(w.data_ptr(), n, k, out.wp.data_ptr(), out.gammas.data_ptr(),
                                              _stream(w.device)))
    return out


def forward_grouped(x: torch.Tensor, packed: PackedGrouped, y: Optional[torch.Tensor] = None,
                    return_quant: bool = False, workspace: Optional[torch.Tensor] = None):
    """y[m][n] = sum_g gammas[n][g] * acc[m][n][g] / s_m over per-group scales; fp32 [M][N]."""
    _cuda(x, "x")
    if x.dim() != 2 or x.shape[1] != packed.k:
        raise ValueError(f"x must be [M][{packed.k}]")
    m, k = x.shape
    n = packed.n
    _same_device(packed.wp, "packed.wp", x.device)
    _same_device(packed.gammas, "packed.gammas", x.device)
    if y is None:
        y = torch.empty((m, n), dtype=torch.float32, device=x.device)
    else:
        _out(y, "y", torch.float32, (m, n), x.device)
    xq = scale = None
    if return_quant:
        xq = torch.empty((m, k), dtype=torch.int8, device=x.device)
        scale = torch.empty(m, dtype=torch.float32, device=x.device)
    hold, ws, wsn = _workspace(int(lib.bitlinear_forward_grouped_workspace_bytes(m, n, k)), x.device, workspace)
    _check("bitlinear_forward_grouped",
           lib.bitlinear_forward_grouped(x.data_ptr(), _dtype_code(x), m, packed.wp.data_ptr(),
                                         packed.gammas.data_ptr(), n, k, y.data_ptr(),
                                         xq.data_ptr() if xq is not None else None,
                                         scale.data_ptr() if scale is not None else None, ws, wsn,
                                         _stream(x.device)))
    return (y, xq, scale) if return_quant else y


def gemm_i32(xq: torch.Tensor, wp: torch.Tensor, acc: Optional[torch.Tensor] = None) -> torch.Tensor:
    """acc[m][n] = sum_k code[n][k] * xq[m][k] as exact int32."""
    _cuda(xq, "xq", torch.int8)
    _cuda(wp, "wp", torch.uint8)
    m, k = xq.shape
    n = wp.shape[0]
    if wp.dim() != 2 or wp.shape[1] * 4 != k:
        raise ValueError("wp must be [N][K/4]")
    _same_device(wp, "wp", xq.device)
    if acc is None:
        acc = torch.empty((m, n), dtype=torch.int32, device=xq.device)
    else:
        _out(acc, "acc", torch.int32, (m, n), xq.device)
    wsn_req = int(lib.bitlinear_gemm_i32_workspace_bytes(m, n, k))
    hold, ws, wsn = _workspace(wsn_req, xq.device, None)
    _check("bitlinear_gemm_i32",
           lib.bitlinear_gemm_i32(xq.data_ptr(), wp.data_ptr(), m, n, k, acc.data_ptr(), ws, wsn,
                                  _stream(xq.device)))
    return acc


def device_error() -> int:
    """The device-side error word (non-zero: a kernel gave up a bounded wait); reading clears it."""
    flag = ctypes.c_int(0)
    _check("bitlinear_device_error", lib.bitlinear_device_error(ctypes.byref(flag)))
    return int(flag.value)


class TcPlan(NamedTuple):
    """Launch plan of the tensor-core contraction (see bitlinear_tc_schedule)."""

    bn: int            # tokens per tile
    grid: int          # CTAs
    row_tiles: int     # tiles along the weight rows, ceil(N / 128)
    k_iters: int       # k-stages of 64 per tile
    dp_tiles: int      # tiles computed whole
    sk_tiles: int      # tiles split by k-stages
    sk_ctas: int       # CTAs that take a run of split stages
    token_tiles: int   # ceil(M / bn)
    sk_bytes: int      # split-tile buffer and counters in the workspace


def tc_schedule(M: int, N: int, K: int, sms: int):
    """(plan, items): the tensor-core contraction's plan for M x N x K on `sms`
    SMs and, per CTA, its work items (tile, k0, k1) in execution order. Host
    arithmetic in the library; no GPU is needed."""
    plan = (ctypes.c_int32 * 9)()
    _check("bitlinear_tc_schedule", lib.bitlinear_tc_schedule(M, N, K, sms, plan, None, None, 0))
    p = TcPlan(*plan)
    counts = (ctypes.c_int32 * p.grid)()
    _check("bitlinear_tc_schedule", lib.bitlinear_tc_schedule(M, N, K, sms, plan, counts, None, 0))
    most = max(counts) if p.grid else 0
    buf = (ctypes.c_int32 * (p.grid * most * 3))()
    _check("bitlinear_tc_schedule", lib.bitlinear_tc_schedule(M, N, K, sms, plan, counts, buf, most))
    items = [[tuple(buf[(b * most + i) * 3:(b * most + i) * 3 + 3]) for i in range(counts[b])] for b in range(p.grid)]
    return p, items


__all__ = ["device_error", "PackedWeight", "BitLinearError", "pack_weights", "absmean", "quantize_pack", "quant_act", "forward",
           "gemm", "gemm_i32", "forward_lut", "PackedGrouped", "pack_weights_grouped", "forward_grouped",
           "pack_workspace_bytes", "forward_workspace_bytes", "tc_schedule", "TcPlan", "lib", "LIB_PATH"]
