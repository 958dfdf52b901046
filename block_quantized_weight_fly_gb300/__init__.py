"""Python binding of libqmv: block-quantized weight GEMV on GB300 (sm_103a).

Argument marshalling only. Every function has the name of the C entry point it
calls (include/qmv.h), takes torch tensors for device buffers, passes their raw
pointers and the current CUDA stream, and raises QmvError on a non-zero status.
All arithmetic runs in the CUDA kernels of libqmv.so; there is no fallback: if
the library has not been built, importing this package raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqmv.so")

QMV_Q8_0, QMV_Q4_K, QMV_Q6_K, QMV_NVFP4, QMV_FP8_ROW, QMV_Q5_K = 1, 2, 3, 4, 5, 6
QMV_IQ4_XS, QMV_IQ3_S, QMV_IQ2_S = 7, 8, 9
FORMATS = {"q8_0": QMV_Q8_0, "q4_k": QMV_Q4_K, "q6_k": QMV_Q6_K, "nvfp4": QMV_NVFP4,
           "fp8_row": QMV_FP8_ROW, "q5_k": QMV_Q5_K, "iq4_xs": QMV_IQ4_XS, "iq3_s": QMV_IQ3_S,
           "iq2_s": QMV_IQ2_S}
GRID_BYTES = {"iq3_s": 512 * 4, "iq2_s": 1024 * 8}
QMV_ENTRY_GEMV, QMV_ENTRY_GROUPED, QMV_ENTRY_W4A4, QMV_ENTRY_SWIGLU = 1, 2, 3, 4
QMV_ENTRY_GROUPED_SWIGLU, QMV_ENTRY_KQUANT, QMV_ENTRY_MLP_LAYER, QMV_ENTRY_INT8DOT = 5, 6, 7, 8
QMV_MAX_M = 8

STATUS = {0: "QMV_OK", 1: "QMV_EINVAL", 2: "QMV_EALIGN", 3: "QMV_EUNSUPPORTED", 4: "QMV_ECUDA",
          5: "QMV_EHEADER", 6: "QMV_ETIMEOUT", 7: "QMV_ERANGE", 8: "QMV_EWORKSPACE"}


class QmvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)} ({qmv_status_str(status)})")


if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with "
                      f"`python block_quantized_weight_fly_gb300/build.py` (no CPU fallback exists)")

_lib = ctypes.CDLL(LIB_PATH)
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_F = ctypes.c_float


def _sig(name, res, args):
    f = getattr(_lib, name)
    f.restype = res
    f.argtypes = args
    return f


_canon_size = _sig("qmv_canon_size", _SZ, [_I, _I64, _I64, _I64])
_pack_size = _sig("qmv_pack_size", _SZ, [_I, _I64, _I64, _I64])
_pack = _sig("qmv_pack", _I, [_I, _P, _I64, _I64, _I64, _P, _P])
_quantize = _sig("qmv_quantize", _I, [_I, _P, _I64, _I64, _F, _P, _P])
_quantize_cb = _sig("qmv_quantize_codebook", _I, [_I, _P, _I64, _I64, _P, _P, _P])
_dequant = _sig("qmv_dequant", _I, [_I, _P, _I64, _I64, _I64, _I64, _I64, _P, _P])
_ws_size = _sig("qmv_workspace_size", _SZ, [_I, _I, _I, _I64, _I64, _I64, _I])
_gemv = _sig("qmv_gemv", _I, [_I, _P, _P, _P, _I, _I64, _I64, _P, _SZ, _P])
_gemv_swiglu = _sig("qmv_gemv_swiglu", _I, [_I, _P, _P, _P, _I, _I64, _I64, _P, _SZ, _P])
_gemv_noalloc = _sig("qmv_gemv_noalloc", _I, [_I, _P, _P, _P, _I, _I64, _I64, _P])
_grouped = _sig("qmv_grouped", _I, [_I, _P, _P, _P, _I, _P, _I, _I, _I64, _I64, _I64, _P, _SZ, _P])
_mlp_layer = _sig("qmv_mlp_layer", _I, [_I, _P, _P, _P, _P, _I, _I64, _I64, _P, _SZ, _P])
_grouped_swiglu = _sig("qmv_grouped_swiglu", _I, [_I, _P, _P, _P, _P, _I, _I, _I64, _I64, _I64, _P, _SZ, _P])
_quant_act = _sig("qmv_quant_act_nvfp4", _I, [_P, _F, _P, _P, _I, _I64, _P])
_w4a4 = _sig("qmv_gemm_nvfp4_w4a4", _I, [_P, _P, _F, _P, _I, _I64, _I64, _P, _SZ, _P])
_kquant = _sig("qmv_gemm_kquant", _I, [_I, _P, _P, _P, _I, _I64, _I64, _P, _SZ, _P])
_int8dot = _sig("qmv_gemv_int8dot", _I, [_I, _P, _P, _P, _I, _I64, _I64, _P, _SZ, _P])
_status_str = _sig("qmv_status_str", ctypes.c_char_p, [_I])
_last_route = _sig("qmv_last_route", _I, [])
_dev_status = _sig("qmv_device_status", _I, [_I])
_split_fault = _sig("qmv_debug_split_k_fault", None, [_I, ctypes.c_uint64])

EXPORTED = ["qmv_canon_size", "qmv_pack_size", "qmv_pack", "qmv_quantize", "qmv_dequant",
            "qmv_workspace_size", "qmv_gemv", "qmv_grouped", "qmv_quant_act_nvfp4",
            "qmv_gemm_nvfp4_w4a4", "qmv_status_str", "qmv_last_route", "qmv_device_status",
            "qmv_gemv_noalloc", "qmv_gemv_swiglu", "qmv_grouped_swiglu", "qmv_gemm_kquant",
            "qmv_debug_split_k_fault", "qmv_quantize_codebook", "qmv_mlp_layer", "qmv_gemv_int8dot"]


def _fmt(fmt) -> int:
    return FORMATS[fmt] if isinstance(fmt, str) else int(fmt)


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _dev(t: torch.Tensor, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(st: int, what: str):
    if st != 0:
        raise QmvError(st, what)


def _bits16(x: torch.Tensor) -> torch.Tensor:
    if x.dtype == torch.bfloat16:
        return x
    if x.dtype in (torch.int16, torch.uint16):
        return x
    raise ValueError("x must be bf16 (or its raw 16-bit patterns)")


def _act(x: torch.Tensor, K: int, rows: int | None = None) -> tuple[torch.Tensor, int]:
    """Check an activation tensor [M, K] (or [K]) and return it with its row count.
    The library reads M * K values through a raw pointer, so a short or strided x
    is refused here rather than read out of bounds on the device."""
    x = _bits16(x)
    if not x.is_contiguous():
        raise ValueError("x must be contiguous")
    if x.dim() == 1:
        M = 1
        if x.shape[0] != K:
            raise ValueError(f"x has {x.shape[0]} values, K = {K}")
    elif x.dim() == 2:
        M = x.shape[0]
        if x.shape[1] != K:
            raise ValueError(f"x has rows of {x.shape[1]} values, K = {K}")
    else:
        raise ValueError("x must be [M, K] or [K]")
    if rows is not None and M != rows:
        raise ValueError(f"x has {M} rows, {rows} expected")
    return x, M


def _out(y: torch.Tensor | None, shape, dev, name: str) -> torch.Tensor:
    """An fp32 output of `shape`: allocated if None, else checked (float32, contiguous,
    on x's device, at least as many values as the library writes)."""
    if y is None:
        return torch.empty(shape, dtype=torch.float32, device=dev)
    if not y.is_cuda or y.device != torch.device(dev):
        raise ValueError(f"{name} must be a CUDA tensor on {dev}")
    if y.dtype != torch.float32:
        raise ValueError(f"{name} must be float32")
    if not y.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    need = 1
    for d in shape:
        need *= int(d)
    if y.numel() < need:
        raise ValueError(f"{name} holds {y.numel()} values, {need} needed")
    return y


# ---- entry points -------------------------------------------------------------
def qmv_status_str(status: int) -> str:
    return _status_str(int(status)).decode()


def qmv_last_route() -> int:
    return int(_last_route())


def qmv_device_status(reset: bool = True) -> int:
    return int(_dev_status(1 if reset else 0))


def qmv_debug_split_k_fault(mode: int, wait_limit_ns: int = 0) -> None:
    """Test hook of the split-K reduction (include/qmv.h): mode 1, peers publish
    nothing and reducers time out after wait_limit_ns; mode 2, reducers give up at
    once and leave their peers' partial sums behind; mode 0, normal operation."""
    _split_fault(int(mode), int(wait_limit_ns))


def qmv_canon_size(fmt, N: int, K: int, E: int = 1) -> int:
    return int(_canon_size(_fmt(fmt), N, K, E))


def qmv_pack_size(fmt, N: int, K: int, E: int = 1) -> int:
    return int(_pack_size(_fmt(fmt), N, K, E))


def qmv_workspace_size(entry: int, fmt, M: int, N: int, K: int, E: int = 1, topk: int = 1) -> int:
    return int(_ws_size(int(entry), _fmt(fmt), M, N, K, E, topk))


def qmv_pack(fmt, canon: torch.Tensor, N: int, K: int, E: int = 1, dst: torch.Tensor | None = None,
             stream=None) -> torch.Tensor:
    _dev(canon, "canon")
    size = qmv_pack_size(fmt, N, K, E)
    if size == 0:
        raise QmvError(3, "qmv_pack_size")
    if canon.numel() * canon.element_size() < qmv_canon_size(fmt, N, K, E):
        raise ValueError("canon is shorter than qmv_canon_size")
    if dst is None:
        dst = torch.empty(size, dtype=torch.uint8, device=canon.device)
    elif not dst.is_cuda or not dst.is_contiguous() or dst.numel() * dst.element_size() < size:
        raise ValueError(f"dst must be a contiguous CUDA tensor of at least {size} bytes")
    _check(_pack(_fmt(fmt), _ptr(canon), N, K, E, _ptr(dst), _stream(stream)), "qmv_pack")
    return dst


def qmv_quantize(fmt, W: torch.Tensor, tensor_scale: float = 0.0, canon: torch.Tensor | None = None,
                 stream=None) -> torch.Tensor:
    _dev(W, "W")
    if W.dtype != torch.float32 or W.dim() != 2:
        raise ValueError("W must be a 2-D float32 tensor")
    rows, K = W.shape
    size = qmv_canon_size(fmt, rows, K, 1)
    if not W.is_contiguous():
        raise ValueError("W must be contiguous")
    if canon is None:
        canon = torch.empty(size, dtype=torch.uint8, device=W.device)
    elif not canon.is_cuda or not canon.is_contiguous() or canon.numel() * canon.element_size() < size:
        raise ValueError(f"canon must be a contiguous CUDA tensor of at least {size} bytes")
    _check(_quantize(_fmt(fmt), _ptr(W), rows, K, float(tensor_scale), _ptr(canon), _stream(stream)),
           "qmv_quantize")
    return canon


def qmv_quantize_codebook(fmt, W: torch.Tensor, codebook, canon: torch.Tensor | None = None,
                          stream=None) -> torch.Tensor:
    """The codebook formats' encoder: IQ4_XS takes 16 int8 values, IQ3_S / IQ2_S the
    grid (uint8 magnitudes, 512 x 4 / 1024 x 8) -- host sequences."""
    _dev(W, "W")
    if W.dtype != torch.float32 or W.dim() != 2 or not W.is_contiguous():
        raise ValueError("W must be a contiguous 2-D float32 tensor")
    name = fmt if isinstance(fmt, str) else next(k for k, v in FORMATS.items() if v == int(fmt))
    vals = [int(v) for v in (codebook.reshape(-1) if hasattr(codebook, "reshape") else codebook)]
    n = GRID_BYTES.get(name, 16)
    if len(vals) != n:
        raise ValueError(f"the {name} table holds {n} values")
    cb = (ctypes.c_int8 * 16)(*vals) if n == 16 else (ctypes.c_uint8 * n)(*vals)
    rows, K = W.shape
    size = qmv_canon_size(fmt, rows, K, 1)
    if canon is None:
        canon = torch.empty(size, dtype=torch.uint8, device=W.device)
    elif not canon.is_cuda or not canon.is_contiguous() or canon.numel() * canon.element_size() < size:
        raise ValueError(f"canon must be a contiguous CUDA tensor of at least {size} bytes")
    _check(_quantize_cb(_fmt(fmt), _ptr(W), rows, K, ctypes.cast(cb, ctypes.c_void_p), _ptr(canon),
                        _stream(stream)), "qmv_quantize_codebook")
    return canon


def qmv_dequant(fmt, packed: torch.Tensor, N: int, K: int, E: int = 1, row0: int = 0,
                rows: int | None = None, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    _dev(packed, "packed")
    rows = N * E - row0 if rows is None else rows
    out = _out(out, (rows, K), packed.device, "out")
    _check(_dequant(_fmt(fmt), _ptr(packed), N, K, E, row0, rows, _ptr(out), _stream(stream)),
           "qmv_dequant")
    return out


def workspace(entry: int, fmt, M: int, N: int, K: int, E: int = 1, topk: int = 1,
              device="cuda") -> torch.Tensor:
    """A zero-filled workspace of the size the entry point needs."""
    size = qmv_workspace_size(entry, fmt, M, N, K, E, topk)
    if size == 0:
        raise QmvError(1, "qmv_workspace_size")
    return torch.zeros(size, dtype=torch.uint8, device=device)


def qmv_gemv(fmt, packed_W: torch.Tensor, x: torch.Tensor, N: int, K: int,
             ws: torch.Tensor, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    _dev(packed_W, "packed_W"); _dev(x, "x"); _dev(ws, "ws")
    x, M = _act(x, K)
    y = _out(y, (M, N), x.device, "y")
    _check(_gemv(_fmt(fmt), _ptr(packed_W), _ptr(x), _ptr(y), M, N, K, _ptr(ws), ws.numel(),
                 _stream(stream)), "qmv_gemv")
    return y


def qmv_gemv_swiglu(fmt, tower: torch.Tensor, x: torch.Tensor, N: int, K: int, ws: torch.Tensor,
                    h: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """h = silu(gate . x) * (up . x) over a 2-expert tower (gate = expert 0, up = expert 1)."""
    _dev(tower, "tower"); _dev(x, "x"); _dev(ws, "ws")
    x, M = _act(x, K)
    h = _out(h, (M, N), x.device, "h")
    _check(_gemv_swiglu(_fmt(fmt), _ptr(tower), _ptr(x), _ptr(h), M, N, K, _ptr(ws), ws.numel(),
                        _stream(stream)), "qmv_gemv_swiglu")
    return h


def qmv_mlp_layer(fmt, gateup: torch.Tensor, down: torch.Tensor, x: torch.Tensor, N_ff: int, K_h: int,
                  ws: torch.Tensor, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y = bf16(silu(x Wg^T) * (x Wu^T)) Wd^T in one launch: gateup = the 2-matrix
    [N_ff, K_h] tower (gate, up), down = the [K_h, N_ff] matrix."""
    _dev(gateup, "gateup"); _dev(down, "down"); _dev(x, "x"); _dev(ws, "ws")
    x, M = _act(x, K_h)
    y = _out(y, (M, K_h), x.device, "y")
    _check(_mlp_layer(_fmt(fmt), _ptr(gateup), _ptr(down), _ptr(x), _ptr(y), M, N_ff, K_h, _ptr(ws), ws.numel(),
                      _stream(stream)), "qmv_mlp_layer")
    return y


def qmv_gemv_noalloc(fmt, packed_W: torch.Tensor, x: torch.Tensor, N: int, K: int,
                     y: torch.Tensor, stream=None) -> torch.Tensor:
    """qmv_gemv with the library's built-in scratch instead of a workspace. y is
    required (the caller owns every buffer); nothing is allocated."""
    _dev(packed_W, "packed_W"); _dev(x, "x"); _dev(y, "y")
    x, M = _act(x, K)
    y = _out(y, (M, N), x.device, "y")
    _check(_gemv_noalloc(_fmt(fmt), _ptr(packed_W), _ptr(x), _ptr(y), M, N, K, _stream(stream)),
           "qmv_gemv_noalloc")
    return y


def qmv_grouped(fmt, tower: torch.Tensor, expert_ids: torch.Tensor, x: torch.Tensor, N: int, K: int,
                E: int, ws: torch.Tensor, x_per_pair: bool = False, y: torch.Tensor | None = None,
                stream=None) -> torch.Tensor:
    _dev(tower, "tower"); _dev(expert_ids, "expert_ids"); _dev(x, "x"); _dev(ws, "ws")
    if expert_ids.dtype != torch.int32 or expert_ids.dim() != 2:
        raise ValueError("expert_ids must be int32 [M, topk]")
    if not expert_ids.is_contiguous():
        raise ValueError("expert_ids must be contiguous")
    M, topk = expert_ids.shape
    x, _ = _act(x, K, M * topk if x_per_pair else M)
    y = _out(y, (M, topk, N), x.device, "y")
    _check(_grouped(_fmt(fmt), _ptr(tower), _ptr(expert_ids), _ptr(x), 1 if x_per_pair else 0, _ptr(y),
                    M, topk, N, K, E, _ptr(ws), ws.numel(), _stream(stream)), "qmv_grouped")
    return y


def qmv_grouped_swiglu(fmt, tower: torch.Tensor, expert_ids: torch.Tensor, x: torch.Tensor, N: int,
                       K: int, E: int, ws: torch.Tensor, h: torch.Tensor | None = None,
                       stream=None) -> torch.Tensor:
    """h[t, j] = silu(gate_e . x[t]) * (up_e . x[t]), e = expert_ids[t, j], over a
    2E-expert tower (gate matrices 0..E-1, then up matrices E..2E-1)."""
    _dev(tower, "tower"); _dev(expert_ids, "expert_ids"); _dev(x, "x"); _dev(ws, "ws")
    if expert_ids.dtype != torch.int32 or expert_ids.dim() != 2:
        raise ValueError("expert_ids must be int32 [M, topk]")
    if not expert_ids.is_contiguous():
        raise ValueError("expert_ids must be contiguous")
    M, topk = expert_ids.shape
    x, _ = _act(x, K, M)
    h = _out(h, (M, topk, N), x.device, "h")
    _check(_grouped_swiglu(_fmt(fmt), _ptr(tower), _ptr(expert_ids), _ptr(x), _ptr(h), M, topk, N, K, E,
                           _ptr(ws), ws.numel(), _stream(stream)), "qmv_grouped_swiglu")
    return h


def qmv_quant_act_nvfp4(x: torch.Tensor, x_scale: float, codes: torch.Tensor | None = None,
                        scales: torch.Tensor | None = None, stream=None):
    _dev(x, "x")
    x = _bits16(x)
    if x.dim() != 2 or not x.is_contiguous():
        raise ValueError("x must be a contiguous [M, K] tensor")
    M, K = x.shape
    for t, n, name in ((codes, M * (K // 2), "codes"), (scales, M * (K // 16), "scales")):
        if t is not None and (t.dtype != torch.uint8 or not t.is_contiguous() or t.numel() < n or not t.is_cuda):
            raise ValueError(f"{name} must be a contiguous CUDA uint8 tensor of at least {n} bytes")
    if codes is None:
        codes = torch.empty((M, K // 2), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty((M, K // 16), dtype=torch.uint8, device=x.device)
    _check(_quant_act(_ptr(x), float(x_scale), _ptr(codes), _ptr(scales), M, K, _stream(stream)),
           "qmv_quant_act_nvfp4")
    return codes, scales


def qmv_gemm_nvfp4_w4a4(packed_W: torch.Tensor, x: torch.Tensor, x_scale: float, N: int, K: int,
                        ws: torch.Tensor, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    _dev(packed_W, "packed_W"); _dev(x, "x"); _dev(ws, "ws")
    x, M = _act(x, K)
    y = _out(y, (M, N), x.device, "y")
    _check(_w4a4(_ptr(packed_W), _ptr(x), float(x_scale), _ptr(y), M, N, K, _ptr(ws), ws.numel(),
                 _stream(stream)), "qmv_gemm_nvfp4_w4a4")
    return y


def qmv_gemm_kquant(fmt, packed_W: torch.Tensor, x: torch.Tensor, N: int, K: int, ws: torch.Tensor,
                    y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y = x . W^T for a K-quant W at prefill sizes (tensor cores, each weight read once)."""
    _dev(packed_W, "packed_W"); _dev(x, "x"); _dev(ws, "ws")
    x, M = _act(x, K)
    y = _out(y, (M, N), x.device, "y")
    _check(_kquant(_fmt(fmt), _ptr(packed_W), _ptr(x), _ptr(y), M, N, K, _ptr(ws), ws.numel(), _stream(stream)),
           "qmv_gemm_kquant")
    return y


def qmv_gemv_int8dot(fmt, packed_W: torch.Tensor, x: torch.Tensor, N: int, K: int, ws: torch.Tensor,
                     y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y = q8(x) . W^T: x quantized to int8 per 32 values, integer dots (Q8_0, Q4_K; M <= 8)."""
    _dev(packed_W, "packed_W"); _dev(x, "x"); _dev(ws, "ws")
    x, M = _act(x, K)
    y = _out(y, (M, N), x.device, "y")
    _check(_int8dot(_fmt(fmt), _ptr(packed_W), _ptr(x), _ptr(y), M, N, K, _ptr(ws), ws.numel(), _stream(stream)),
           "qmv_gemv_int8dot")
    return y
