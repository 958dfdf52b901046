"""CPU oracle for the block-quantized weight GEMV -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA product path never does; the two
share no code. The arithmetic lives in ``oracle.c`` (plain single-threaded C,
fp32 dequantization with round-to-nearest-even, fp64 dot products); this module
only builds it with gcc and marshals numpy arrays through ctypes.

Every function cites the passage it follows in ``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

Q8_0, Q4_K, Q6_K, NVFP4, FP8_ROW, Q5_K, IQ4_XS, IQ3_S, IQ2_S = 1, 2, 3, 4, 5, 6, 7, 8, 9
FORMATS = {"q8_0": Q8_0, "q4_k": Q4_K, "q6_k": Q6_K, "nvfp4": NVFP4, "fp8_row": FP8_ROW,
           "q5_k": Q5_K, "iq4_xs": IQ4_XS, "iq3_s": IQ3_S, "iq2_s": IQ2_S}
CODEBOOK_FORMATS = ("iq4_xs", "iq3_s", "iq2_s")
GRID_SHAPES = {"iq3_s": (512, 4), "iq2_s": (1024, 8)}

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, -O2, no FMA contraction)."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(os.path.join(_HERE, "oracle.h")))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c99",
                               "-fPIC", "-shared", "-Wall", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    lib.or_fp16_to_f32.restype = ctypes.c_float
    lib.or_fp16_to_f32.argtypes = [ctypes.c_uint16]
    lib.or_f32_to_fp16.restype = ctypes.c_uint16
    lib.or_f32_to_fp16.argtypes = [ctypes.c_float]
    lib.or_bf16_to_f32.restype = ctypes.c_float
    lib.or_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.or_f64_to_bf16.restype = ctypes.c_uint16
    lib.or_f64_to_bf16.argtypes = [ctypes.c_double]
    lib.or_e4m3_to_f32.restype = ctypes.c_float
    lib.or_e4m3_to_f32.argtypes = [ctypes.c_uint8]
    lib.or_f32_to_e4m3.restype = ctypes.c_uint8
    lib.or_f32_to_e4m3.argtypes = [ctypes.c_float]
    lib.or_e2m1_to_f32.restype = ctypes.c_float
    lib.or_e2m1_to_f32.argtypes = [ctypes.c_uint8]
    lib.or_f32_to_e2m1.restype = ctypes.c_uint8
    lib.or_f32_to_e2m1.argtypes = [ctypes.c_float]
    lib.or_block_values.restype = I64
    lib.or_block_values.argtypes = [ctypes.c_int]
    lib.or_canon_bytes.restype = I64
    lib.or_canon_bytes.argtypes = [ctypes.c_int, I64, I64]
    lib.or_encode.restype = ctypes.c_int
    lib.or_encode.argtypes = [ctypes.c_int, P, I64, I64, ctypes.c_float, P]
    lib.or_encode_cb.restype = ctypes.c_int
    lib.or_encode_cb.argtypes = [ctypes.c_int, P, I64, I64, P, P]
    lib.or_grid_bytes.restype = I64
    lib.or_grid_bytes.argtypes = [ctypes.c_int]
    lib.or_block_to_float.restype = ctypes.c_int
    lib.or_block_to_float.argtypes = [ctypes.c_int, P, I64, I64, P]
    lib.or_gemv_f64.restype = None
    lib.or_gemv_f64.argtypes = [P, I64, I64, P, I64, P, P]
    lib.or_unique_experts.restype = I64
    lib.or_unique_experts.argtypes = [P, I64, P]
    lib.or_quant_act_nvfp4.restype = None
    lib.or_quant_act_nvfp4.argtypes = [P, I64, I64, ctypes.c_float, P, P]
    lib.or_swiglu_f64.restype = None
    lib.or_swiglu_f64.argtypes = [P, P, I64, P]
    lib.or_quant_act_q8.restype = None
    lib.or_quant_act_q8.argtypes = [P, I64, I64, P, P]
    lib.or_int8dot_f64.restype = None
    lib.or_int8dot_f64.argtypes = [P, I64, I64, P, I64, P, P]
    lib.or_w4a4_f64.restype = None
    lib.or_w4a4_f64.argtypes = [P, I64, I64, ctypes.c_float, P, I64, P, P]
    _lib = lib
    return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _fmt(fmt) -> int:
    return FORMATS[fmt] if isinstance(fmt, str) else int(fmt)


# ---- scalar formats ---------------------------------------------------------
def fp16_to_f32(h: int) -> float:
    return _load().or_fp16_to_f32(h)


def f32_to_fp16(f: float) -> int:
    return _load().or_f32_to_fp16(f)


def bf16_to_f32(b: int) -> float:
    return _load().or_bf16_to_f32(b)


def f64_to_bf16(v: float) -> int:
    return _load().or_f64_to_bf16(float(v))


def f64_to_bf16_array(a: np.ndarray) -> np.ndarray:
    """Elementwise bf16 round-to-nearest-even (uint16 bit patterns)."""
    a = np.asarray(a, dtype=np.float64)
    f = _load().or_f64_to_bf16
    return np.array([f(float(v)) for v in a.reshape(-1)], dtype=np.uint16).reshape(a.shape)


def e4m3_to_f32(c: int) -> float:
    return _load().or_e4m3_to_f32(c)


def f32_to_e4m3(f: float) -> int:
    return _load().or_f32_to_e4m3(f)


def e2m1_to_f32(c: int) -> float:
    return _load().or_e2m1_to_f32(c)


def f32_to_e2m1(f: float) -> int:
    return _load().or_f32_to_e2m1(f)


# ---- sizes --------------------------------------------------------------------
def block_values(fmt) -> int:
    return int(_load().or_block_values(_fmt(fmt)))


def canon_bytes(fmt, rows: int, K: int) -> int:
    return int(_load().or_canon_bytes(_fmt(fmt), rows, K))


# ---- matrices -----------------------------------------------------------------
def grid_bytes(fmt) -> int:
    return int(_load().or_grid_bytes(_fmt(fmt)))


def encode(fmt, W: np.ndarray, tensor_scale: float = 0.0, codebook=None) -> np.ndarray:
    """fp32 W[rows, K] -> canonical bytes (synthetic-data encoder). The codebook
    formats take their table: IQ4_XS the matrix's codebook (16 int8 values), IQ3_S
    and IQ2_S the grid (uint8 magnitudes [512, 4] / [1024, 8])."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    rows, K = W.shape
    out = np.zeros(canon_bytes(fmt, rows, K), dtype=np.uint8)
    if _fmt(fmt) in (IQ4_XS, IQ3_S, IQ2_S):
        if _fmt(fmt) == IQ4_XS:
            cb = np.ascontiguousarray(codebook, dtype=np.int8).reshape(-1)
            assert cb.shape == (16,)
        else:
            cb = np.ascontiguousarray(codebook, dtype=np.uint8).reshape(-1)
            assert cb.size == grid_bytes(fmt)
        rc = _load().or_encode_cb(_fmt(fmt), _ptr(W), rows, K, _ptr(cb), _ptr(out))
    else:
        rc = _load().or_encode(_fmt(fmt), _ptr(W), rows, K, float(tensor_scale), _ptr(out))
    if rc:
        raise ValueError(f"or_encode failed ({rc}) for fmt={fmt} K={K}")
    return out


def block_to_float(fmt, canon: np.ndarray, rows: int, K: int) -> np.ndarray:
    """BlockToFloat: canonical bytes of `rows` rows -> fp32 W[rows, K]."""
    canon = np.ascontiguousarray(canon, dtype=np.uint8)
    if canon.size < canon_bytes(fmt, rows, K):
        raise ValueError("canonical buffer too small")
    W = np.empty((rows, K), dtype=np.float32)
    rc = _load().or_block_to_float(_fmt(fmt), _ptr(canon), rows, K, _ptr(W))
    if rc:
        raise ValueError(f"or_block_to_float failed ({rc})")
    return W


def gemv_f64(W: np.ndarray, x_bf16: np.ndarray):
    """y[M, N] = x . W^T in fp64 and den[M, N] = sum_k |w x| (error scale)."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    if x.ndim == 1:
        x = x[None, :]
    N, K = W.shape
    M = x.shape[0]
    assert x.shape[1] == K
    y = np.empty((M, N), dtype=np.float64)
    den = np.empty((M, N), dtype=np.float64)
    _load().or_gemv_f64(_ptr(W), N, K, _ptr(x), M, _ptr(y), _ptr(den))
    return y, den


def unique_experts(ids: np.ndarray) -> np.ndarray:
    ids = np.ascontiguousarray(ids, dtype=np.int32).reshape(-1)
    out = np.empty(max(ids.size, 1), dtype=np.int32)
    u = _load().or_unique_experts(_ptr(ids), ids.size, _ptr(out))
    return out[:u].copy()


def quant_act_nvfp4(x_bf16: np.ndarray, x_scale: float):
    """bf16 x[M, K] -> (codes [M, K/2] uint8, scales [M, K/16] uint8)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    M, K = x.shape
    codes = np.zeros((M, K // 2), dtype=np.uint8)
    scales = np.zeros((M, K // 16), dtype=np.uint8)
    _load().or_quant_act_nvfp4(_ptr(x), M, K, float(x_scale), _ptr(codes), _ptr(scales))
    return codes, scales


def w4a4_f64(W: np.ndarray, x_bf16: np.ndarray, x_scale: float):
    """W4A4 reference: the activation quantized by the oracle's NVFP4 quantizer under
    the static x_scale and dequantized (e2m1 * e4m3 * x_scale), then fp64 dots with the
    BlockToFloat weights W[N, K]. Returns (y [M, N], den [M, N] = sum |terms|)."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    if x.ndim == 1:
        x = x[None, :]
    N, K = W.shape
    M = x.shape[0]
    assert x.shape[1] == K and K % 16 == 0
    y = np.empty((M, N), dtype=np.float64)
    den = np.empty((M, N), dtype=np.float64)
    _load().or_w4a4_f64(_ptr(x), M, K, float(x_scale), _ptr(W), N, _ptr(y), _ptr(den))
    return y, den


def quant_act_q8(x_bf16: np.ndarray):
    """bf16 x[M, K] -> (int8 codes [M, K], fp32 scales [M, K/32]): d = amax / 127 per
    32 values, q = clamp(rint(x / d), -127, 127)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    if x.ndim == 1:
        x = x[None, :]
    M, K = x.shape
    codes = np.zeros((M, K), dtype=np.int8)
    scales = np.zeros((M, K // 32), dtype=np.float32)
    _load().or_quant_act_q8(_ptr(x), M, K, _ptr(codes), _ptr(scales))
    return codes, scales


def int8dot_f64(W: np.ndarray, x_bf16: np.ndarray):
    """The int8-dot reference: x quantized by quant_act_q8, then fp64 dots with the
    BlockToFloat weights W[N, K]. Returns (y [M, N], den [M, N] = sum |terms|)."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    if x.ndim == 1:
        x = x[None, :]
    N, K = W.shape
    M = x.shape[0]
    assert x.shape[1] == K and K % 32 == 0
    y = np.empty((M, N), dtype=np.float64)
    den = np.empty((M, N), dtype=np.float64)
    _load().or_int8dot_f64(_ptr(x), M, K, _ptr(W), N, _ptr(y), _ptr(den))
    return y, den


def swiglu_f64(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """h = silu(g) * u elementwise, fp64 (the SwiGLU behind the gate/up projection)."""
    g = np.ascontiguousarray(g, dtype=np.float64)
    u = np.ascontiguousarray(u, dtype=np.float64)
    assert g.shape == u.shape
    h = np.empty_like(g)
    _load().or_swiglu_f64(_ptr(g), _ptr(u), g.size, _ptr(h))
    return h


def grouped_f64(tower_canon_rows, ids: np.ndarray, x_bf16: np.ndarray, x_per_pair: bool):
    """Reference for the grouped per-expert GEMV over a stacked tower.

    ``tower_canon_rows(e)`` returns the fp32 dequantized rows W_e[N, K] of expert
    e (BlockToFloat of that expert's slice). For every (token t, slot j):
    y[t, j, :] = W_{ids[t, j]} . x_row(t, j), x_row = x[t] or x[t*topk + j].
    """
    ids = np.asarray(ids, dtype=np.int32)
    M, topk = ids.shape
    ys, dens = {}, {}
    cache = {}
    for t in range(M):
        for j in range(topk):
            e = int(ids[t, j])
            if e not in cache:
                cache[e] = tower_canon_rows(e)
            xr = x_bf16[t * topk + j] if x_per_pair else x_bf16[t]
            y, den = gemv_f64(cache[e], xr[None, :])
            ys[(t, j)] = y[0]
            dens[(t, j)] = den[0]
    N = next(iter(ys.values())).shape[0]
    Y = np.zeros((M, topk, N))
    D = np.zeros((M, topk, N))
    for (t, j), v in ys.items():
        Y[t, j] = v
        D[t, j] = dens[(t, j)]
    return Y, D
