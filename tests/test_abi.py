"""The C-ABI library loads on a machine without a GPU, exports every entry point the
header declares, and its host-side validation answers without touching a device."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qmv.h")
LIB = os.path.join(ROOT, "block_quantized_weight_fly_gb300", "libqmv.so")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qmv_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        import importlib.util
        spec = importlib.util.spec_from_file_location(
            "qmv_build", os.path.join(ROOT, "block_quantized_weight_fly_gb300", "build.py"))
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
        mod.build()
    return ctypes.CDLL(LIB)


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert "qmv_gemv" in names and "qmv_grouped" in names and "qmv_pack" in names
    for n in names:
        assert hasattr(lib, n), n


def test_binding_exposes_every_declared_symbol(lib):
    import block_quantized_weight_fly_gb300 as q
    for n in _declared():
        assert n in q.EXPORTED and callable(getattr(q, n)), n


def test_sizes_match_oracle(lib):
    import block_quantized_weight_fly_gb300 as q
    for fmt in ("q8_0", "q4_k", "q5_k", "q6_k", "nvfp4", "fp8_row", "iq4_xs", "iq3_s", "iq2_s"):
        for N, K in ((512, 1024), (17408, 5120), (248320, 5120), (300, 768)):
            assert q.qmv_canon_size(fmt, N, K) == oracle.canon_bytes(fmt, N, K)
    # the packed layout moves the canonical bytes; only row/K padding and alignment add
    for fmt, per in (("q8_0", 34 / 32), ("q4_k", 144 / 256), ("q5_k", 176 / 256), ("q6_k", 210 / 256),
                     ("nvfp4", 18 / 32), ("fp8_row", 1.0), ("iq4_xs", 136 / 256), ("iq3_s", 110 / 256),
                     ("iq2_s", 82 / 256)):
        N, K = 17408, 5120
        body = q.qmv_pack_size(fmt, N, K) - 256
        # IQ4_XS adds its 16-byte codebook once per 128 x 256 slab; IQ3_S / IQ2_S their
        # f16 grid once
        extra = {"iq4_xs": 16 * (N // 128) * (K // 256), "iq3_s": 4096, "iq2_s": 16384}.get(fmt, 0)
        assert N * K * per + extra <= body <= N * K * per + extra + 4 * N + 512
    assert q.qmv_pack_size("q4_k", 100, 100) == 0          # K not a multiple of 256
    assert q.qmv_pack_size("q5_k", 100, 1000) == 0
    assert q.qmv_pack_size("q8_0", 100, 48) == 0           # K not a multiple of 32


def test_host_validation_without_device(lib):
    import block_quantized_weight_fly_gb300 as q
    P = ctypes.c_void_p
    gemv = q._gemv
    one = P(256)
    # null pointers, M out of range, bad format, misalignment: refused before any launch
    assert gemv(2, None, one, one, 1, 128, 256, one, 1 << 20, None) == 1
    assert gemv(2, one, one, one, 0, 128, 256, one, 1 << 20, None) == 1
    assert gemv(2, one, one, one, 9, 128, 256, one, 1 << 20, None) == 1
    assert gemv(99, one, one, one, 1, 128, 256, one, 1 << 20, None) == 1          # not a format
    assert gemv(0, one, one, one, 1, 128, 256, one, 1 << 20, None) == 1
    assert gemv(7, one, one, one, 1, 128, 100, one, 1 << 20, None) == 3             # IQ4_XS: K % 256
    assert gemv(6, one, one, one, 1, 128, 100, one, 1 << 20, None) == 3
    assert gemv(2, one, one, one, 1, 128, 100, one, 1 << 20, None) == 3
    assert gemv(2, P(257), one, one, 1, 128, 256, one, 1 << 20, None) == 2
    assert gemv(2, one, P(258), one, 1, 128, 256, one, 1 << 20, None) == 2
    assert q._grouped(2, one, one, one, 2, one, 1, 1, 128, 256, 4, one, 1 << 20, None) == 1
    assert q._grouped(2, one, one, one, 0, one, 1, 9, 128, 256, 4, one, 1 << 20, None) == 1
    assert q.qmv_status_str(0) == "ok" and "workspace" in q.qmv_status_str(8)


def test_host_validation_new_entries(lib):
    """The grouped SwiGLU and prefill entries refuse bad arguments before any launch."""
    import block_quantized_weight_fly_gb300 as q
    P = ctypes.c_void_p
    one = P(256)
    gs = q._grouped_swiglu       # fmt, tower, ids, x, h, M, topk, N, K, E, ws, ws_bytes, stream
    assert gs(2, None, one, one, one, 1, 1, 128, 256, 4, one, 1 << 20, None) == 1   # null tower
    assert gs(2, one, one, one, one, 0, 1, 128, 256, 4, one, 1 << 20, None) == 1    # M = 0
    assert gs(2, one, one, one, one, 9, 1, 128, 256, 4, one, 1 << 20, None) == 1    # M > 8
    assert gs(2, one, one, one, one, 1, 9, 128, 256, 4, one, 1 << 20, None) == 1    # topk > 8
    assert gs(2, one, one, one, one, 1, 1, 128, 256, 0, one, 1 << 20, None) == 1    # E = 0
    assert gs(2, one, one, one, one, 1, 1, 128, 100, 4, one, 1 << 20, None) == 3    # K % 256
    assert gs(2, P(257), one, one, one, 1, 1, 128, 256, 4, one, 1 << 20, None) == 2  # tower alignment
    kq = q._kquant               # fmt, W, x, y, M, N, K, ws, ws_bytes, stream
    assert kq(2, None, one, one, 512, 128, 256, one, 1 << 20, None) == 1
    assert kq(2, one, one, one, 0, 128, 256, one, 1 << 20, None) == 1
    assert kq(99, one, one, one, 512, 128, 256, one, 1 << 20, None) == 1             # not a format
    for fmt in (1, 4, 5, 7, 8, 9):                                                   # Q8_0, NVFP4, FP8, IQ
        assert kq(fmt, one, one, one, 512, 128, 256, one, 1 << 20, None) == 3
    assert kq(2, one, one, one, 512, 128, 300, one, 1 << 20, None) == 3              # K % 256
    assert kq(6, one, one, one, 512, 128, 300, one, 1 << 20, None) == 3
    assert kq(2, one, P(264), one, 512, 128, 256, one, 1 << 20, None) == 2           # x alignment
    i8 = q._int8dot              # fmt, W, x, y, M, N, K, ws, ws_bytes, stream
    assert i8(2, None, one, one, 1, 128, 256, one, 1 << 20, None) == 1
    assert i8(2, one, one, one, 0, 128, 256, one, 1 << 20, None) == 1                # M = 0
    assert i8(2, one, one, one, 9, 128, 256, one, 1 << 20, None) == 1                # M > 8
    assert i8(99, one, one, one, 1, 128, 256, one, 1 << 20, None) == 1               # not a format
    for fmt in (3, 4, 5, 6, 7, 8, 9):                                                # Q8_0 and Q4_K only
        assert i8(fmt, one, one, one, 1, 128, 256, one, 1 << 20, None) == 3
    assert i8(1, one, one, one, 1, 128, 48, one, 1 << 20, None) == 3                 # K % 32
    assert i8(2, one, one, one, 1, 128, 288, one, 1 << 20, None) == 3                # K % 256
    assert i8(2, P(257), one, one, 1, 128, 256, one, 1 << 20, None) == 2             # W alignment
    assert i8(1, one, one, one, 2, 128, 256, one, 511, None) == 8                    # workspace too small
    assert q.qmv_workspace_size(q.QMV_ENTRY_INT8DOT, "q4_k", 3, 128, 5120) == 15360 + 2048
    assert q.qmv_workspace_size(q.QMV_ENTRY_INT8DOT, "q6_k", 1, 128, 5120) == 0


def test_host_validation_remaining_entries(lib):
    """The dense SwiGLU, no-workspace GEMV, activation quantizer, W4A4 GEMM, pack,
    dequant and quantize entries refuse bad arguments before any launch (every case
    below fails a host check, so nothing is launched on any machine)."""
    import block_quantized_weight_fly_gb300 as q
    P = ctypes.c_void_p
    one = P(256)
    nan = float("nan")
    sw = q._gemv_swiglu          # fmt, tower, x, h, M, N, K, ws, ws_bytes, stream
    assert sw(2, None, one, one, 1, 128, 256, one, 1 << 20, None) == 1
    assert sw(2, one, one, one, 0, 128, 256, one, 1 << 20, None) == 1
    assert sw(2, one, one, one, 9, 128, 256, one, 1 << 20, None) == 1
    assert sw(2, one, one, one, 1, 128, 100, one, 1 << 20, None) == 3
    assert sw(2, P(257), one, one, 1, 128, 256, one, 1 << 20, None) == 2
    assert q._gemv(2, one, one, one, 1, 0, 256, one, 1 << 20, None) == 1          # N = 0
    assert q._gemv(2, one, one, one, 1, 128, 256, P(260), 1 << 20, None) == 2     # ws alignment
    na = q._gemv_noalloc         # fmt, W, x, y, M, N, K, stream
    assert na(2, None, one, one, 1, 128, 256, None) == 1
    assert na(2, one, one, one, 9, 128, 256, None) == 1
    assert na(2, one, one, one, 1, 128, 100, None) == 3
    qa = q._quant_act            # x, x_scale, codes, scales, M, K, stream
    assert qa(None, 1.0, one, one, 4, 256, None) == 1
    assert qa(one, 1.0, one, one, 0, 256, None) == 1
    assert qa(one, -1.0, one, one, 4, 256, None) == 1                            # negative scale
    assert qa(one, nan, one, one, 4, 256, None) == 1
    assert qa(one, 1.0, one, one, 4, 40, None) == 3                              # K % 16
    w4 = q._w4a4                 # W, x, x_scale, y, M, N, K, ws, ws_bytes, stream
    assert w4(None, one, 1.0, one, 512, 128, 256, one, 1 << 24, None) == 1
    assert w4(one, one, 1.0, one, 0, 128, 256, one, 1 << 24, None) == 1
    assert w4(one, one, nan, one, 512, 128, 256, one, 1 << 24, None) == 1
    assert w4(one, one, 1.0, one, 512, 128, 40, one, 1 << 24, None) == 3         # K % 256
    assert w4(P(257), one, 1.0, one, 512, 128, 256, one, 1 << 24, None) == 2
    pk = q._pack                 # fmt, canon, N, K, E, dst, stream
    assert pk(2, None, 128, 256, 1, one, None) == 1
    assert pk(2, one, 128, 256, 0, one, None) == 1                               # E = 0
    assert pk(99, one, 128, 256, 1, one, None) == 1
    assert pk(2, one, 128, 100, 1, one, None) == 3
    assert pk(2, one, 128, 256, 1, P(257), None) == 2
    dq = q._dequant              # fmt, packed, N, K, E, row0, rows, out, stream
    assert dq(2, None, 128, 256, 1, 0, 128, one, None) == 1
    assert dq(2, one, 128, 256, 1, 100, 100, one, None) == 1                     # rows past N
    assert dq(2, one, 128, 256, 1, -1, 10, one, None) == 1
    qz = q._quantize             # fmt, W, rows, K, tensor_scale, canon, stream
    assert qz(2, None, 128, 256, 0.0, one, None) == 1
    assert qz(99, one, 128, 256, 0.0, one, None) == 1
    assert qz(2, one, 128, 100, 0.0, one, None) == 3
    assert qz(7, one, 128, 256, 0.0, one, None) == 3                             # IQ4_XS needs a codebook
    assert qz(9, one, 128, 256, 0.0, one, None) == 3                             # IQ2_S needs its grid
    qc = q._quantize_cb          # fmt, W, rows, K, codebook, canon, stream
    assert qc(7, None, 128, 256, one, one, None) == 1
    assert qc(7, one, 128, 256, None, one, None) == 1                            # no codebook
    assert qc(2, one, 128, 256, one, one, None) == 3                             # not a codebook format
    assert qc(99, one, 128, 256, one, one, None) == 1
    assert qc(7, one, 128, 100, one, one, None) == 3                             # K % 256
    assert qc(7, P(258), 128, 256, one, one, None) == 2
    # workspace sizes of impossible requests are 0
    assert q._ws_size(1, 2, 0, 128, 256, 1, 1) == 0                              # M = 0
    assert q._ws_size(9, 2, 1, 128, 256, 1, 1) == 0                              # no such entry
    assert q._ws_size(1, 2, 9, 128, 256, 1, 1) == 0                              # M > 8
