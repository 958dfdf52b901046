"""GPU: the int8-dot decode GEMV (qmv_gemv_int8dot) against the CPU oracle.

- the activation quantizer's codes and block scales (left in the workspace) equal the
  oracle's quant_act_q8 bit for bit, on N(0, 1) rows and on crafted blocks: all zero,
  a single non-zero value, ties x/d = k + 1/2, subnormal bf16, the largest bf16, mixed
  signs at the clamp;
- y against the oracle's int8dot_f64 (fp64 dots of the BlockToFloat weights with the
  quantized x), normalised error <= 1e-5, for Q8_0 (ragged K: a last k-group of one
  32-value chunk) and Q4_K, ragged N, M = 1, 3, 8;
- against the bf16-x GEMV, the difference stays within what x's rounding allows:
  sum_k |w_k| d_b / 2 (plus the tolerance);
- the rows of an M-row call equal one-row calls bit for bit;
- at the Qwen3.8-27B MLP shapes, sampled rows against the oracle;
- a header that disagrees with the arguments latches status 5 and leaves y alone.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from cases import TOL, device_matrix, host_dequant, host_matrix, host_rows_dequant, norm_err, sample_rows

pytestmark = pytest.mark.gpu

QWEN_HIDDEN, QWEN_MLP = 5120, 17408


@pytest.fixture(scope="module")
def q():
    import block_quantized_weight_fly_gb300 as q
    torch.cuda.set_device(0)
    q.qmv_device_status(reset=True)
    return q


def _call(q, fmt, packed, x, N, K, ws=None):
    M = x.shape[0]
    if ws is None:
        ws = q.workspace(q.QMV_ENTRY_INT8DOT, fmt, M, N, K)
    y = q.qmv_gemv_int8dot(fmt, packed, x, N, K, ws)
    assert q.qmv_last_route() == q.FORMATS[fmt] * 100 + 13
    return y, ws


# Q4_K: the quantizer stores each 8-value slice in a packed Q4_K word's nibble order
# (byte SLICE_POS[p] holds element p of the slice); Q8_0 in element order
SLICE_POS = {"q4_k": [0, 2, 4, 6, 1, 3, 5, 7], "q8_0": list(range(8))}


def _ws_codes(ws, fmt, M, K):
    """the quantizer's output in the workspace, back in element order: codes [M][K]
    int8, scales [M][K/32] fp32. Rows of x are Kp = 256 x (k-groups) bytes apart; in
    k-group g, slice t (values 8t .. 8t+7) of chunk j sits at byte 64t + 8j."""
    G = -(-K // 256)
    Kp = 256 * G
    w = ws.cpu().numpy()
    raw = w[:M * Kp].view(np.int8).reshape(M, G, 4, 8, 8)           # [m][g][t][j][slot]
    codes = raw.transpose(0, 1, 3, 2, 4)[..., SLICE_POS[fmt]].reshape(M, Kp)[:, :K]
    off = (M * Kp + 255) // 256 * 256
    scales = w[off:off + M * (Kp // 32) * 4].view(np.float32).reshape(M, Kp // 32)[:, :K // 32]
    return np.ascontiguousarray(codes), np.ascontiguousarray(scales)


def _crafted_x(K, huge=False):
    """bf16 bit patterns [8, K]: N(0, 1) rows with crafted 32-value blocks in front
    (huge: row 3 reaches the largest finite bf16, where the dot products overflow fp32,
    so only the quantizer is compared)"""
    x = synth.bf16_bits(synth.activations(301, 8, K)).copy()
    f = lambda v: np.frombuffer(np.asarray(v, dtype=np.float32).tobytes(), dtype=np.uint32) >> 16
    x[0, 0:32] = 0                                           # all zero: d = 0, codes 0
    x[0, 32:64] = 0
    x[0, 40] = f(-3.0)[0]                                    # one non-zero value: q = -127
    # ties: amax = 127 gives d = 1 exactly, so x = k + 1/2 lands on x/d = k + 1/2
    blk = np.array([127.0] + [k + 0.5 for k in range(-15, 16)], dtype=np.float32)
    x[1, 0:32] = f(blk)
    x[2, 0:32] = np.arange(1, 33, dtype=np.uint16)           # positive subnormal bf16
    x[2, 32:64] = 0x8000 | np.arange(1, 33, dtype=np.uint16)  # negative subnormal
    if huge:
        x[3, 0:32] = f(np.linspace(-3.3895e38, 3.3895e38, 32))   # up to the largest bf16
        x[3, 32] = 0x7F7F                                        # the largest finite bf16
        x[3, 33] = 0xFF7F
    else:
        x[3, 0:32] = f(np.linspace(-1.0e4, 1.0e4, 32))
    x[4, 0:32] = f(np.array([(-1) ** i * (127.0 - i) for i in range(32)], dtype=np.float32))
    return x


@pytest.mark.parametrize("fmt,N,K", [("q8_0", 300, 800), ("q8_0", 640, 1024), ("q4_k", 300, 768),
                                     ("q4_k", 1024, 2048)])
@pytest.mark.parametrize("M", [1, 3, 8])
def test_int8dot_against_oracle(q, fmt, N, K, M):
    seed = 311 + N + K
    _, canon = host_matrix(fmt, seed, N, K)
    packed = q.qmv_pack(fmt, torch.from_numpy(canon).cuda(), N, K)
    xb = _crafted_x(K)[:M] if M > 1 else synth.bf16_bits(synth.activations(seed, 1, K))
    x = torch.from_numpy(xb.view(np.int16).copy()).view(torch.bfloat16).cuda()
    y, ws = _call(q, fmt, packed, x, N, K)
    torch.cuda.synchronize()
    assert q.qmv_device_status() == 0
    codes, scales = _ws_codes(ws, fmt, M, K)
    rc, rs = oracle.quant_act_q8(xb)
    assert np.array_equal(codes, rc)
    assert np.array_equal(scales.view(np.uint32), rs.view(np.uint32))
    D = host_dequant(fmt, canon, N, K)
    yref, den = oracle.int8dot_f64(D, xb)
    yg = y.cpu().numpy()
    assert np.all(np.isfinite(yg))
    assert norm_err(yg, yref, den) <= TOL
    # the int8 rounding of x moves the result by at most sum_k |w_k| d_b / 2 from the
    # bf16-x GEMV
    yx, denx = oracle.gemv_f64(D, xb)
    half = np.repeat(rs.astype(np.float64), 32, axis=1) / 2          # [M, K]
    shift = half @ np.abs(D.astype(np.float64)).T                     # [M, N]
    assert np.all(np.abs(yg - yx) <= shift * (1 + 1e-6) + TOL * (den + denx))


def test_int8dot_quantizer_crafted(q):
    """every crafted block, all eight rows, Q8_0 at K = 1024"""
    fmt, N, K = "q8_0", 128, 1024
    _, canon = host_matrix(fmt, 331, N, K)
    packed = q.qmv_pack(fmt, torch.from_numpy(canon).cuda(), N, K)
    xb = _crafted_x(K, huge=True)
    x = torch.from_numpy(xb.view(np.int16).copy()).view(torch.bfloat16).cuda()
    y, ws = _call(q, fmt, packed, x, N, K)
    torch.cuda.synchronize()
    codes, scales = _ws_codes(ws, fmt, 8, K)
    rc, rs = oracle.quant_act_q8(xb)
    assert np.array_equal(codes, rc)
    assert np.array_equal(scales.view(np.uint32), rs.view(np.uint32))
    assert np.all(codes[0, :32] == 0) and codes[0, 40] == -127
    assert int(np.abs(rc).max()) <= 127 and int(rc.min()) >= -127


@pytest.mark.parametrize("fmt", ["q8_0", "q4_k"])
def test_int8dot_rows_equal_single_rows(q, fmt):
    N, K = 512, 1536
    _, canon = host_matrix(fmt, 341, N, K)
    packed = q.qmv_pack(fmt, torch.from_numpy(canon).cuda(), N, K)
    x = synth.activations(343, 8, K).cuda()
    singles = [_call(q, fmt, packed, x[m:m + 1], N, K)[0][0].clone() for m in range(8)]
    for M in (8, 5, 2):
        yM, _ = _call(q, fmt, packed, x[:M], N, K)
        for m in range(M):
            assert torch.equal(yM[m], singles[m]), (M, m)
    assert q.qmv_device_status() == 0


@pytest.mark.parametrize("fmt,N,K", [("q4_k", QWEN_MLP, QWEN_HIDDEN), ("q8_0", QWEN_HIDDEN, QWEN_MLP)])
@pytest.mark.parametrize("M", [1, 8])
def test_int8dot_full_size_sampled(q, fmt, N, K, M):
    seed = 351 + M
    packed = device_matrix(q, fmt, seed, N, K)
    x = synth.activations(seed + 1, M, K).cuda()
    y, _ = _call(q, fmt, packed, x, N, K)
    torch.cuda.synchronize()
    assert q.qmv_device_status() == 0
    rows = sample_rows(N, 24, seed)
    D = host_rows_dequant(fmt, seed, rows, N, K)
    yref, den = oracle.int8dot_f64(D, synth.bf16_bits(x))
    assert norm_err(y.cpu().numpy()[:, rows], yref, den) <= TOL
    assert bool(torch.isfinite(y).all())
    del packed
    torch.cuda.empty_cache()


def test_int8dot_header_mismatch(q):
    fmt, N, K, M = "q4_k", 256, 512, 2
    _, canon = host_matrix(fmt, 361, N, K)
    packed = q.qmv_pack(fmt, torch.from_numpy(canon).cuda(), N, K)
    x = synth.activations(363, M, K).cuda()
    y = torch.full((M, 128), 7.0, device="cuda")
    ws = q.workspace(q.QMV_ENTRY_INT8DOT, fmt, M, 128, K)
    q.qmv_device_status(reset=True)
    q.qmv_gemv_int8dot(fmt, packed, x, 128, K, ws, y=y)          # N disagrees with the header
    torch.cuda.synchronize()
    assert q.qmv_device_status(reset=True) == 5
    assert bool((y == 7.0).all())
    with pytest.raises(q.QmvError) as ei:
        q.qmv_gemv_int8dot(fmt, packed, x, N, K, ws[:100])
    assert ei.value.status == 8
    with pytest.raises(q.QmvError) as ei:
        q.qmv_gemv_int8dot("q6_k", packed, x, N, K, ws)
    assert ei.value.status == 3
