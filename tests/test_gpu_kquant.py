"""GPU parity of the K-quant (Q4_K, Q5_K, Q6_K) prefill GEMM on the tensor cores
(tcgen05 kind::f16).

Expected values come from the CPU oracle only: BlockToFloat of the weights and fp64
dots with the bf16 activations -- the same definition the GEMV meets. The bound is
the GEMV's: |y - y_ref| <= 1e-5 sum_k |w x| per output. Q6_K's scale is split into
two exact f16 terms (16 sh + sl); a test with arbitrary block bytes covers every
int8 scale, including -128, and every 6-bit code.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from cases import TOL, device_matrix, host_dequant, host_matrix, host_rows_dequant, norm_err, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import block_quantized_weight_fly_gb300 as q
    torch.cuda.set_device(0)
    q.qmv_device_status(reset=True)
    return q


def flags_view(q, ws, M, K):
    """The per-SM publication flags at the end of the workspace."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    m_pad = -(-M // 128) * 128
    off = m_pad * K * 2 + (m_pad // 128) * (K // 256) * 4096 + sms * 128 * 128 * 4
    return ws[off:off + 4 * sms]


@pytest.mark.parametrize("fmt", ["q4_k", "q5_k", "q6_k"])
@pytest.mark.parametrize("M,N,K", [(128, 128, 256), (1, 128, 256), (129, 200, 512), (300, 384, 1024),
                                   (257, 1000, 2048), (512, 640, 4096)])
def test_kquant_parity(q, fmt, M, N, K):
    W, canon = host_matrix(fmt, 51, N, K)
    D = host_dequant(fmt, canon, N, K)
    x = synth.activations(53 + M, M, K)
    ref, den = oracle.gemv_f64(D, synth.bf16_bits(x))
    packed = q.qmv_pack(fmt, torch.from_numpy(canon).cuda(), N, K)
    ws = q.workspace(q.QMV_ENTRY_KQUANT, fmt, M, N, K)
    y = q.qmv_gemm_kquant(fmt, packed, x.cuda(), N, K, ws)
    assert q.qmv_last_route() == q.FORMATS[fmt] * 100 + 11
    y = y.cpu().numpy()
    assert q.qmv_device_status() == 0
    assert norm_err(y, ref, den) <= TOL
    assert int(flags_view(q, ws, M, K).count_nonzero()) == 0


@pytest.mark.parametrize("fmt,M,N,K", [("q4_k", 2048, 384, 1024), ("q5_k", 1000, 260, 512), ("q6_k", 1000, 260, 512)])
def test_kquant_large_and_ragged_m(q, fmt, M, N, K):
    """Many token tiles (M = 2048: 16 tiles) and a ragged last token tile (M = 1000)."""
    W, canon = host_matrix(fmt, 65, N, K)
    D = host_dequant(fmt, canon, N, K)
    x = synth.activations(67, M, K)
    ref, den = oracle.gemv_f64(D, synth.bf16_bits(x))
    packed = q.qmv_pack(fmt, torch.from_numpy(canon).cuda(), N, K)
    ws = q.workspace(q.QMV_ENTRY_KQUANT, fmt, M, N, K)
    y = q.qmv_gemm_kquant(fmt, packed, x.cuda(), N, K, ws).cpu().numpy()
    assert q.qmv_device_status() == 0
    assert norm_err(y, ref, den) <= TOL
    assert int(flags_view(q, ws, M, K).count_nonzero()) == 0


@pytest.mark.parametrize("fmt,M,N,K", [("q4_k", 256, 256, 2048), ("q4_k", 384, 130, 4096), ("q5_k", 256, 300, 2048),
                                       ("q6_k", 256, 300, 2048)])
def test_kquant_split_k_deterministic(q, fmt, M, N, K):
    """Few tiles over many CTAs: every tile is split across CTAs and finished from
    its peers' partial tiles. Two calls give identical bits, the flags end at zero."""
    W, canon = host_matrix(fmt, 57, N, K)
    D = host_dequant(fmt, canon, N, K)
    x = synth.activations(59, M, K)
    ref, den = oracle.gemv_f64(D, synth.bf16_bits(x))
    packed = q.qmv_pack(fmt, torch.from_numpy(canon).cuda(), N, K)
    ws = q.workspace(q.QMV_ENTRY_KQUANT, fmt, M, N, K)
    xd = x.cuda()
    y1 = q.qmv_gemm_kquant(fmt, packed, xd, N, K, ws).cpu()
    y2 = q.qmv_gemm_kquant(fmt, packed, xd, N, K, ws).cpu()
    assert q.qmv_device_status() == 0
    assert torch.equal(y1, y2)
    assert norm_err(y1.numpy(), ref, den) <= TOL
    assert int(flags_view(q, ws, M, K).count_nonzero()) == 0


@pytest.mark.parametrize("fmt,N,K", [("q4_k", 17408, 5120), ("q4_k", 5120, 17408), ("q5_k", 17408, 5120),
                                     ("q6_k", 10240, 5120)])
def test_kquant_full_size_sampled(q, fmt, N, K):
    """The 27B MLP matrices and the Q6_K fused attn_qkv [10240, 5120] at M = 512 (the
    prefill configuration), sampled rows."""
    M, seed = 512, 61
    packed = device_matrix(q, fmt, seed, N, K)
    rows = sample_rows(N, 24, seed)
    Dr = host_rows_dequant(fmt, seed, rows, N, K)
    x = synth.activations(seed + 1, M, K)
    ref, den = oracle.gemv_f64(Dr, synth.bf16_bits(x))
    ws = q.workspace(q.QMV_ENTRY_KQUANT, fmt, M, N, K)
    y = q.qmv_gemm_kquant(fmt, packed, x.cuda(), N, K, ws)
    got = y[:, torch.from_numpy(rows).cuda()].cpu().numpy()
    assert q.qmv_device_status() == 0
    assert norm_err(got, ref, den) <= TOL
    assert int(flags_view(q, ws, M, K).count_nonzero()) == 0


def test_kquant_errors(q):
    N, K, M = 256, 512, 130
    W, canon = host_matrix("q4_k", 63, N, K)
    packed = q.qmv_pack("q4_k", torch.from_numpy(canon).cuda(), N, K)
    x = synth.activations(63, M, K).cuda()
    ws = q.workspace(q.QMV_ENTRY_KQUANT, "q4_k", M, N, K)
    for fmt in ("q8_0", "nvfp4", "fp8_row", "iq4_xs", "iq2_s"):
        with pytest.raises(q.QmvError) as ei:
            q.qmv_gemm_kquant(fmt, packed, x, N, K, ws)
        assert ei.value.status == 3
    with pytest.raises(q.QmvError) as ei:
        q.qmv_gemm_kquant("q4_k", packed, x, N, K, ws[:4096])
    assert ei.value.status == 8
    assert q.qmv_workspace_size(q.QMV_ENTRY_KQUANT, "q4_k", M, N, 300) == 0
    # arguments that disagree with the packed header: detected on the device, y untouched
    y = torch.full((M, N - 128), 3.0, device="cuda")
    q.qmv_device_status(reset=True)
    q.qmv_gemm_kquant("q4_k", packed, x, N - 128, K, ws, y=y)
    assert q.qmv_device_status(reset=True) == 5
    assert bool((y == 3.0).all())
    assert int(flags_view(q, ws, M, K).count_nonzero()) == 0


@pytest.mark.parametrize("M", [1, 130])
def test_kquant_q6k_any_bytes(q, M):
    """Q6_K blocks of arbitrary bytes (every int8 scale, -128 included, and every code)
    with a positive fp16 d: the two-term scale split stays exact."""
    N, K = 256, 1024
    rng = np.random.default_rng(91 + M)
    blocks = rng.integers(0, 256, size=(N * K // 256, 210), dtype=np.uint8)
    d = rng.uniform(1e-4, 1e-3, size=N * K // 256).astype(np.float16).view(np.uint16)
    blocks[:, 208] = d & 0xFF
    blocks[:, 209] = d >> 8
    blocks[0, 192:208] = np.array([0x80, 0x7F] * 8, dtype=np.uint8)      # scales -128, 127
    canon = blocks.reshape(-1)
    D = host_dequant("q6_k", canon, N, K)
    x = synth.activations(93, M, K)
    ref, den = oracle.gemv_f64(D, synth.bf16_bits(x))
    packed = q.qmv_pack("q6_k", torch.from_numpy(canon).cuda(), N, K)
    ws = q.workspace(q.QMV_ENTRY_KQUANT, "q6_k", M, N, K)
    y = q.qmv_gemm_kquant("q6_k", packed, x.cuda(), N, K, ws).cpu().numpy()
    assert q.qmv_device_status() == 0
    assert norm_err(y, ref, den) <= TOL
