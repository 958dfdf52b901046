"""GPU parity of the fused gate|up GEMV with the SwiGLU epilogue.

Expected values: the oracle's fp64 GEMV of the dequantized gate and up rows, then
its fp64 SwiGLU. Bound per output: the GEMV tolerance (1e-5 of sum |w x|) carried
through h = silu(g) u -- |silu'| <= 1.1 -- plus the fp32 rounding of the epilogue
itself (exp, division, product; 1e-6 relative is generous for a few ulp):
  |h - h_ref| <= 1.1 tau den_g (|u_ref| + tau den_u) + |silu(g_ref)| tau den_u + 1e-6 |h_ref|.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from cases import TOL, host_dequant, host_matrix

pytestmark = pytest.mark.gpu

FMTS = ["q4_k", "q5_k", "q6_k", "q8_0", "nvfp4", "fp8_row", "iq4_xs", "iq3_s", "iq2_s"]


@pytest.fixture(scope="module")
def q():
    import block_quantized_weight_fly_gb300 as q
    torch.cuda.set_device(0)
    q.qmv_device_status(reset=True)
    return q


def swiglu_bound(g, dg, u, du, h):
    s = np.abs(oracle.swiglu_f64(g, np.ones_like(g)))
    return 1.1 * TOL * dg * (np.abs(u) + TOL * du) + s * TOL * du + 1e-6 * np.abs(h) + 1e-30


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("N,K", [(300, 512), (1000, 2048), (129, 768), (2000, 1280)])
@pytest.mark.parametrize("M", [1, 3, 8])
def test_swiglu_parity(q, fmt, N, K, M):
    if fmt in ("q4_k", "q5_k", "q6_k", "iq4_xs", "iq3_s", "iq2_s") and K % 256:
        pytest.skip("K-quants and IQ4_XS need K % 256 == 0")
    W, canon = host_matrix(fmt, 61, N, K, 2)                 # gate = expert 0, up = expert 1
    D = host_dequant(fmt, canon, N, K, 2)
    x = synth.activations(67 + M, M, K)
    xb = synth.bf16_bits(x)
    g, dg = oracle.gemv_f64(D[:N], xb)
    u, du = oracle.gemv_f64(D[N:], xb)
    href = oracle.swiglu_f64(g, u)
    tower = q.qmv_pack(fmt, torch.from_numpy(canon).cuda(), N, K, 2)
    ws = q.workspace(q.QMV_ENTRY_SWIGLU, fmt, M, N, K)
    h = q.qmv_gemv_swiglu(fmt, tower, x.cuda(), N, K, ws)
    assert q.qmv_last_route() == q.FORMATS[fmt] * 100 + 9
    h = h.cpu().numpy().astype(np.float64)
    assert q.qmv_device_status() == 0
    err = np.abs(h - href) / swiglu_bound(g, dg, u, du, href)
    assert float(err.max()) <= 1.0, float(err.max())
    assert int(ws.count_nonzero()) == 0


def test_swiglu_full_size_q4k(q):
    """The 27B MLP gate|up at full size, M = 1 and 8, sampled rows."""
    from cases import device_matrix, host_rows_dequant, sample_rows
    N, K, seed = 17408, 5120, 71
    tower = device_matrix(q, "q4_k", seed, N, K, 2)
    rows = sample_rows(N, 40, seed)
    Dg = host_rows_dequant("q4_k", seed, rows, N, K)
    Du = host_rows_dequant("q4_k", seed, N + rows, N, K)
    for M in (1, 8):
        x = synth.activations(seed + M, M, K)
        xb = synth.bf16_bits(x)
        g, dg = oracle.gemv_f64(Dg, xb)
        u, du = oracle.gemv_f64(Du, xb)
        href = oracle.swiglu_f64(g, u)
        ws = q.workspace(q.QMV_ENTRY_SWIGLU, "q4_k", M, N, K)
        h = q.qmv_gemv_swiglu("q4_k", tower, x.cuda(), N, K, ws)
        got = h[:, torch.from_numpy(rows).cuda()].cpu().numpy().astype(np.float64)
        assert q.qmv_device_status() == 0
        err = np.abs(got - href) / swiglu_bound(g, dg, u, du, href)
        assert float(err.max()) <= 1.0, (M, float(err.max()))


# ---------------------------------------------------------------------------
# grouped: the routed experts' gate|up over a 2E-expert tower
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M,topk,E", [(1, 8, 16), (1, 1, 3), (4, 2, 5), (8, 4, 6), (8, 8, 8)])
def test_grouped_swiglu_parity(q, fmt, M, topk, E):
    N, K = 200, 512
    W, canon = host_matrix(fmt, 83, N, K, 2 * E)          # gate experts 0..E-1, up experts E..2E-1
    D = host_dequant(fmt, canon, N, K, 2 * E)
    ids = synth.expert_ids(83 + M + E, M, topk, E)
    x = synth.activations(89 + M, M, K)
    xb = synth.bf16_bits(x)
    g, dg = oracle.grouped_f64(lambda e: D[e * N:(e + 1) * N], ids, xb, False)
    u, du = oracle.grouped_f64(lambda e: D[(E + e) * N:(E + e + 1) * N], ids, xb, False)
    href = oracle.swiglu_f64(g, u)
    tower = q.qmv_pack(fmt, torch.from_numpy(canon).cuda(), N, K, 2 * E)
    ws = q.workspace(q.QMV_ENTRY_GROUPED_SWIGLU, fmt, M, N, K, E, topk)
    h = q.qmv_grouped_swiglu(fmt, tower, torch.from_numpy(ids).cuda(), x.cuda(), N, K, E, ws)
    assert q.qmv_last_route() == q.FORMATS[fmt] * 100 + 10
    h = h.cpu().numpy().astype(np.float64)
    assert q.qmv_device_status() == 0
    err = np.abs(h - href) / swiglu_bound(g, dg, u, du, href)
    assert float(err.max()) <= 1.0, float(err.max())
    assert int(ws.count_nonzero()) == 0


def test_grouped_swiglu_ragged_and_shared(q):
    """K with a ragged last k-group (Q8_0, K = 800), N not a multiple of 128, and
    experts shared by several tokens (8 tokens over 3 experts)."""
    fmt, N, K, E, M, topk = "q8_0", 333, 800, 3, 8, 2
    W, canon = host_matrix(fmt, 97, N, K, 2 * E)
    D = host_dequant(fmt, canon, N, K, 2 * E)
    ids = synth.expert_ids(97, M, topk, E)
    x = synth.activations(97, M, K)
    xb = synth.bf16_bits(x)
    g, dg = oracle.grouped_f64(lambda e: D[e * N:(e + 1) * N], ids, xb, False)
    u, du = oracle.grouped_f64(lambda e: D[(E + e) * N:(E + e + 1) * N], ids, xb, False)
    href = oracle.swiglu_f64(g, u)
    tower = q.qmv_pack(fmt, torch.from_numpy(canon).cuda(), N, K, 2 * E)
    ws = q.workspace(q.QMV_ENTRY_GROUPED_SWIGLU, fmt, M, N, K, E, topk)
    h = q.qmv_grouped_swiglu(fmt, tower, torch.from_numpy(ids).cuda(), x.cuda(), N, K, E, ws)
    h = h.cpu().numpy().astype(np.float64)
    assert q.qmv_device_status() == 0
    err = np.abs(h - href) / swiglu_bound(g, dg, u, du, href)
    assert float(err.max()) <= 1.0, float(err.max())
    assert int(ws.count_nonzero()) == 0


def test_grouped_swiglu_id_range(q):
    """An id naming an up matrix (E <= id < 2E) is outside the gate half: the call
    latches the range status and leaves h as it was."""
    fmt, N, K, E = "q4_k", 128, 256, 3
    W, canon = host_matrix(fmt, 5, N, K, 2 * E)
    tower = q.qmv_pack(fmt, torch.from_numpy(canon).cuda(), N, K, 2 * E)
    ws = q.workspace(q.QMV_ENTRY_GROUPED_SWIGLU, fmt, 1, N, K, E, 2)
    x = synth.activations(5, 1, K).cuda()
    h = torch.full((1, 2, N), 7.0, device="cuda")
    q.qmv_device_status(reset=True)
    q.qmv_grouped_swiglu(fmt, tower, torch.tensor([[0, E]], dtype=torch.int32, device="cuda"), x, N, K, E,
                         ws, h=h)
    assert q.qmv_device_status(reset=True) == 7
    assert bool((h == 7.0).all())
    assert int(ws.count_nonzero()) == 0
