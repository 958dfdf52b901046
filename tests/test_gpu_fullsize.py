"""GPU parity at the full sizes of the benchmark configurations, in the launch
configuration the benchmark times (the same entry points, grids and workspaces).

The weights are generated on the device (seeded generator -> the library's
quantizer -> qmv_pack). The expected values come from the CPU oracle alone: it
regenerates the sampled rows from the same seed, encodes them with its own
encoder, dequantizes them (BlockToFloat) and takes fp64 dots. The library's
quantizer is bit-exact with the oracle's encoder (test_gpu_parity), so both sides
hold the same weights; every sampled output must be within the normalised
tolerance 1e-5.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from cases import TOL, device_matrix, host_dequant, host_rows_dequant, norm_err, sample_rows

pytestmark = pytest.mark.gpu

QWEN_HIDDEN, QWEN_MLP, QWEN_VOCAB = 5120, 17408, 248320

DENSE = [
    ("q4_k", QWEN_MLP, QWEN_HIDDEN),     # gate / up
    ("q4_k", QWEN_HIDDEN, QWEN_MLP),     # down
    ("q5_k", QWEN_MLP, QWEN_HIDDEN),
    ("q5_k", QWEN_HIDDEN, QWEN_MLP),
    ("q6_k", QWEN_VOCAB, QWEN_HIDDEN),   # untied output head
    ("q6_k", 10240, QWEN_HIDDEN),        # fused attn_qkv
    ("nvfp4", QWEN_MLP, QWEN_HIDDEN),
    ("nvfp4", QWEN_HIDDEN, QWEN_MLP),
    ("fp8_row", 6144, QWEN_HIDDEN),
]


@pytest.fixture(scope="module")
def q():
    import block_quantized_weight_fly_gb300 as q
    torch.cuda.set_device(0)
    q.qmv_device_status(reset=True)
    return q


@pytest.mark.parametrize("fmt,N,K", DENSE, ids=[f"{f}-{n}x{k}" for f, n, k in DENSE])
def test_dense_full_size_sampled(q, fmt, N, K):
    seed = 500 + N % 97 + K % 89
    packed = device_matrix(q, fmt, seed, N, K)
    rows = sample_rows(N, 48, seed)
    D = host_rows_dequant(fmt, seed, rows, N, K)
    for M in (1, 8):
        x = synth.activations(seed + M, M, K)
        ref, den = oracle.gemv_f64(D, synth.bf16_bits(x))
        ws = q.workspace(q.QMV_ENTRY_GEMV, fmt, M, N, K)
        y = q.qmv_gemv(fmt, packed, x.cuda(), N, K, ws)
        route = q.qmv_last_route()
        got = y[:, torch.from_numpy(rows).cuda()].cpu().numpy()
        assert q.qmv_device_status() == 0
        assert route == q.FORMATS[fmt] * 100 + (1 if M == 1 else 2)
        e = norm_err(got, ref, den)
        assert e <= TOL, (M, e)
        assert bool(torch.isfinite(y).all())
        assert int(ws.count_nonzero()) == 0
    del packed
    torch.cuda.empty_cache()


@pytest.mark.parametrize("mat", ["gate", "down"])
@pytest.mark.parametrize("M", [1, 4, 8])
def test_tower_full_size_sampled(q, mat, M):
    """Stacked Q4_K tower of 288 experts, top-8 routing drawn without replacement;
    gate [2048, 4096] with x[M, K], down [4096, 2048] with one x row per pair."""
    E, topk = 288, 8
    N, K = (2048, 4096) if mat == "gate" else (4096, 2048)
    x_per_pair = mat == "down"
    seed = 700 + (mat == "down")
    tower = device_matrix(q, "q4_k", seed, N, K, E)
    ids = synth.expert_ids(seed + M, M, topk, E)
    x = synth.activations(seed + 10 * M, M * topk if x_per_pair else M, K)
    ws = q.workspace(q.QMV_ENTRY_GROUPED, "q4_k", M, N, K, E, topk)
    y = q.qmv_grouped("q4_k", tower, torch.from_numpy(ids).cuda(), x.cuda(), N, K, E, ws,
                      x_per_pair=x_per_pair)
    assert q.qmv_last_route() == q.FORMATS["q4_k"] * 100 + 3
    y = y.cpu().numpy()
    assert q.qmv_device_status() == 0
    assert int(ws.count_nonzero()) == 0
    xb = synth.bf16_bits(x)
    rows = sample_rows(N, 16, seed + M)
    # every routed expert of the first tokens, sampled rows of each
    for t in range(min(M, 2)):
        for j in range(topk):
            e = int(ids[t, j])
            D = host_rows_dequant("q4_k", seed, e * N + rows, N, K)
            xr = xb[t * topk + j] if x_per_pair else xb[t]
            ref, den = oracle.gemv_f64(D, xr[None, :])
            err = norm_err(y[t, j, rows][None, :], ref, den)
            assert err <= TOL, (t, j, e, err)
    del tower
    torch.cuda.empty_cache()


@pytest.mark.parametrize("fmt,mat", [("iq4_xs", "down"), ("iq3_s", "down"), ("iq2_s", "gate")])
@pytest.mark.parametrize("M", [1, 8])
def test_codebook_tower_full_size_sampled(q, fmt, mat, M):
    """The 288-expert towers in the codebook formats the pages list for them ("A 320B
    MoE on a free Kaggle TPU", table of formats by layer): IQ2_S gate [2048, 4096]
    (x shared per token), IQ3_S and IQ4_XS down [4096, 2048] (one x row per pair; IQ4_XS
    with a codebook per expert, the grid formats with one grid per tower), top-8;
    sampled rows of every routed expert of the first tokens against the oracle."""
    E, topk = 288, 8
    N, K = (2048, 4096) if mat == "gate" else (4096, 2048)
    x_per_pair = mat == "down"
    seed = 740 + {"iq4_xs": 0, "iq3_s": 1, "iq2_s": 2}[fmt]
    tower = device_matrix(q, fmt, seed, N, K, E)
    ids = synth.expert_ids(seed + M, M, topk, E)
    x = synth.activations(seed + 10 * M, M * topk if x_per_pair else M, K)
    ws = q.workspace(q.QMV_ENTRY_GROUPED, fmt, M, N, K, E, topk)
    y = q.qmv_grouped(fmt, tower, torch.from_numpy(ids).cuda(), x.cuda(), N, K, E, ws, x_per_pair=x_per_pair)
    assert q.qmv_last_route() == q.FORMATS[fmt] * 100 + 3
    y = y.cpu().numpy()
    assert q.qmv_device_status() == 0
    assert int(ws.count_nonzero()) == 0
    xb = synth.bf16_bits(x)
    rows = sample_rows(N, 16, seed + M)
    for t in range(min(M, 2)):
        for j in range(topk):
            e = int(ids[t, j])
            D = host_rows_dequant(fmt, seed, e * N + rows, N, K)
            xr = xb[t * topk + j] if x_per_pair else xb[t]
            ref, den = oracle.gemv_f64(D, xr[None, :])
            err = norm_err(y[t, j, rows][None, :], ref, den)
            assert err <= TOL, (t, j, e, err)
    del tower
    torch.cuda.empty_cache()


def test_tower_swiglu_full_size_sampled(q):
    """Fused gate|up SwiGLU over the 288-expert tower at its full gate/up shape
    [2048, 4096] (a 576-expert tower: gates, then ups), top-8, M = 1 and 8; sampled
    rows of every routed expert of the first tokens against the oracle's fp64
    gate and up dots and its SwiGLU, within the bound carried through silu."""
    E, topk, N, K, seed = 288, 8, 2048, 4096, 720
    tower = device_matrix(q, "q4_k", seed, N, K, 2 * E)
    rows = sample_rows(N, 12, seed)
    for M in (1, 8):
        ids = synth.expert_ids(seed + M, M, topk, E)
        x = synth.activations(seed + 10 * M, M, K)
        ws = q.workspace(q.QMV_ENTRY_GROUPED_SWIGLU, "q4_k", M, N, K, E, topk)
        h = q.qmv_grouped_swiglu("q4_k", tower, torch.from_numpy(ids).cuda(), x.cuda(), N, K, E, ws)
        assert q.qmv_last_route() == q.FORMATS["q4_k"] * 100 + 10
        h = h.cpu().numpy().astype(np.float64)
        assert q.qmv_device_status() == 0
        assert int(ws.count_nonzero()) == 0
        xb = synth.bf16_bits(x)
        for t in range(min(M, 2)):
            for j in range(topk):
                e = int(ids[t, j])
                g, dg = oracle.gemv_f64(host_rows_dequant("q4_k", seed, e * N + rows, N, K), xb[t][None, :])
                u, du = oracle.gemv_f64(host_rows_dequant("q4_k", seed, (E + e) * N + rows, N, K), xb[t][None, :])
                href = oracle.swiglu_f64(g, u)
                s = np.abs(oracle.swiglu_f64(g, np.ones_like(g)))
                bound = 1.1 * TOL * dg * (np.abs(u) + TOL * du) + s * TOL * du + 1e-6 * np.abs(href) + 1e-30
                err = np.abs(h[t, j, rows][None, :] - href) / bound
                assert float(err.max()) <= 1.0, (M, t, j, e, float(err.max()))
    del tower
    torch.cuda.empty_cache()


@pytest.mark.parametrize("mat", ["gate", "up", "down"])
def test_q4k_mlp_whole_output(q, mat):
    """The headline configuration's whole output, not a sample: the Q4_K MLP matrices
    of Qwen3.8-27B (gate, up [17408, 5120], down [5120, 17408]) at M = 1 and M = 8,
    every one of the N x M outputs against the oracle's fp64 dots over its own
    encoding and BlockToFloat of the same seeded weights."""
    N, K = (QWEN_MLP, QWEN_HIDDEN) if mat != "down" else (QWEN_HIDDEN, QWEN_MLP)
    seed = {"gate": 811, "up": 812, "down": 813}[mat]
    # the seeded generator gives the same bits on the device as on the host (integer
    # hash, exact fp32); drawing the 89 M weights there only saves time. The encoding,
    # BlockToFloat and dots are the oracle's own.
    W = synth.weights(seed, N, K, device="cuda").cpu().numpy()
    canon = oracle.encode("q4_k", W)
    del W
    D = host_dequant("q4_k", canon, N, K)
    x = synth.activations(seed, 8, K)
    ref, den = oracle.gemv_f64(D, synth.bf16_bits(x))
    del D
    packed = q.qmv_pack("q4_k", torch.from_numpy(canon).cuda(), N, K)
    for M in (1, 8):
        ws = q.workspace(q.QMV_ENTRY_GEMV, "q4_k", M, N, K)
        y = q.qmv_gemv("q4_k", packed, x[:M].cuda(), N, K, ws).cpu().numpy()
        assert q.qmv_device_status() == 0
        assert y.shape == (M, N)
        e = norm_err(y, ref[:M], den[:M])
        assert e <= TOL, (M, e)
    del packed
    torch.cuda.empty_cache()
