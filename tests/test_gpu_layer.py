"""GPU: the dense MLP layer in one launch (qmv_mlp_layer).

y = bf16(silu(x Wg^T) * (x Wu^T)) Wd^T. Checked:
- bit for bit against the same computation from the separate entry points
  (qmv_gemv_swiglu, a bf16 round-to-nearest-even of h, qmv_gemv): the layer uses the
  same cells in both passes, so the results must be identical;
- against the CPU oracle: its fp64 gate and up dots, its SwiGLU, its bf16 rounding
  of h, then its fp64 dot with the down matrix. Bound per output: the GEMV tolerance
  on the down pass, plus |w| times the error h can carry into it -- the SwiGLU bound
  of the gate|up pass, and one bf16 step of h wherever h lies that close to a
  rounding midpoint (there the rounding may go either way);
- rows of an M-row call against one-row calls (bit for bit);
- at the Qwen3.8-27B MLP shapes, M = 1 and 8, against the separate entry points.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from cases import TOL, device_matrix, host_dequant, host_matrix

pytestmark = pytest.mark.gpu

QWEN_HIDDEN, QWEN_MLP = 5120, 17408


@pytest.fixture(scope="module")
def q():
    import block_quantized_weight_fly_gb300 as q
    torch.cuda.set_device(0)
    q.qmv_device_status(reset=True)
    return q


def _layer(q, fmt, gu, dn, x, N_ff, K_h, ws):
    y = q.qmv_mlp_layer(fmt, gu, dn, x, N_ff, K_h, ws)
    assert q.qmv_last_route() == q.FORMATS[fmt] * 100 + 12
    return y


def _separate(q, fmt, gu, dn, x, N_ff, K_h):
    M = x.shape[0]
    ws1 = q.workspace(q.QMV_ENTRY_SWIGLU, fmt, M, N_ff, K_h)
    h = q.qmv_gemv_swiglu(fmt, gu, x, N_ff, K_h, ws1)
    ws2 = q.workspace(q.QMV_ENTRY_GEMV, fmt, M, K_h, N_ff)
    return q.qmv_gemv(fmt, dn, h.to(torch.bfloat16), K_h, N_ff, ws2)


def _bf16_step(h):
    """the spacing of bf16 values around |h| (fp64)"""
    a = np.maximum(np.abs(h), 2.0**-126)
    return np.ldexp(1.0, np.floor(np.log2(a)).astype(int) - 7)


@pytest.mark.parametrize("fmt", ["q4_k", "q6_k", "nvfp4", "q8_0", "iq4_xs"])
@pytest.mark.parametrize("M", [1, 3, 8])
def test_layer_equals_separate_calls_and_oracle(q, fmt, M):
    N_ff, K_h = 768, 512
    _, cgu = host_matrix(fmt, 81, N_ff, K_h, 2)          # gate = expert 0, up = expert 1
    _, cdn = host_matrix(fmt, 83, K_h, N_ff)
    gu = q.qmv_pack(fmt, torch.from_numpy(cgu).cuda(), N_ff, K_h, 2)
    dn = q.qmv_pack(fmt, torch.from_numpy(cdn).cuda(), K_h, N_ff)
    x = synth.activations(85 + M, M, K_h)
    xd = x.cuda()
    ws = q.workspace(q.QMV_ENTRY_MLP_LAYER, fmt, M, N_ff, K_h)
    y = _layer(q, fmt, gu, dn, xd, N_ff, K_h, ws)
    y2 = _layer(q, fmt, gu, dn, xd, N_ff, K_h, ws)         # a second call on the same workspace
    ys = _separate(q, fmt, gu, dn, xd, N_ff, K_h)
    torch.cuda.synchronize()
    assert q.qmv_device_status() == 0
    assert torch.equal(y, ys) and torch.equal(y2, ys)
    # the oracle
    Dgu = host_dequant(fmt, cgu, N_ff, K_h, 2)
    Ddn = host_dequant(fmt, cdn, K_h, N_ff)
    xb = synth.bf16_bits(x)
    g, dg = oracle.gemv_f64(Dgu[:N_ff], xb)
    u, du = oracle.gemv_f64(Dgu[N_ff:], xb)
    h = oracle.swiglu_f64(g, u)
    hb = oracle.f64_to_bf16_array(h)
    yref, den = oracle.gemv_f64(Ddn, hb)
    s = np.abs(oracle.swiglu_f64(g, np.ones_like(g)))
    eh = 1.1 * TOL * dg * (np.abs(u) + TOL * du) + s * TOL * du + 1e-6 * np.abs(h) + 1e-30   # |h_gpu - h|
    step = _bf16_step(h)
    # where the exact h is within eh of a rounding midpoint, the two roundings may differ
    near = np.abs(np.abs(h) - (np.floor(np.abs(h) / step) + 0.5) * step) <= eh
    dh = eh + np.where(near, step, 0.0)                  # |bf16(h_gpu) - bf16(h)| at most
    bound = TOL * den + (np.abs(Ddn.astype(np.float64)) @ dh.T).T
    err = np.abs(y.cpu().numpy().astype(np.float64) - yref)
    assert np.all(err <= bound), float((err / bound).max())


def test_layer_rows_equal_single_rows(q):
    fmt, N_ff, K_h = "q4_k", 1024, 768
    _, cgu = host_matrix(fmt, 87, N_ff, K_h, 2)
    _, cdn = host_matrix(fmt, 89, K_h, N_ff)
    gu = q.qmv_pack(fmt, torch.from_numpy(cgu).cuda(), N_ff, K_h, 2)
    dn = q.qmv_pack(fmt, torch.from_numpy(cdn).cuda(), K_h, N_ff)
    x = synth.activations(91, 8, K_h).cuda()
    singles = []
    for m in range(8):
        ws = q.workspace(q.QMV_ENTRY_MLP_LAYER, fmt, 1, N_ff, K_h)
        singles.append(_layer(q, fmt, gu, dn, x[m:m + 1], N_ff, K_h, ws)[0].clone())
    for M in (8, 3):
        ws = q.workspace(q.QMV_ENTRY_MLP_LAYER, fmt, M, N_ff, K_h)
        yM = _layer(q, fmt, gu, dn, x[:M], N_ff, K_h, ws)
        for m in range(M):
            assert torch.equal(yM[m], singles[m]), (M, m)
    assert q.qmv_device_status() == 0


@pytest.mark.parametrize("fmt", ["q4_k", "iq2_s"])
def test_layer_full_size(q, fmt):
    """The Qwen3.8-27B MLP (gate, up [17408, 5120], down [5120, 17408]) at M = 1 and 8,
    every output against the separate entry points, bit for bit."""
    gu = device_matrix(q, fmt, 93, QWEN_MLP, QWEN_HIDDEN, 2)
    dn = device_matrix(q, fmt, 95, QWEN_HIDDEN, QWEN_MLP)
    for M in (1, 8):
        x = synth.activations(97 + M, M, QWEN_HIDDEN).cuda()
        ws = q.workspace(q.QMV_ENTRY_MLP_LAYER, fmt, M, QWEN_MLP, QWEN_HIDDEN)
        y = _layer(q, fmt, gu, dn, x, QWEN_MLP, QWEN_HIDDEN, ws)
        ys = _separate(q, fmt, gu, dn, x, QWEN_MLP, QWEN_HIDDEN)
        torch.cuda.synchronize()
        assert q.qmv_device_status() == 0
        assert torch.equal(y, ys), M
        assert bool(torch.isfinite(y).all())
    del gu, dn
    torch.cuda.empty_cache()


def test_layer_errors(q):
    fmt, N_ff, K_h, M = "q4_k", 512, 256, 2
    _, cgu = host_matrix(fmt, 99, N_ff, K_h, 2)
    _, cdn = host_matrix(fmt, 101, K_h, N_ff)
    gu = q.qmv_pack(fmt, torch.from_numpy(cgu).cuda(), N_ff, K_h, 2)
    dn = q.qmv_pack(fmt, torch.from_numpy(cdn).cuda(), K_h, N_ff)
    x = synth.activations(99, M, K_h).cuda()
    ws = q.workspace(q.QMV_ENTRY_MLP_LAYER, fmt, M, N_ff, K_h)
    with pytest.raises(q.QmvError) as ei:
        q.qmv_mlp_layer(fmt, gu, dn, x, N_ff, K_h, ws[:1024])
    assert ei.value.status == 8
    with pytest.raises(q.QmvError) as ei:
        q.qmv_mlp_layer(fmt, gu, dn, x, 500, K_h, ws)           # N_ff not a multiple of 256 (down's K)
    assert ei.value.status == 3
    with pytest.raises(ValueError):
        q.qmv_mlp_layer(fmt, gu, dn, x, N_ff, 300, ws)          # x rows disagree with K_h
    # arguments that disagree with the packed headers: detected on the device, status 5
    q.qmv_device_status(reset=True)
    y = q.qmv_mlp_layer(fmt, gu, dn, x, N_ff - 256, K_h, q.workspace(q.QMV_ENTRY_MLP_LAYER, fmt, M, N_ff - 256, K_h))
    torch.cuda.synchronize()
    assert q.qmv_device_status(reset=True) == 5
