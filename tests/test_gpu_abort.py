"""GPU: the split-K reduction's bounded wait really runs out, and the library
recovers.

Every wait in the stream kernel is bounded and latches QMV_ETIMEOUT instead of
trapping. Here a test hook makes the peers of split row tiles publish nothing, so
each reducer's wait for their partial sums expires after 1 ms: the call must latch
QMV_ETIMEOUT (read through qmv_device_status), nothing faults, and after the
documented recovery (status cleared, workspace zero-filled) the next call gives the
oracle's result. No wait is left without its bound and no GPU fault is provoked:
the waits that run out are plain polls of global memory words.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from cases import TOL, host_dequant, host_matrix, norm_err

pytestmark = pytest.mark.gpu

QMV_ETIMEOUT = 6


@pytest.fixture(scope="module")
def q():
    import block_quantized_weight_fly_gb300 as q
    torch.cuda.set_device(0)
    q.qmv_device_status(reset=True)
    yield q
    q.qmv_debug_split_k_fault(0)


def _case(q, fmt, N, K, M, seed):
    W, canon = host_matrix(fmt, seed, N, K)
    D = host_dequant(fmt, canon, N, K)
    x = synth.activations(seed, M, K)
    ref, den = oracle.gemv_f64(D, synth.bf16_bits(x))
    packed = q.qmv_pack(fmt, torch.from_numpy(canon).cuda(), N, K)
    return packed, x.cuda(), ref, den


@pytest.mark.parametrize("M", [1, 8])
def test_gemv_peer_wait_times_out_then_recovers(q, M):
    # 2 row tiles x 20 k-groups: every row tile is split among many CTAs
    fmt, N, K = "q4_k", 256, 5120
    packed, x, ref, den = _case(q, fmt, N, K, M, 61)
    ws = q.workspace(q.QMV_ENTRY_GEMV, fmt, M, N, K)
    q.qmv_device_status(reset=True)
    q.qmv_debug_split_k_fault(1, 1_000_000)           # 1 ms
    try:
        q.qmv_gemv(fmt, packed, x, N, K, ws)
        st = q.qmv_device_status(reset=True)
    finally:
        q.qmv_debug_split_k_fault(0)
    assert st == QMV_ETIMEOUT
    ws.zero_()
    y = q.qmv_gemv(fmt, packed, x, N, K, ws).cpu().numpy()
    assert q.qmv_device_status() == 0
    assert norm_err(y, ref, den) <= TOL
    assert int(ws.count_nonzero()) == 0


def test_grouped_peer_wait_times_out_then_recovers(q):
    fmt, N, K, E, M, topk = "q4_k", 256, 4096, 6, 1, 2
    W, canon = host_matrix(fmt, 63, N, K, E)
    D = host_dequant(fmt, canon, N, K, E)
    ids = synth.expert_ids(63, M, topk, E)
    x = synth.activations(63, M, K)
    Y, Dn = oracle.grouped_f64(lambda e: D[e * N:(e + 1) * N], ids, synth.bf16_bits(x), False)
    tower = q.qmv_pack(fmt, torch.from_numpy(canon).cuda(), N, K, E)
    ws = q.workspace(q.QMV_ENTRY_GROUPED, fmt, M, N, K, E, topk)
    idd = torch.from_numpy(ids).cuda()
    q.qmv_device_status(reset=True)
    q.qmv_debug_split_k_fault(1, 1_000_000)
    try:
        q.qmv_grouped(fmt, tower, idd, x.cuda(), N, K, E, ws)
        st = q.qmv_device_status(reset=True)
    finally:
        q.qmv_debug_split_k_fault(0)
    assert st == QMV_ETIMEOUT
    ws.zero_()
    y = q.qmv_grouped(fmt, tower, idd, x.cuda(), N, K, E, ws).cpu().numpy()
    assert q.qmv_device_status() == 0
    assert norm_err(y, Y, Dn) <= TOL


def test_abandoned_gather_leaves_pieces_and_zero_fill_recovers(q):
    """Mode 2: reducers give up at once, so the peers' partial sums stay in the
    workspace (non-zero words) -- the state the header's 'zero-fill after a status
    error' rule is for. The call after the zero-fill is exact again."""
    fmt, N, K, M = "q4_k", 256, 5120, 1
    packed, x, ref, den = _case(q, fmt, N, K, M, 65)
    ws = q.workspace(q.QMV_ENTRY_GEMV, fmt, M, N, K)
    q.qmv_device_status(reset=True)
    q.qmv_debug_split_k_fault(2)
    try:
        q.qmv_gemv(fmt, packed, x, N, K, ws)
        st = q.qmv_device_status(reset=True)
    finally:
        q.qmv_debug_split_k_fault(0)
    assert st == QMV_ETIMEOUT
    assert int(ws.count_nonzero()) > 0
    ws.zero_()
    y = q.qmv_gemv(fmt, packed, x, N, K, ws).cpu().numpy()
    assert q.qmv_device_status() == 0
    assert norm_err(y, ref, den) <= TOL
    assert np.isfinite(y).all()
