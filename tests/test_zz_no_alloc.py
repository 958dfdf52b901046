"""qmv_gemv_noalloc (the library's built-in scratch in place of a workspace)
against qmv_gemv through the C ABI, two calls in a row each.

Collected last on purpose: it must pass alone in a fresh process and after every
other test has used the library (and its scratch-free entry points).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from cases import TOL, host_dequant, host_matrix, norm_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import block_quantized_weight_fly_gb300 as q
    torch.cuda.set_device(0)
    q.qmv_device_status(reset=True)
    return q


@pytest.mark.parametrize("fmt,N,K", [("q4_k", 1000, 2048), ("nvfp4", 300, 512), ("q8_0", 129, 768)])
@pytest.mark.parametrize("M", [1, 8, 3])
def test_noalloc_matches_gemv_two_calls(q, fmt, N, K, M):
    W, canon = host_matrix(fmt, 31, N, K)
    D = host_dequant(fmt, canon, N, K)
    packed = q.qmv_pack(fmt, torch.from_numpy(canon).cuda(), N, K)
    ws = q.workspace(q.QMV_ENTRY_GEMV, fmt, M, N, K)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    for call, seed in enumerate((41, 42)):                 # two calls in a row, new x each
        x = synth.activations(seed, M, K)
        _, den = oracle.gemv_f64(D, synth.bf16_bits(x))
        xd = x.cuda()
        y_ref = q.qmv_gemv(fmt, packed, xd, N, K, ws).cpu().numpy()
        y.fill_(float("nan"))
        q.qmv_gemv_noalloc(fmt, packed, xd, N, K, y)
        assert q.qmv_last_route() == q.FORMATS[fmt] * 100 + (1 if M == 1 else 2)
        got = y.cpu().numpy()
        assert q.qmv_device_status() == 0
        assert np.isfinite(got).all(), f"call {call}: outputs left unwritten"
        e = norm_err(got, y_ref, den)
        assert e <= TOL, f"call {call}: {e}"


def test_noalloc_argument_errors(q):
    N, K = 256, 512
    _, canon = host_matrix("q4_k", 37, N, K)
    packed = q.qmv_pack("q4_k", torch.from_numpy(canon).cuda(), N, K)
    x = synth.activations(37, 1, K).cuda()
    y = torch.empty((1, N), dtype=torch.float32, device="cuda")
    with pytest.raises(q.QmvError) as ei:
        q.qmv_gemv_noalloc("q4_k", packed, x, N, 300, y)     # K not a multiple of 256
    assert ei.value.status == 3
    x9 = synth.activations(37, 9, K).cuda()
    with pytest.raises(q.QmvError) as ei:
        q.qmv_gemv_noalloc("q4_k", packed, x9, N, K, torch.empty((9, N), device="cuda"))
    assert ei.value.status == 1
    # the scratch this GPU needs (one CTA per SM, 128 rows x 8 words each at M > 1)
    # fits the built-in array
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    need = -(-(sms * 128 * 8 * 4) // 256) * 256
    assert need <= (1 << 20), (sms, need)
