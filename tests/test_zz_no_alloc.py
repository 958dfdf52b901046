"""qmv_gemv_noalloc: the decode GEMV for callers that cannot hand the library any
device memory per call (an engine whose allocator already holds the whole device
for its own pool, a plugin interface that passes only input and output pointers).
Its split-K scratch is an array built into the library; it allocates nothing.

Checked through the C ABI, two calls in a row each: against the CPU oracle within
the tolerance, and against qmv_gemv bit for bit (both add in the same cells). Also:
a call that starts on scratch a failed call left dirty, the largest scratch this GPU
uses (M = 8 on the 27B gate shape, every SM busy) against the oracle, and argument
errors.

Collected last on purpose: it must pass alone in a fresh process and after every
other test has used the library.
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


@pytest.mark.parametrize("fmt,N,K", [("q4_k", 1000, 2048), ("nvfp4", 300, 512), ("q8_0", 129, 768)])
@pytest.mark.parametrize("M", [1, 8, 3])
def test_noalloc_matches_oracle_and_gemv_two_calls(q, fmt, N, K, M):
    W, canon = host_matrix(fmt, 31, N, K)
    D = host_dequant(fmt, canon, N, K)
    packed = q.qmv_pack(fmt, torch.from_numpy(canon).cuda(), N, K)
    ws = q.workspace(q.QMV_ENTRY_GEMV, fmt, M, N, K)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    for call, seed in enumerate((41, 42)):                 # two calls in a row, new x each
        x = synth.activations(seed, M, K)
        ref, den = oracle.gemv_f64(D, synth.bf16_bits(x))
        xd = x.cuda()
        y_gemv = q.qmv_gemv(fmt, packed, xd, N, K, ws)
        y.fill_(float("nan"))
        q.qmv_gemv_noalloc(fmt, packed, xd, N, K, y)
        assert q.qmv_last_route() == q.FORMATS[fmt] * 100 + (1 if M == 1 else 2)
        got = y.cpu().numpy()
        assert q.qmv_device_status() == 0
        assert np.isfinite(got).all(), f"call {call}: outputs left unwritten"
        e = norm_err(got, ref, den)
        assert e <= TOL, f"call {call}: {e}"
        assert torch.equal(y, y_gemv), f"call {call}: differs from qmv_gemv"


def test_noalloc_after_a_failed_call_left_scratch_dirty(q):
    """A call whose reducers gave up (test hook, mode 2) leaves partial sums in the
    built-in scratch; the next call clears what it uses first and is exact."""
    fmt, N, K, M = "q4_k", 256, 5120, 1
    W, canon = host_matrix(fmt, 71, N, K)
    D = host_dequant(fmt, canon, N, K)
    packed = q.qmv_pack(fmt, torch.from_numpy(canon).cuda(), N, K)
    x = synth.activations(71, M, K)
    ref, den = oracle.gemv_f64(D, synth.bf16_bits(x))
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    q.qmv_device_status(reset=True)
    q.qmv_debug_split_k_fault(2)
    try:
        q.qmv_gemv_noalloc(fmt, packed, x.cuda(), N, K, y)
        st = q.qmv_device_status(reset=True)
    finally:
        q.qmv_debug_split_k_fault(0)
    assert st == QMV_ETIMEOUT
    for _ in range(2):
        y.fill_(float("nan"))
        q.qmv_gemv_noalloc(fmt, packed, x.cuda(), N, K, y)
        assert q.qmv_device_status() == 0
        assert norm_err(y.cpu().numpy(), ref, den) <= TOL


def test_noalloc_largest_scratch_on_this_gpu(q):
    """M = 8 on the 27B gate shape [17408, 5120]: the row tiles spread over every SM,
    so the call uses the most scratch the entry needs on this GPU; every output
    against the oracle."""
    fmt, N, K, M = "q4_k", 17408, 5120, 8
    W = synth.weights(73, N, K, device="cuda").cpu().numpy()   # the generator's bits, drawn faster
    canon = oracle.encode(fmt, W)
    del W
    D = host_dequant(fmt, canon, N, K)
    x = synth.activations(73, M, K)
    ref, den = oracle.gemv_f64(D, synth.bf16_bits(x))
    del D
    packed = q.qmv_pack(fmt, torch.from_numpy(canon).cuda(), N, K)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    for _ in range(2):
        y.fill_(float("nan"))
        q.qmv_gemv_noalloc(fmt, packed, x.cuda(), N, K, y)
        assert q.qmv_device_status() == 0
        assert norm_err(y.cpu().numpy(), ref, den) <= TOL


def test_noalloc_argument_errors(q):
    N, K = 256, 512
    _, canon = host_matrix("q4_k", 37, N, K)
    packed = q.qmv_pack("q4_k", torch.from_numpy(canon).cuda(), N, K)
    x = synth.activations(37, 1, K).cuda()
    y = torch.empty((1, N), dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):
        q.qmv_gemv_noalloc("q4_k", packed, x, N, 300, y)     # x rows disagree with K
    xk = synth.activations(37, 1, 320).cuda()
    with pytest.raises(q.QmvError) as ei:
        q.qmv_gemv_noalloc("q4_k", packed, xk, N, 320, torch.empty((1, N), device="cuda"))
    assert ei.value.status == 3                              # K not a multiple of 256
    x9 = synth.activations(37, 9, K).cuda()
    with pytest.raises(q.QmvError) as ei:
        q.qmv_gemv_noalloc("q4_k", packed, x9, N, K, torch.empty((9, N), device="cuda"))
    assert ei.value.status == 1
    with pytest.raises(ValueError):
        q.qmv_gemv_noalloc("q4_k", packed, x, N, K, torch.empty((1, N - 1), device="cuda"))   # y too short
    with pytest.raises(ValueError):
        q.qmv_gemv_noalloc("q4_k", packed, x, N, K, torch.empty((N, 2), device="cuda")[:, 0])  # strided y
