"""GPU: one accumulation order for every batch size (bitwise M-invariance).

Verification rows of a speculative step (M = 2..8) must round exactly like
single-token decode ("Qwen3.8-27B on one Tenstorrent P150", section "Quality, then
a better quant", the exact-speculation fix among the two exactness fixes of Oct 3).
The library's order of the fp32 sums depends on the matrix shape and the SM count
only (fixed cells of the slab sequence, fixed per-unit combinations), never on M,
the grid, the routing of other tokens, or the entry point's workspace. So every row
of an M-row call must equal the one-row call on that row bit for bit:
torch.equal, not a tolerance. Covered: all six formats at the Qwen3.8-27B shapes,
the fused gate|up SwiGLU, the 288-expert tower at M in {1, 4, 8} (gate with shared
x, down with one x row per pair) and its fused form, and the no-workspace entry.
"""
import pytest
import torch

import synth
from cases import device_matrix

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
    ("q8_0", 512, 1024),                 # the tiny configuration
    ("q8_0", QWEN_HIDDEN, QWEN_HIDDEN),
    ("iq4_xs", 4096, 2048),              # a 288-expert model's down projection, one expert
    ("iq3_s", 4096, 2048),
    ("iq2_s", 2048, 4096),               # its gate / up
]


@pytest.fixture(scope="module")
def q():
    import block_quantized_weight_fly_gb300 as q
    torch.cuda.set_device(0)
    q.qmv_device_status(reset=True)
    return q


def _rows_equal(q, call, x, M_list=(8, 3)):
    """call(x_rows) -> y [rows, ...]; every row of each M-row call equals the one-row call."""
    singles = [call(x[m:m + 1])[0].clone() for m in range(x.shape[0])]
    for M in M_list:
        yM = call(x[:M])
        for m in range(M):
            assert torch.equal(yM[m], singles[m]), (M, m, float((yM[m] - singles[m]).abs().max()))
    torch.cuda.synchronize()
    assert q.qmv_device_status() == 0


@pytest.mark.parametrize("fmt,N,K", DENSE, ids=[f"{f}-{n}x{k}" for f, n, k in DENSE])
def test_gemv_rows_equal_single_row(q, fmt, N, K):
    seed = 900 + N % 97 + K % 89
    packed = device_matrix(q, fmt, seed, N, K)
    x = synth.activations(seed, 8, K).cuda()
    ws = q.workspace(q.QMV_ENTRY_GEMV, fmt, 8, N, K)

    def call(xr):
        y = q.qmv_gemv(fmt, packed, xr, N, K, ws)
        assert int(ws.count_nonzero()) == 0
        return y

    _rows_equal(q, call, x)
    del packed
    torch.cuda.empty_cache()


@pytest.mark.parametrize("fmt", ["q4_k", "q6_k", "nvfp4", "q8_0"])
def test_noalloc_equals_gemv_bitwise(q, fmt):
    """The no-workspace entry adds in the cells of qmv_gemv: same bits at M = 1 and 8."""
    N, K = (QWEN_MLP, QWEN_HIDDEN) if fmt != "q8_0" else (QWEN_HIDDEN, QWEN_HIDDEN)
    packed = device_matrix(q, fmt, 41, N, K)
    x = synth.activations(41, 8, K).cuda()
    for M in (1, 8):
        ws = q.workspace(q.QMV_ENTRY_GEMV, fmt, M, N, K)
        y = q.qmv_gemv(fmt, packed, x[:M], N, K, ws)
        y2 = torch.empty_like(y)
        q.qmv_gemv_noalloc(fmt, packed, x[:M], N, K, y2)
        torch.cuda.synchronize()
        assert torch.equal(y, y2), M
    assert q.qmv_device_status() == 0


@pytest.mark.parametrize("fmt", ["q4_k", "nvfp4", "q6_k"])
def test_swiglu_rows_equal_single_row(q, fmt):
    N, K = QWEN_MLP, QWEN_HIDDEN
    tower = device_matrix(q, fmt, 43, N, K, 2)
    x = synth.activations(43, 8, K).cuda()
    ws = q.workspace(q.QMV_ENTRY_SWIGLU, fmt, 8, N, K)
    _rows_equal(q, lambda xr: q.qmv_gemv_swiglu(fmt, tower, xr, N, K, ws), x)


def _grouped_rows_equal(q, call, ids, x, x_per_pair, topk):
    M = ids.shape[0]
    yM = call(ids, x)
    for t in range(M):
        xr = x[t * topk:(t + 1) * topk] if x_per_pair else x[t:t + 1]
        y1 = call(ids[t:t + 1], xr)
        assert torch.equal(yM[t], y1[0]), (M, t, float((yM[t] - y1[0]).abs().max()))
    torch.cuda.synchronize()
    assert q.qmv_device_status() == 0


@pytest.mark.parametrize("mat", ["gate", "down"])
def test_tower_rows_equal_single_token(q, mat):
    """288-expert Q4_K tower, top-8: each token of an M = 4 and an M = 8 call (experts
    shared with other tokens, in other segment positions) equals that token alone."""
    E, topk = 288, 8
    N, K = (2048, 4096) if mat == "gate" else (4096, 2048)
    x_per_pair = mat == "down"
    tower = device_matrix(q, "q4_k", 47, N, K, E)
    for M in (4, 8):
        ids = torch.from_numpy(synth.expert_ids(470 + M, M, topk, E)).cuda()
        # token 1 routes to token 0's experts in other slots: each of them is one segment
        # with two x rows
        ids[1] = torch.roll(ids[0], 3)
        x = synth.activations(47 + M, M * topk if x_per_pair else M, K).cuda()
        ws = q.workspace(q.QMV_ENTRY_GROUPED, "q4_k", M, N, K, E, topk)

        def call(i, xr):
            y = q.qmv_grouped("q4_k", tower, i.contiguous(), xr.contiguous(), N, K, E, ws, x_per_pair=x_per_pair)
            assert int(ws.count_nonzero()) == 0
            return y

        _grouped_rows_equal(q, call, ids, x, x_per_pair, topk)


@pytest.mark.parametrize("fmt", ["q8_0", "q5_k", "q6_k", "nvfp4", "fp8_row", "iq4_xs", "iq3_s", "iq2_s"])
def test_grouped_rows_equal_single_token_formats(q, fmt):
    E, topk, N, K, M = 24, 8, 640, 2048, 8
    tower = device_matrix(q, fmt, 53, N, K, E)
    ids = torch.from_numpy(synth.expert_ids(53, M, topk, E)).cuda()
    x = synth.activations(53, M, K).cuda()
    ws = q.workspace(q.QMV_ENTRY_GROUPED, fmt, M, N, K, E, topk)
    _grouped_rows_equal(q, lambda i, xr: q.qmv_grouped(fmt, tower, i.contiguous(), xr.contiguous(), N, K, E, ws),
                        ids, x, False, topk)


def test_grouped_swiglu_rows_equal_single_token(q):
    E, topk, N, K, M = 288, 8, 2048, 4096, 8
    tower = device_matrix(q, "q4_k", 59, N, K, 2 * E)
    ids = torch.from_numpy(synth.expert_ids(59, M, topk, E)).cuda()
    x = synth.activations(59, M, K).cuda()
    ws = q.workspace(q.QMV_ENTRY_GROUPED_SWIGLU, "q4_k", M, N, K, E, topk)
    _grouped_rows_equal(q, lambda i, xr: q.qmv_grouped_swiglu("q4_k", tower, i.contiguous(), xr.contiguous(), N, K,
                                                              E, ws), ids, x, False, topk)
