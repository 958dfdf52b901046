"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

- quantizer: canonical bytes bit-exact with the oracle encoders;
- pack + dequant: BlockToFloat of the packed layout bit-exact with the oracle;
- GEMV and grouped GEMV: every output within the normalised tolerance 1e-5 of the
  oracle's fp64 dot product of the dequantized weights, on shapes spanning several
  row tiles, several k-groups and ragged tails, at M = 1..8;
- error statuses, determinism, guard words around the output, route ids.
Full-size shapes are in test_gpu_fullsize.py.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from cases import (TOL, grid, host_dequant, host_matrix, norm_err, tensor_scale)

pytestmark = pytest.mark.gpu

FMTS = ["q8_0", "q4_k", "q5_k", "q6_k", "nvfp4", "fp8_row", "iq4_xs", "iq3_s", "iq2_s"]


@pytest.fixture(scope="module")
def q():
    import block_quantized_weight_fly_gb300 as q
    torch.cuda.set_device(0)
    q.qmv_device_status(reset=True)
    return q


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _kq(fmt):
    """formats whose K granule is 256"""
    return fmt in ("q4_k", "q5_k", "q6_k", "iq4_xs", "iq3_s", "iq2_s")


# ---------------------------------------------------------------------------
# quantizer
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("fmt", FMTS)
def test_quantize_bit_exact(q, fmt):
    rows, K = 24, 1024
    W = synth.weights(3, rows, K).numpy()
    W[0] = 0.0
    W[1] = -np.abs(W[1])
    W[2, :256] = 0.0123
    W[3] *= 1e-4
    W[4, 5] = 0.5                                      # an outlier
    if fmt in ("iq4_xs", "iq3_s", "iq2_s"):
        cb = synth.codebook(3) if fmt == "iq4_xs" else grid(fmt, 3)
        want = oracle.encode(fmt, W, codebook=cb)
        got = q.qmv_quantize_codebook(fmt, torch.from_numpy(W).cuda(), cb).cpu().numpy()
    else:
        want = oracle.encode(fmt, W, tensor_scale(fmt))
        got = q.qmv_quantize(fmt, torch.from_numpy(W).cuda(), tensor_scale(fmt)).cpu().numpy()
    torch.cuda.synchronize()
    assert got.shape == want.shape
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, f"{bad.size} bytes differ, first at {bad[:8]}"


# ---------------------------------------------------------------------------
# pack + dequant
# ---------------------------------------------------------------------------
SHAPES_DQ = [(300, 512, 1), (128, 256, 1), (7, 1024, 1), (200, 512, 3)]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("N,K,E", SHAPES_DQ + [(129, 96, 2)])
def test_dequant_bit_exact(q, fmt, N, K, E):
    if _kq(fmt) and K % 256:
        pytest.skip("K-quants need K % 256 == 0")
    W, canon = host_matrix(fmt, 5, N, K, E)
    want = host_dequant(fmt, canon, N, K, E)
    packed = q.qmv_pack(fmt, torch.from_numpy(canon).cuda(), N, K, E)
    got = q.qmv_dequant(fmt, packed, N, K, E).cpu().numpy()
    assert q.qmv_device_status() == 0
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    # a row window in the middle of the tower
    r0, nr = min(N * E - 1, 3), min(N * E - 3, 50)
    got2 = q.qmv_dequant(fmt, packed, N, K, E, row0=r0, rows=nr).cpu().numpy()
    assert np.array_equal(got2.view(np.uint32), want[r0:r0 + nr].view(np.uint32))


# ---------------------------------------------------------------------------
# GEMV
# ---------------------------------------------------------------------------
SHAPES_GEMV = [(512, 1024), (300, 512), (1000, 2048), (129, 768), (1, 256), (2000, 1280)]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("N,K", SHAPES_GEMV)
@pytest.mark.parametrize("M", [1, 3, 8])
def test_gemv_parity(q, fmt, N, K, M):
    if _kq(fmt) and K % 256:
        pytest.skip("K-quants need K % 256 == 0")
    W, canon = host_matrix(fmt, 11, N, K)
    D = host_dequant(fmt, canon, N, K)
    x = synth.activations(11, M, K)
    ref, den = oracle.gemv_f64(D, synth.bf16_bits(x))
    packed = q.qmv_pack(fmt, torch.from_numpy(canon).cuda(), N, K)
    ws = q.workspace(q.QMV_ENTRY_GEMV, fmt, M, N, K)
    y = q.qmv_gemv(fmt, packed, x.cuda(), N, K, ws)
    route = q.qmv_last_route()
    y = y.cpu().numpy()
    assert q.qmv_device_status() == 0
    assert route == q.FORMATS[fmt] * 100 + (1 if M == 1 else 2)
    e = norm_err(y, ref, den)
    assert e <= TOL, e
    # the workspace is all zero again for the next call
    assert int(ws.count_nonzero()) == 0


def test_gemv_tiny_config_q8_0(q):
    """Q8_0 [N=512, K=1024], M = 1 bf16 row, seed 0 -- the small configuration."""
    N, K = 512, 1024
    W, canon = host_matrix("q8_0", 0, N, K)
    x = synth.activations(0, 1, K)
    ref, den = oracle.gemv_f64(host_dequant("q8_0", canon, N, K), synth.bf16_bits(x))
    packed = q.qmv_pack("q8_0", torch.from_numpy(canon).cuda(), N, K)
    ws = q.workspace(q.QMV_ENTRY_GEMV, "q8_0", 1, N, K)
    y = q.qmv_gemv("q8_0", packed, x.cuda(), N, K, ws).cpu().numpy()
    assert q.qmv_device_status() == 0
    assert norm_err(y, ref, den) <= TOL


@pytest.mark.parametrize("fmt", ["q4_k", "nvfp4", "iq4_xs", "iq2_s"])
def test_gemv_deterministic_and_guarded(q, fmt):
    N, K, M = 1000, 2048, 4
    W, canon = host_matrix(fmt, 13, N, K)
    packed = q.qmv_pack(fmt, torch.from_numpy(canon).cuda(), N, K)
    x = synth.activations(13, M, K).cuda()
    ws = q.workspace(q.QMV_ENTRY_GEMV, fmt, M, N, K)
    canary = -1.2345e30
    buf = torch.full((M * N + 64,), canary, dtype=torch.float32, device="cuda")
    y1 = q.qmv_gemv(fmt, packed, x, N, K, ws, y=buf[32:32 + M * N].view(M, N)).clone()
    y2 = q.qmv_gemv(fmt, packed, x, N, K, ws)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    assert bool((buf[:32] == canary).all()) and bool((buf[32 + M * N:] == canary).all())


@pytest.mark.parametrize("lo,hi", [(-50, 40), (-60, 0), (0, 57)])
@pytest.mark.parametrize("M", [1, 3])
def test_q4k_activation_range(q, lo, hi, M):
    """The Q4_K decoders scale x by 2^63 / 2^67: exact products for
    2^-60 <= |x| < 2^61. Activations with magnitudes spread over that range (per
    element 2^e, e uniform in [lo, hi]) still meet the tolerance."""
    fmt, N, K = "q4_k", 1000, 2048
    W, canon = host_matrix(fmt, 19, N, K)
    z = synth.activations(19, M, K).float()
    rng = np.random.default_rng((lo + 100) * 1000 + hi + 100 + M)
    e = torch.from_numpy(rng.integers(lo, hi + 1, size=(M, K)).astype(np.float32))
    x = (z * torch.pow(2.0, e)).to(torch.bfloat16)
    ref, den = oracle.gemv_f64(host_dequant(fmt, canon, N, K), synth.bf16_bits(x))
    packed = q.qmv_pack(fmt, torch.from_numpy(canon).cuda(), N, K)
    ws = q.workspace(q.QMV_ENTRY_GEMV, fmt, M, N, K)
    y = q.qmv_gemv(fmt, packed, x.cuda(), N, K, ws).cpu().numpy()
    assert q.qmv_device_status() == 0
    assert np.isfinite(y).all()
    assert norm_err(y, ref, den) <= TOL


@pytest.mark.parametrize("lo,hi", [(-50, 40), (-60, 0), (0, 52)])
@pytest.mark.parametrize("M", [1, 3])
def test_q6k_activation_range(q, lo, hi, M):
    """The Q6_K decoders scale x by 2^63 .. 2^71: exact products for
    2^-60 <= |x| < 2^56 (|z| < 8 here, so e <= 52)."""
    fmt, N, K = "q6_k", 1000, 2048
    W, canon = host_matrix(fmt, 23, N, K)
    z = synth.activations(23, M, K).float()
    rng = np.random.default_rng((lo + 100) * 1000 + hi + 100 + M)
    e = torch.from_numpy(rng.integers(lo, hi + 1, size=(M, K)).astype(np.float32))
    x = (z * torch.pow(2.0, e)).to(torch.bfloat16)
    ref, den = oracle.gemv_f64(host_dequant(fmt, canon, N, K), synth.bf16_bits(x))
    packed = q.qmv_pack(fmt, torch.from_numpy(canon).cuda(), N, K)
    ws = q.workspace(q.QMV_ENTRY_GEMV, fmt, M, N, K)
    y = q.qmv_gemv(fmt, packed, x.cuda(), N, K, ws).cpu().numpy()
    assert q.qmv_device_status() == 0
    assert np.isfinite(y).all()
    assert norm_err(y, ref, den) <= TOL


@pytest.mark.parametrize("lo,hi", [(-12, 12), (-14, 0), (0, 12)])
@pytest.mark.parametrize("M", [1, 3])
def test_iq4_xs_activation_range(q, lo, hi, M):
    """IQ4_XS feeds x to the MMA in f16: exact for 2^-14 <= |x| < 65504 (|z| < 8 here,
    so e <= 12). Activations spread over that range (per element 2^e) meet the
    tolerance, including the largest codebook offsets."""
    fmt, N, K = "iq4_xs", 1000, 2048
    W, canon = host_matrix(fmt, 29, N, K)
    z = synth.activations(29, M, K).float()
    rng = np.random.default_rng((lo + 100) * 1000 + hi + 100 + M)
    e = torch.from_numpy(rng.integers(lo, hi + 1, size=(M, K)).astype(np.float32))
    x = (z * torch.pow(2.0, e)).to(torch.bfloat16)
    ref, den = oracle.gemv_f64(host_dequant(fmt, canon, N, K), synth.bf16_bits(x))
    packed = q.qmv_pack(fmt, torch.from_numpy(canon).cuda(), N, K)
    ws = q.workspace(q.QMV_ENTRY_GEMV, fmt, M, N, K)
    y = q.qmv_gemv(fmt, packed, x.cuda(), N, K, ws).cpu().numpy()
    assert q.qmv_device_status() == 0
    assert np.isfinite(y).all()
    assert norm_err(y, ref, den) <= TOL


# ---------------------------------------------------------------------------
# grouped
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M,topk,E", [(1, 8, 10), (4, 8, 10), (8, 8, 12), (3, 2, 3), (8, 1, 2)])
@pytest.mark.parametrize("x_per_pair", [False, True])
def test_grouped_parity(q, fmt, M, topk, E, x_per_pair):
    N, K = 200, 512
    W, canon = host_matrix(fmt, 19, N, K, E)
    D = host_dequant(fmt, canon, N, K, E)
    ids = synth.expert_ids(19 + M, M, topk, E)
    x = synth.activations(19, M * topk if x_per_pair else M, K)
    Y, Dn = oracle.grouped_f64(lambda e: D[e * N:(e + 1) * N], ids, synth.bf16_bits(x), x_per_pair)
    tower = q.qmv_pack(fmt, torch.from_numpy(canon).cuda(), N, K, E)
    ws = q.workspace(q.QMV_ENTRY_GROUPED, fmt, M, N, K, E, topk)
    y = q.qmv_grouped(fmt, tower, torch.from_numpy(ids).cuda(), x.cuda(), N, K, E, ws,
                      x_per_pair=x_per_pair)
    assert q.qmv_last_route() == q.FORMATS[fmt] * 100 + 3
    y = y.cpu().numpy()
    assert q.qmv_device_status() == 0
    assert norm_err(y, Y, Dn) <= TOL
    assert int(ws.count_nonzero()) == 0


# ---------------------------------------------------------------------------
# errors
# ---------------------------------------------------------------------------
def test_errors(q):
    N, K = 256, 512
    W, canon = host_matrix("q4_k", 23, N, K)
    packed = q.qmv_pack("q4_k", torch.from_numpy(canon).cuda(), N, K)
    x = synth.activations(23, 1, K).cuda()
    ws = q.workspace(q.QMV_ENTRY_GEMV, "q4_k", 1, N, K)
    with pytest.raises(q.QmvError) as ei:
        q.qmv_gemv("q4_k", packed, x, N, K, ws[:1024])
    assert ei.value.status == 8
    with pytest.raises(q.QmvError) as ei:
        q.qmv_gemv("q4_k", packed, synth.activations(23, 1, 288).cuda(), N, 288, ws)   # K % 256 != 0
    assert ei.value.status == 3
    # arguments that disagree with the packed header: detected on the device
    q.qmv_device_status(reset=True)
    q.qmv_gemv("q4_k", packed, x, N - 128, K, ws)
    assert q.qmv_device_status(reset=True) == 5
    q.qmv_gemv("q6_k", packed, x, N, K, ws)
    assert q.qmv_device_status(reset=True) == 5
    # an expert id outside [0, E)
    E = 3
    _, ct = host_matrix("q4_k", 23, N, K, E)
    tower = q.qmv_pack("q4_k", torch.from_numpy(ct).cuda(), N, K, E)
    ids = torch.tensor([[0, 3]], dtype=torch.int32, device="cuda")
    wsg = q.workspace(q.QMV_ENTRY_GROUPED, "q4_k", 1, N, K, E, 2)
    q.qmv_grouped("q4_k", tower, ids, x, N, K, E, wsg)
    assert q.qmv_device_status(reset=True) == 7
    # and the library still works afterwards
    ref, den = oracle.gemv_f64(host_dequant("q4_k", canon, N, K), synth.bf16_bits(x.cpu()))
    ws2 = q.workspace(q.QMV_ENTRY_GEMV, "q4_k", 1, N, K)
    y = q.qmv_gemv("q4_k", packed, x, N, K, ws2).cpu().numpy()
    assert q.qmv_device_status() == 0
    assert norm_err(y, ref, den) <= TOL


# ---------------------------------------------------------------------------
# NVFP4 activation quantizer (W4A4 prefill input)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("M,K", [(1, 256), (7, 5120), (512, 1024), (3, 48)])
def test_quant_act_nvfp4_bit_exact(q, M, K):
    x = synth.activations(31 + M, M, K)
    xb = synth.bf16_bits(x)
    xf = x.float().numpy()
    xf[0, :16] = 0.0                                  # an all-zero block: scale 0, codes 0
    if K >= 64:
        xf[-1, 16:32] *= 1e-3                         # a small block next to normal ones
        xf[-1, 40] = 300.0                            # an outlier that saturates its block
    x = torch.from_numpy(xf).to(torch.bfloat16)
    xb = synth.bf16_bits(x)
    x_scale = float(np.float32(np.abs(xf).max()) / np.float32(2688.0))
    codes_ref, scales_ref = oracle.quant_act_nvfp4(xb, x_scale)
    codes, scales = q.qmv_quant_act_nvfp4(x.cuda(), x_scale)
    assert q.qmv_last_route() == q.FORMATS["nvfp4"] * 100 + 8
    assert np.array_equal(scales.cpu().numpy(), scales_ref)
    assert np.array_equal(codes.cpu().numpy(), codes_ref)
