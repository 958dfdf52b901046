"""GPU parity of the NVFP4 W4A4 prefill GEMM (tcgen05 block-scaled MMA).

Expected values come from the CPU oracle only: its NVFP4 activation quantizer
(the same static x_scale), its BlockToFloat of the weights, and fp64 dots of the
dequantized operands. The quantized activations are dequantized with the
oracle's own scalar decoders (E2M1 and E4M3 tables built from them).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from cases import TOL, device_matrix, host_dequant, host_matrix, host_rows_dequant, norm_err, sample_rows

pytestmark = pytest.mark.gpu

E2M1 = np.array([oracle.e2m1_to_f32(c) for c in range(16)], dtype=np.float64)
E4M3 = np.array([oracle.e4m3_to_f32(c) for c in range(256)], dtype=np.float64)


@pytest.fixture(scope="module")
def q():
    import block_quantized_weight_fly_gb300 as q
    torch.cuda.set_device(0)
    q.qmv_device_status(reset=True)
    return q


def act_dequant(x, x_scale):
    """Oracle-quantized activations, dequantized in fp64: e2m1(c) * e4m3(s_b) * x_scale."""
    xb = synth.bf16_bits(x)
    codes, scales = oracle.quant_act_nvfp4(xb, x_scale)
    M, K = xb.shape
    c = np.empty((M, K), dtype=np.int64)
    c[:, 0::2] = codes & 15
    c[:, 1::2] = codes >> 4
    s = np.repeat(scales.astype(np.int64), 16, axis=1)
    return E2M1[c] * E4M3[s] * np.float64(x_scale)


def x_scale_of(x):
    return float(np.float32(np.abs(x.float().numpy()).max()) / np.float32(2688.0))


def ref_w4a4(Wd, Xd):
    """fp64 y[m][n] = sum_k Xd[m,k] Wd[n,k] and the normalising sum of |terms|."""
    Wd = Wd.astype(np.float64)
    return Xd @ Wd.T, np.abs(Xd) @ np.abs(Wd).T


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (200, 384, 1024), (130, 640, 512), (1, 128, 256)])
def test_w4a4_small(q, M, N, K):
    W, canon = host_matrix("nvfp4", 41, N, K)
    Wd = host_dequant("nvfp4", canon, N, K)
    x = synth.activations(43 + M, M, K)
    xs = x_scale_of(x)
    ref, den = ref_w4a4(Wd, act_dequant(x, xs))
    packed = q.qmv_pack("nvfp4", torch.from_numpy(canon).cuda(), N, K)
    ws = q.workspace(q.QMV_ENTRY_W4A4, "nvfp4", M, N, K)
    y = q.qmv_gemm_nvfp4_w4a4(packed, x.cuda(), xs, N, K, ws)
    assert q.qmv_last_route() == q.FORMATS["nvfp4"] * 100 + 4
    y = y.cpu().numpy()
    assert q.qmv_device_status() == 0
    assert np.isfinite(y).all()
    assert norm_err(y, ref, den) <= TOL


@pytest.mark.parametrize("M,N,K", [(256, 512, 4096), (384, 768, 2048), (300, 1280, 3072)])
def test_w4a4_split_k_deterministic_and_clean(q, M, N, K):
    """Shapes whose output tiles are split between many CTAs: the finishing CTAs add
    the published partial sums, every publication flag is zero again after the call,
    and a second call with the same workspace gives the same bits."""
    W, canon = host_matrix("nvfp4", 47, N, K)
    Wd = host_dequant("nvfp4", canon, N, K)
    x = synth.activations(53 + M, M, K)
    xs = x_scale_of(x)
    ref, den = ref_w4a4(Wd, act_dequant(x, xs))
    packed = q.qmv_pack("nvfp4", torch.from_numpy(canon).cuda(), N, K)
    ws = q.workspace(q.QMV_ENTRY_W4A4, "nvfp4", M, N, K)
    y1 = q.qmv_gemm_nvfp4_w4a4(packed, x.cuda(), xs, N, K, ws).clone()
    # workspace: activation planes, then one 128 KB partial-sum slot and one flag per SM
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    planes = -(-((K // 256) * (-(-M // 128) * 128) * 144) // 256) * 256
    flags = ws[planes + sms * 131072:planes + sms * 131072 + 4 * sms]
    assert int(flags.count_nonzero()) == 0
    y2 = q.qmv_gemm_nvfp4_w4a4(packed, x.cuda(), xs, N, K, ws)
    assert q.qmv_device_status() == 0
    assert torch.equal(y1, y2)
    assert int(flags.count_nonzero()) == 0
    assert norm_err(y1.cpu().numpy(), ref, den) <= TOL


@pytest.mark.parametrize("N,K", [(17408, 5120), (5120, 17408)])
def test_w4a4_full_size_sampled(q, N, K):
    """The prefill configuration, M = 512: weights generated on the device, sampled
    output columns (weight rows) checked against the oracle for every token."""
    M, seed = 512, 900 + N % 7
    packed = device_matrix(q, "nvfp4", seed, N, K)
    x = synth.activations(seed + 1, M, K)
    xs = x_scale_of(x)
    ws = q.workspace(q.QMV_ENTRY_W4A4, "nvfp4", M, N, K)
    y = q.qmv_gemm_nvfp4_w4a4(packed, x.cuda(), xs, N, K, ws)
    rows = sample_rows(N, 24, seed)
    got = y[:, torch.from_numpy(rows).cuda()].cpu().numpy()
    assert q.qmv_device_status() == 0
    Wd = host_rows_dequant("nvfp4", seed, rows, N, K)
    ref, den = ref_w4a4(Wd, act_dequant(x, xs))
    assert norm_err(got, ref, den) <= TOL
    assert bool(torch.isfinite(y).all())


def test_w4a4_errors(q):
    N, K, M = 256, 512, 128
    W, canon = host_matrix("nvfp4", 47, N, K)
    packed = q.qmv_pack("nvfp4", torch.from_numpy(canon).cuda(), N, K)
    x = synth.activations(47, M, K).cuda()
    ws = q.workspace(q.QMV_ENTRY_W4A4, "nvfp4", M, N, K)
    with pytest.raises(q.QmvError) as ei:
        q.qmv_gemm_nvfp4_w4a4(packed, x, 0.01, N, K, ws[:1024])
    assert ei.value.status == 8
    assert q.qmv_workspace_size(q.QMV_ENTRY_W4A4, "nvfp4", M, N, 300) == 0
    q.qmv_device_status(reset=True)
    q.qmv_gemm_nvfp4_w4a4(packed, x, 0.01, N - 128, K, ws)   # disagrees with the header
    assert q.qmv_device_status(reset=True) == 5
