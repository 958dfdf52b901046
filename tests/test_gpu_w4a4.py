"""GPU parity of the NVFP4 W4A4 prefill GEMM (tcgen05 block-scaled MMA).

Expected values come from the CPU oracle alone (oracle.w4a4_f64): its NVFP4
activation quantizer under the same static x_scale, the dequantized activations,
its BlockToFloat of the weights and fp64 dots, with the sum of |terms| as the
error scale. The test assembles no expected value of its own.
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


def x_scale_of(x):
    return float(np.float32(np.abs(x.float().numpy()).max()) / np.float32(2688.0))


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (200, 384, 1024), (130, 640, 512), (1, 128, 256)])
def test_w4a4_small(q, M, N, K):
    W, canon = host_matrix("nvfp4", 41, N, K)
    Wd = host_dequant("nvfp4", canon, N, K)
    x = synth.activations(43 + M, M, K)
    xs = x_scale_of(x)
    ref, den = oracle.w4a4_f64(Wd, synth.bf16_bits(x), xs)
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
    ref, den = oracle.w4a4_f64(Wd, synth.bf16_bits(x), xs)
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
    ref, den = oracle.w4a4_f64(Wd, synth.bf16_bits(x), xs)
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
