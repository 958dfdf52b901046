"""The seeded generator: host (numpy) and torch integer evaluations agree bit for
bit, the moments are those of N(0, 1), and routed ids are distinct per token."""
import numpy as np
import pytest
import torch

import synth


def _torch_path(seed, stream, idx):
    lo = idx & synth.M32
    hi = idx >> 32
    S = torch.zeros_like(idx)
    for j in range(6):
        h = synth.lowbias32(synth.lowbias32(lo ^ synth._key(seed, stream, j)) ^ hi)
        S += (h & 0xFFFF) + (h >> 16)
    return (S - 393210).to(torch.float32) / 65536.0


def test_numpy_and_torch_integer_paths_agree():
    idx = torch.arange(1 << 16, dtype=torch.int64) * 104729 + (5 << 32)
    a = synth.normal_at(7, synth.STREAM_W, idx)
    b = _torch_path(7, synth.STREAM_W, idx)
    assert torch.equal(a, b)


def test_moments_and_support():
    z = synth.normal_at(0, synth.STREAM_X, torch.arange(1 << 20))
    assert abs(float(z.mean())) < 5e-3 and abs(float(z.std()) - 1.0) < 5e-3
    assert float(z.abs().max()) <= 6.0
    w = synth.weights(0, 64, 4096)
    assert abs(float(w.std()) - 0.02) < 2e-4 and float(w.abs().max()) <= 0.12


def test_rows_regenerate_independently():
    W = synth.weights(3, 40, 256)
    rows = [0, 7, 39]
    assert torch.equal(synth.weights_rows(3, rows, 256), W[rows])


@pytest.mark.gpu
def test_device_generator_matches_host():
    idx = torch.arange(1 << 18, dtype=torch.int64) * 7919 + (3 << 32)
    a = synth.normal_at(11, synth.STREAM_W, idx)
    b = synth.normal_at(11, synth.STREAM_W, idx.cuda()).cpu()
    assert torch.equal(a, b)
    x = synth.activations(2, 3, 512)
    xg = synth.activations(2, 3, 512, device="cuda").cpu()
    assert torch.equal(x.view(torch.int16), xg.view(torch.int16))
