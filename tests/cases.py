"""Shared helpers for the GPU parity tests: building inputs on the oracle side
(host, oracle encoders) and on the device side (seeded generator + the library's
quantizer), and the normalised error of BASELINE's tolerance.

The error of one output element is |y - y_ref| / sum_k |w_k x_k| (fp64), the bound
is 1e-5; an element whose denominator is zero must be exactly zero.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

TOL = 1e-5

# NVFP4 tensor scale of synthetic N(0, 0.02) weights: the generator's support is
# |z| <= 6, so |w| <= 0.12 and s_T = 0.12 / (448 * 6) is a static per-tensor constant
NVFP4_WEIGHT_AMAX = np.float32(0.12)
NVFP4_TS = float(NVFP4_WEIGHT_AMAX / np.float32(2688.0))


def tensor_scale(fmt) -> float:
    return NVFP4_TS if fmt == "nvfp4" else 0.0


# formats whose canonical stream is per matrix (a tower is E streams back to back)
PER_MATRIX = ("nvfp4", "fp8_row", "iq4_xs")


def codebook(fmt, seed, e):
    """The IQ4_XS codebook of expert e of a seeded tower (each expert its own); None
    for the other formats."""
    return synth.codebook(seed + 7919 * e) if fmt == "iq4_xs" else None


GRID_FORMATS = {"iq3_s": (512, 4, 8), "iq2_s": (1024, 8, 4)}     # entries, width, levels


def grid(fmt, seed):
    """The grid of a seeded IQ3_S / IQ2_S tower (one table for all its experts)."""
    ne, gw, lv = GRID_FORMATS[fmt]
    return synth.grid(seed, ne, gw, lv)


def _encode(fmt, W, seed, e):
    return oracle.encode(fmt, W, tensor_scale(fmt), codebook=codebook(fmt, seed, e))


def _encode_tower_rows(fmt, W, seed):
    """K-quants: rows in any grouping; grid formats: the tower's grid, then the rows."""
    if fmt in GRID_FORMATS:
        return oracle.encode(fmt, W, codebook=grid(fmt, seed))
    return oracle.encode(fmt, W, tensor_scale(fmt))


def norm_err(y, ref, den) -> float:
    y = np.asarray(y, dtype=np.float64)
    zero = den == 0
    if np.any(zero):
        assert np.all(y[zero] == 0.0)
    d = np.where(zero, 1.0, den)
    e = np.abs(y - ref) / d
    e[zero] = 0.0
    return float(e.max()) if e.size else 0.0


def host_matrix(fmt, seed, N, K, E=1):
    """fp32 W[E*N, K] (host, synth) and its canonical bytes (oracle encoder).

    Formats whose canonical stream is per matrix (NVFP4, FP8_ROW) are encoded one
    expert at a time and concatenated."""
    W = synth.weights(seed, E * N, K).numpy()
    if fmt in PER_MATRIX:
        canon = np.concatenate([_encode(fmt, W[e * N:(e + 1) * N], seed, e) for e in range(E)])
    else:
        canon = _encode_tower_rows(fmt, W, seed)
    return W, canon


def host_dequant(fmt, canon, N, K, E=1):
    if fmt in PER_MATRIX:
        per = oracle.canon_bytes(fmt, N, K)
        return np.concatenate([oracle.block_to_float(fmt, canon[e * per:(e + 1) * per], N, K)
                               for e in range(E)])
    return oracle.block_to_float(fmt, canon, E * N, K)


def host_rows_dequant(fmt, seed, rows, N, K):
    """Oracle-side BlockToFloat of selected tower rows, regenerated from the seed
    (row = e*N + n). NVFP4 uses the static tensor scale; FP8 row scales are per row,
    so each row is a one-row matrix."""
    W = synth.weights_rows(seed, rows, K).numpy()
    if fmt == "iq4_xs":
        # blocks are per row: each row encodes alone with its expert's codebook
        out = np.empty_like(W)
        for i, r in enumerate(np.asarray(rows).reshape(-1)):
            c = _encode(fmt, W[i:i + 1], seed, int(r) // N)
            out[i] = oracle.block_to_float(fmt, c, 1, K)[0]
        return out
    if fmt in ("nvfp4", "fp8_row"):
        out = np.empty_like(W)
        for i in range(W.shape[0]):
            c = oracle.encode(fmt, W[i:i + 1], tensor_scale(fmt))
            out[i] = oracle.block_to_float(fmt, c, 1, K)[0]
        return out
    c = _encode_tower_rows(fmt, W, seed)
    return oracle.block_to_float(fmt, c, W.shape[0], K)


def device_matrix(q, fmt, seed, N, K, E=1, dev="cuda"):
    """Packed device tower generated on the device: synth (torch CUDA) -> the library
    quantizer -> qmv_pack. Returns the packed buffer."""
    chunk_rows = max(1, (1 << 26) // K)
    canon_parts = []
    for e in range(E):
        parts = []
        for r0 in range(0, N, chunk_rows):
            n = min(chunk_rows, N - r0)
            W = synth.weights(seed, n, K, device=dev, row0=e * N + r0)
            if fmt in ("nvfp4", "fp8_row"):
                parts.append(W)
            elif fmt == "iq4_xs":
                # the blocks of this chunk, without the codebook the encoder appends
                parts.append(q.qmv_quantize_codebook(fmt, W, codebook(fmt, seed, e))[:n * (K // 256) * 136])
            elif fmt in GRID_FORMATS:
                # the blocks of this chunk, without the grid the encoder puts first
                parts.append(q.qmv_quantize_codebook(fmt, W, grid(fmt, seed))[oracle.grid_bytes(fmt):])
            else:
                parts.append(q.qmv_quantize(fmt, W))
        if fmt == "iq4_xs":
            cb = torch.from_numpy(codebook(fmt, seed, e).view(np.uint8).copy()).to(dev)
            canon_parts.append(torch.cat(parts + [cb]))
        elif fmt in ("nvfp4", "fp8_row"):
            # per-matrix stream: quantize the whole expert matrix at once
            Wm = torch.cat(parts)
            canon_parts.append(q.qmv_quantize(fmt, Wm, tensor_scale(fmt)))
            del Wm
        else:
            canon_parts.append(torch.cat(parts))
        del parts
    if fmt in GRID_FORMATS:
        canon_parts.insert(0, torch.from_numpy(grid(fmt, seed).reshape(-1).copy()).to(dev))
    canon = torch.cat(canon_parts)
    del canon_parts
    packed = q.qmv_pack(fmt, canon, N, K, E)
    del canon
    return packed


def sample_rows(N, count, seed=0):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 127, 128, 129, N // 2, N - 129, N - 128, N - 2, N - 1]
    extra = rng.choice(N, size=min(count, N), replace=False).tolist()
    rows = sorted(set([r for r in fixed + extra if 0 <= r < N]))
    return np.array(rows, dtype=np.int64)
