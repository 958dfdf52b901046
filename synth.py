"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds none of the method's arithmetic: it draws fp32 weight values,
bf16 activations and routed expert ids. Quantization (encoding) and everything
after it live in the CUDA library and, independently, in the CPU oracle.

One counter-based generator, evaluated with exact integer and IEEE-754 fp32 ops
only, so the same element index gives the same bits on the host (numpy uint32
arithmetic) and on the GPU (torch int64 arithmetic on CUDA tensors):

  key_j      = lowbias32(seed * 0x9E3779B9 + stream * 0x85EBCA6B + j * 0xC2B2AE35)
  h_j(i)     = lowbias32(lowbias32(lo32(i) ^ key_j) ^ hi32(i))           j = 0..5
  S(i)       = sum over the twelve 16-bit halves of h_0..h_5               (integer)
  z(i)       = float32(S(i) - 393210) / 65536                              (exact)

lowbias32 is Chris Wellons' 32-bit integer hash (two xorshift-multiply rounds,
constants 0x7feb352d and 0x846ca68b). z is the Irwin-Hall sum of twelve uniforms
minus six: mean 0, variance 1 (to within 2^-32), support [-6, 6].

  weights:      w = 0.02f * z  (fp32 multiply)      -- N(0, 0.02)
  activations:  x = bf16_rne(z)                      -- N(0, 1)
  expert ids:   per token, a partial Fisher-Yates shuffle of range(E) driven by
                the same hash: top-k distinct ids, uniform without replacement.
  codebooks:    the same shuffle over -127..127: n distinct int8 values, sorted.
  grids:        per entry and position, one of a few magnitude levels (the same
                shuffle over 1..63), picked by the hash.

Element index i of a weight matrix W[N, K] of stream s is r*K + k; a stacked
tower of E experts uses r = e*N + n, so any subset of rows can be regenerated on
its own (the oracle regenerates only the rows it checks).
"""
from __future__ import annotations

import numpy as np
import torch

M32 = 0xFFFFFFFF

# stream ids, one per synthetic tensor role
STREAM_W = 1
STREAM_X = 2
STREAM_IDS = 3
STREAM_CODEBOOK = 4


def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    """(x * c) mod 2^32 for x in [0, 2^32) held in int64, without overflow."""
    lo = c & 0xFFFF
    hi = c >> 16
    return ((x * lo) + (((x * hi) & 0xFFFF) << 16)) & M32


def lowbias32(x: torch.Tensor) -> torch.Tensor:
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def _lowbias32_int(x: int) -> int:
    x &= M32
    x ^= x >> 16
    x = (x * 0x7FEB352D) & M32
    x ^= x >> 15
    x = (x * 0x846CA68B) & M32
    x ^= x >> 16
    return x


def _key(seed: int, stream: int, j: int) -> int:
    return _lowbias32_int(seed * 0x9E3779B9 + stream * 0x85EBCA6B + j * 0xC2B2AE35)


def _lowbias32_np(x: np.ndarray) -> np.ndarray:
    """lowbias32 on a uint32 numpy array (uint32 arithmetic wraps mod 2^32)."""
    x = x ^ (x >> np.uint32(16))
    x = x * np.uint32(0x7FEB352D)
    x = x ^ (x >> np.uint32(15))
    x = x * np.uint32(0x846CA68B)
    x = x ^ (x >> np.uint32(16))
    return x


def normal_at_np(seed: int, stream: int, idx: np.ndarray) -> np.ndarray:
    """z(i) on the host with numpy uint32 arithmetic (same bits as normal_at)."""
    idx = np.asarray(idx, dtype=np.int64)
    lo = (idx & M32).astype(np.uint32)
    hi = (idx >> 32).astype(np.uint32)
    S = np.zeros(idx.shape, dtype=np.int64)
    with np.errstate(over="ignore"):
        for j in range(6):
            h = _lowbias32_np(_lowbias32_np(lo ^ np.uint32(_key(seed, stream, j))) ^ hi)
            S += (h & np.uint32(0xFFFF)).astype(np.int64) + (h >> np.uint32(16)).astype(np.int64)
    return (S - 393210).astype(np.float32) / np.float32(65536.0)


def normal_at(seed: int, stream: int, idx: torch.Tensor) -> torch.Tensor:
    """z(i) for an int64 tensor of element indices (any device) -> float32."""
    if not idx.is_cuda:
        return torch.from_numpy(normal_at_np(seed, stream, idx.numpy()))
    idx = idx.to(torch.int64)
    lo = idx & M32
    hi = idx >> 32
    S = torch.zeros_like(idx)
    for j in range(6):
        h = lowbias32(lowbias32(lo ^ _key(seed, stream, j)) ^ hi)
        S += (h & 0xFFFF) + (h >> 16)
    return (S - 393210).to(torch.float32) / 65536.0


def weights_rows(seed: int, rows, K: int, device="cpu", stream: int = STREAM_W) -> torch.Tensor:
    """fp32 W[len(rows), K] ~ N(0, 0.02) for the given global row indices."""
    rows = torch.as_tensor(rows, dtype=torch.int64, device=device).reshape(-1, 1)
    k = torch.arange(K, dtype=torch.int64, device=device).reshape(1, -1)
    z = normal_at(seed, stream, rows * K + k)
    return z * torch.tensor(0.02, dtype=torch.float32, device=z.device)


def weights(seed: int, N: int, K: int, device="cpu", row0: int = 0,
            chunk_rows: int | None = None, stream: int = STREAM_W) -> torch.Tensor:
    """fp32 W[N, K] (global rows row0 .. row0+N-1), generated in row chunks."""
    out = torch.empty((N, K), dtype=torch.float32, device=device)
    if chunk_rows is None:
        chunk_rows = max(1, (1 << 24) // max(K, 1))
    for r in range(0, N, chunk_rows):
        n = min(chunk_rows, N - r)
        out[r:r + n] = weights_rows(seed, torch.arange(row0 + r, row0 + r + n), K, device, stream)
    return out


def activations(seed: int, M: int, K: int, device="cpu", stream: int = STREAM_X) -> torch.Tensor:
    """bf16 x[M, K] ~ N(0, 1)."""
    idx = torch.arange(M * K, dtype=torch.int64, device=device).reshape(M, K)
    return normal_at(seed, stream, idx).to(torch.bfloat16)


def expert_ids(seed: int, M: int, topk: int, E: int, stream: int = STREAM_IDS) -> np.ndarray:
    """int32 ids[M, topk]: per token, topk distinct experts uniform over range(E)."""
    out = np.empty((M, topk), dtype=np.int32)
    key = _key(seed, stream, 0)
    for t in range(M):
        perm = list(range(E))
        for j in range(topk):
            h = _lowbias32_int(_lowbias32_int((t * 64 + j) ^ key) ^ 0x68E31DA4)
            r = j + h % (E - j)
            perm[j], perm[r] = perm[r], perm[j]
            out[t, j] = perm[j]
    return out


def codebook(seed: int, n: int = 16, stream: int = STREAM_CODEBOOK) -> np.ndarray:
    """int8 codebook[n]: n distinct values drawn uniformly from -127..127 (a partial
    Fisher-Yates shuffle driven by the hash), ascending."""
    key = _key(seed, stream, 0)
    perm = list(range(-127, 128))
    for j in range(n):
        h = _lowbias32_int(_lowbias32_int(j ^ key) ^ 0x3C6EF372)
        r = j + h % (len(perm) - j)
        perm[j], perm[r] = perm[r], perm[j]
    return np.array(sorted(perm[:n]), dtype=np.int8)


def grid(seed: int, entries: int, width: int, levels: int, stream: int = STREAM_CODEBOOK) -> np.ndarray:
    """uint8 grid[entries, width] of magnitudes: `levels` distinct values drawn from
    1..63 (the same shuffle), each entry value one of them picked by the hash."""
    key = _key(seed, stream, 1)
    perm = list(range(1, 64))
    for j in range(levels):
        h = _lowbias32_int(_lowbias32_int(j ^ key) ^ 0x3C6EF372)
        r = j + h % (len(perm) - j)
        perm[j], perm[r] = perm[r], perm[j]
    lv = np.array(sorted(perm[:levels]), dtype=np.uint8)
    idx = np.arange(entries * width, dtype=np.uint32)
    with np.errstate(over="ignore"):
        h = _lowbias32_np(_lowbias32_np(idx ^ np.uint32(key)) ^ np.uint32(0x5BD1E995))
    return lv[(h % np.uint32(levels)).astype(np.int64)].reshape(entries, width)


def bf16_bits(x: torch.Tensor) -> np.ndarray:
    """The raw uint16 bit patterns of a bf16 tensor, as numpy (host copy)."""
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
