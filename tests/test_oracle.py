"""Pins for the CPU oracle: checks against things other than the oracle itself.

- page-printed byte counts (tests/golden/page_sizes.txt);
- library conversions (numpy float16, torch float8_e4m3fn) and exhaustive code tables
  against the closed-form format definitions;
- hand-built blocks whose decoded values are worked out by hand and written literally;
- encode -> decode round-trip error bounds derived from each quantizer;
- exact rational arithmetic (fractions.Fraction) and numpy fp64 matmul for the dot products;
- the closed-form expected number of distinct routed experts.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_sizes.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, value, _unit, _where = [p.strip() for p in line.split("|")]
        vals[name] = float(value)
    return vals


# ---------------------------------------------------------------------------
# byte sizes printed on the pages
# ---------------------------------------------------------------------------
def test_block_sizes_match_pages():
    g = _golden()
    assert oracle.canon_bytes("q6_k", 1, 256) == g["q6_k_block_bytes"] == 210
    assert oracle.canon_bytes("q8_0", 1, 32) == g["q8_0_block_bytes"] == 34
    assert math.ceil(oracle.canon_bytes("q6_k", 1, 256) / 4) == g["q6_k_block_words"]
    assert math.ceil(oracle.canon_bytes("q8_0", 1, 32) / 4) == g["q8_0_block_words"]
    # fixtures: 32 Q6_K blocks and 512 Q8_0 blocks
    assert oracle.canon_bytes("q6_k", 1, 32 * 256) == g["fixture_q6_k_bytes"]
    assert oracle.canon_bytes("q8_0", 1, 512 * 32) == g["fixture_q8_0_bytes"]
    # the untied head [248320 rows, 5120] at Q6_K, and its bf16 twin, in GiB
    head = oracle.canon_bytes("q6_k", 248320, 5120)
    assert head == 1_042_944_000
    assert round(head / 2**30, 2) == g["output_head_q6_k_5120x248320_packed"]
    assert round(248320 * 5120 * 2 / 2**30, 2) == g["output_head_bf16_twin"]
    # token_embd at 144 B / 256 is the K-quant size closest to the printed 0.68
    emb = oracle.canon_bytes("q4_k", 5120, 248320) / 2**30
    candidates = {110: "q3_k", 144: "q4_k", 176: "q5_k", 210: "q6_k"}
    best = min(candidates, key=lambda b: abs(5120 * 248320 / 256 * b / 2**30 - g["token_embd_q4_k_5120x248320_packed"]))
    assert candidates[best] == "q4_k" and abs(emb - 0.68) < 0.02


def test_nvfp4_fp8_sizes():
    # NVFP4: 4-bit codes + one E4M3 byte per 16 values + one fp32 tensor scale
    assert oracle.canon_bytes("nvfp4", 17408, 5120) == 44_564_480 + 5_570_560 + 4
    # FP8 row: one byte per value + one fp32 per row
    assert oracle.canon_bytes("fp8_row", 6144, 5120) == 31_457_280 + 24_576
    assert oracle.canon_bytes("q4_k", 2048, 4096) == 4_718_592


# ---------------------------------------------------------------------------
# scalar formats
# ---------------------------------------------------------------------------
def test_fp16_decode_exhaustive_vs_numpy():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = codes.view(np.float16).astype(np.float32)
    got = np.array([oracle.fp16_to_f32(int(c)) for c in codes], dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_bf16_decode_exhaustive():
    # bf16 is the upper half of an IEEE binary32: decode = the code shifted into the top bits
    codes = np.arange(65536, dtype=np.uint32)
    ref = (codes << 16).view(np.float32)
    got = np.array([oracle.bf16_to_f32(int(c)) for c in codes], dtype=np.float32)
    nan = np.isnan(ref)          # a signalling NaN comes back quieted through a Python float
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2 * 127
    assert np.array_equal(got.view(np.uint32)[~nan], ref.view(np.uint32)[~nan])


def test_block_lengths():
    # values per quantization block: Q8_0 32, K-quant superblocks 256, NVFP4 16
    assert [oracle.block_values(f) for f in ("q8_0", "q4_k", "q5_k", "q6_k", "nvfp4")] == [32, 256, 256, 256, 16]


def test_bf16_rounding_of_doubles():
    """or_f64_to_bf16: every bf16 value maps to itself; fp32 inputs round as torch's
    fp32 -> bf16 conversion (round to nearest even); midpoints between neighbours go to
    the even one; overflow gives infinity."""
    pats = np.arange(0, 1 << 16, dtype=np.uint32)
    vals = (pats << 16).view(np.float32)
    finite = np.isfinite(vals)
    got = oracle.f64_to_bf16_array(vals[finite].astype(np.float64))
    assert np.array_equal(got[vals[finite] != 0], pats[finite][vals[finite] != 0].astype(np.uint16))
    rng = np.random.default_rng(3)
    v = np.concatenate([rng.standard_normal(20000), rng.standard_normal(2000) * 1e-39,
                        rng.standard_normal(2000) * 1e37]).astype(np.float32)
    want = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.f64_to_bf16_array(v.astype(np.float64)), want)
    # 1 + 2^-8 is the midpoint of 1 and 1 + 2^-7: to 1 (even); 1 + 3 * 2^-8 to 1 + 2^-6
    assert oracle.f64_to_bf16(1 + 2.0**-8) == 0x3F80 and oracle.f64_to_bf16(1 + 3 * 2.0**-8) == 0x3F82
    assert oracle.f64_to_bf16(-(1 + 2.0**-8)) == 0xBF80
    assert oracle.f64_to_bf16(1e39) == 0x7F80 and oracle.f64_to_bf16(-1e39) == 0xFF80


def test_fp16_encode_vs_numpy_rne():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * np.float32(0.02),
        (rng.standard_normal(2000) * 1e-5).astype(np.float32),       # subnormal range
        (rng.standard_normal(1000) * 2e4).astype(np.float32),        # near overflow
        np.array([0.0, -0.0, 65504.0, 65519.0, 65520.0, 1e9, 2.0**-25, 2.0**-24 * 1.5,
                  1.0 + 2.0**-11, 1.0 + 3 * 2.0**-11], dtype=np.float32),   # ties
    ])
    with np.errstate(over="ignore"):                    # 65520 and above round to inf on purpose
        ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f32_to_fp16(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


def _e4m3_closed_form(c):
    s, e, m = c >> 7, (c >> 3) & 15, c & 7
    if e == 15 and m == 7:
        return float("nan")
    v = 2.0**-6 * m / 8 if e == 0 else 2.0 ** (e - 7) * (1 + m / 8)
    return -v if s else v


def test_e4m3_table_exhaustive():
    lib = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    for c in range(256):
        got = oracle.e4m3_to_f32(c)
        want = _e4m3_closed_form(c)
        if math.isnan(want):
            assert math.isnan(got) and math.isnan(lib[c])
        else:
            assert got == want == lib[c], c
    assert oracle.e4m3_to_f32(0x38) == 1.0 and oracle.e4m3_to_f32(0x7E) == 448.0
    assert oracle.e4m3_to_f32(0x01) == 2.0**-9 and oracle.e4m3_to_f32(0x08) == 2.0**-6


def test_e4m3_encode_rne_sat():
    # every finite code round-trips
    for c in range(256):
        v = _e4m3_closed_form(c)
        if not math.isnan(v) and c != 0x80:
            assert oracle.f32_to_e4m3(v) == c
    # against torch's RNE cast where it does not overflow, incl. midpoints
    finite = sorted({abs(_e4m3_closed_form(c)) for c in range(128) if c != 0x7F})
    mids = [(a + b) / 2 for a, b in zip(finite, finite[1:])]
    rng = np.random.default_rng(2)
    vals = np.concatenate([np.array(mids + finite, dtype=np.float32),
                           (rng.standard_normal(3000) * 50).astype(np.float32)])
    vals = np.concatenate([vals, -vals])
    vals = vals[np.abs(vals) < 464]
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.f32_to_e4m3(float(v)) for v in vals], dtype=np.uint8)
    assert np.array_equal(got, ref)
    # saturation beyond the largest finite value (448 = 0x7E)
    for v in (464.0, 470.0, 1e6, float("inf")):
        assert oracle.f32_to_e4m3(v) == 0x7E and oracle.f32_to_e4m3(-v) == 0xFE


def test_e2m1_table_and_ties():
    table = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    for c in range(16):
        want = table[c & 7] * (-1 if c & 8 else 1)
        assert oracle.e2m1_to_f32(c) == want
        if c != 8:
            assert oracle.f32_to_e2m1(want) == c
    ties = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0,
            6.5: 6.0, 7.0: 6.0, 100.0: 6.0, 0.3: 0.5, 0.2: 0.0}
    for v, want in ties.items():
        assert oracle.e2m1_to_f32(oracle.f32_to_e2m1(v)) == want, v
        assert oracle.e2m1_to_f32(oracle.f32_to_e2m1(-v)) == -want, v
    # brute force nearest, ties to the even code
    rng = np.random.default_rng(3)
    for v in rng.uniform(-8, 8, 2000).astype(np.float32):
        mags = np.array(table)
        d = np.abs(np.abs(float(v)) - mags)
        best = np.flatnonzero(d == d.min())
        code = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        if abs(float(v)) > 6:
            code = 7
        got = oracle.f32_to_e2m1(float(v))
        assert got & 7 == code and (got >> 3) == (1 if np.signbit(v) else 0), v


# ---------------------------------------------------------------------------
# hand-built blocks (layouts as read: see oracle.h); values worked out by hand
# ---------------------------------------------------------------------------
def test_q8_0_handbuilt():
    blk = bytearray(34)
    blk[0:2] = (0x3C00).to_bytes(2, "little")          # d = 1.0
    for i in range(32):
        blk[2 + i] = (i - 16) & 0xFF
    w = oracle.block_to_float("q8_0", np.frombuffer(bytes(blk), np.uint8), 1, 32)[0]
    assert list(w) == [float(i - 16) for i in range(32)]
    blk[0:2] = (0x3800).to_bytes(2, "little")          # d = 0.5
    blk[2] = 0x81                                        # -127
    w = oracle.block_to_float("q8_0", np.frombuffer(bytes(blk), np.uint8), 1, 32)[0]
    assert w[0] == -63.5 and w[1] == -7.5 and w[31] == 7.5


def _q4k_block(d16, dmin16, sc, mn, q):
    bits = 0
    for f in range(8):
        bits |= sc[f] << (6 * f)
        bits |= mn[f] << (6 * (8 + f))
    blk = bytearray(144)
    blk[0:2] = d16.to_bytes(2, "little")
    blk[2:4] = dmin16.to_bytes(2, "little")
    blk[4:16] = bits.to_bytes(12, "little")
    for b in range(128):
        blk[16 + b] = q[2 * b] | (q[2 * b + 1] << 4)
    return bytes(blk)


def test_q4_k_handbuilt_values():
    blk = _q4k_block(0x3C00, 0x3C00, [j + 1 for j in range(8)], list(range(8)),
                     [e % 16 for e in range(256)])
    w = oracle.block_to_float("q4_k", np.frombuffer(blk, np.uint8), 1, 256)[0]
    # e=0: j=0, q=0 -> 0      e=15: j=0 (sc 1, m 0), q=15 -> 15     e=33: j=1 (sc 2, m 1), q=1 -> 1
    # e=100: j=3 (sc 4, m 3), q=4 -> 13     e=160: j=5 (sc 6, m 5), q=0 -> -5
    # e=255: j=7 (sc 8, m 7), q=15 -> 113
    hand = {0: 0.0, 15: 15.0, 33: 1.0, 100: 13.0, 160: -5.0, 255: 113.0}
    for e, v in hand.items():
        assert w[e] == v, (e, w[e], v)
    # d = 0.5, dmin = 0.25 (0x3400), sc_j = 63, m_j = 63, q = 15 everywhere:
    # w = 0.5*63*15 - 0.25*63 = 472.5 - 15.75 = 456.75
    blk = _q4k_block(0x3800, 0x3400, [63] * 8, [63] * 8, [15] * 256)
    w = oracle.block_to_float("q4_k", np.frombuffer(blk, np.uint8), 1, 256)[0]
    assert np.all(w == 456.75)


def _q5k_block(d16, dmin16, sc, mn, q):
    """Q5_K as read: Q4_K's header, a 32-byte plane of fifth bits, then the nibbles."""
    q4 = _q4k_block(d16, dmin16, sc, mn, [v & 15 for v in q])
    qh = 0
    for e in range(256):
        qh |= ((q[e] >> 4) & 1) << e
    return q4[:16] + qh.to_bytes(32, "little") + q4[16:]


def test_q5_k_handbuilt_values():
    blk = _q5k_block(0x3C00, 0x3C00, [j + 1 for j in range(8)], list(range(8)),
                     [e % 32 for e in range(256)])
    assert len(blk) == 176
    w = oracle.block_to_float("q5_k", np.frombuffer(blk, np.uint8), 1, 256)[0]
    # w = sc_j * q - m_j with d = dmin = 1, q = e mod 32, sc_j = j + 1, m_j = j
    # e=0: 0      e=16: j=0, q=16 -> 16      e=31: q=31 -> 31      e=33: j=1, q=1 -> 2-1 = 1
    # e=50: j=1, q=18 -> 36-1 = 35     e=100: j=3, q=4 -> 16-3 = 13     e=255: j=7, q=31 -> 248-7 = 241
    hand = {0: 0.0, 16: 16.0, 31: 31.0, 33: 1.0, 50: 35.0, 100: 13.0, 255: 241.0}
    for e, v in hand.items():
        assert w[e] == v, (e, w[e], v)
    # d = 0.5, dmin = 0.25, sc = m = 63:  q = 16 -> 504 - 15.75;  q = 31 -> 976.5 - 15.75
    blk = _q5k_block(0x3800, 0x3400, [63] * 8, [63] * 8, [16] * 128 + [31] * 128)
    w = oracle.block_to_float("q5_k", np.frombuffer(blk, np.uint8), 1, 256)[0]
    assert np.all(w[:128] == 488.25) and np.all(w[128:] == 960.75)


@pytest.mark.parametrize("e_hot", [0, 7, 8, 77, 200, 255])
def test_q5_k_fifth_bit_position(e_hot):
    """One set bit in the qh plane at byte e/8, bit e%8 moves exactly element e by 16."""
    blk = bytearray(176)
    blk[0:2] = (0x3C00).to_bytes(2, "little")
    bits = sum(1 << (6 * f) for f in range(8))          # sc_j = 1, m_j = 0
    blk[4:16] = bits.to_bytes(12, "little")
    blk[16 + e_hot // 8] = 1 << (e_hot % 8)
    w = oracle.block_to_float("q5_k", np.frombuffer(bytes(blk), np.uint8), 1, 256)[0]
    expect = np.zeros(256, np.float32)
    expect[e_hot] = 16.0
    assert np.array_equal(w, expect)


def test_q5_k_without_fifth_bits_is_q4_k():
    """A Q5_K block whose qh plane is zero decodes exactly like the Q4_K block with
    the same header and nibbles (the 5-bit format extends the 4-bit one)."""
    W = synth.weights(21, 2, 512).numpy()
    c4 = oracle.encode("q4_k", W).reshape(2, 2, 144)
    c5 = np.concatenate([c4[..., :16], np.zeros((2, 2, 32), np.uint8), c4[..., 16:]], -1)
    D4 = oracle.block_to_float("q4_k", c4.reshape(-1), 2, 512)
    D5 = oracle.block_to_float("q5_k", c5.reshape(-1), 2, 512)
    assert np.array_equal(D4, D5)


def test_q6_k_handbuilt():
    # d = 0.5, sc_j = +1 (even j) / -1 (odd j), q_e = e mod 64  ->  w = 0.5 (q-32) sc_j
    blk = bytearray(210)
    for e in range(256):
        q = e % 64
        blk[e // 2] |= (q & 15) << (4 * (e & 1))
        blk[128 + e // 4] |= ((q >> 4) & 3) << (2 * (e & 3))
    for j in range(16):
        blk[192 + j] = 1 if j % 2 == 0 else 0xFF
    blk[208:210] = (0x3800).to_bytes(2, "little")
    w = oracle.block_to_float("q6_k", np.frombuffer(bytes(blk), np.uint8), 1, 256)[0]
    # e=0: q=0, j=0 (sc +1): 0.5*(-32) = -16      e=16: q=16, j=1 (sc -1): 0.5*(-16)*(-1) = 8
    # e=31: q=31, j=1 (sc -1): 0.5*(-1)*(-1) = 0.5  e=63: q=63, j=3 (sc -1): 0.5*31*(-1) = -15.5
    # e=64: q=0, j=4 (sc +1): -16                    e=255: q=63, j=15 (sc -1): -15.5
    hand = {0: -16.0, 16: 8.0, 31: 0.5, 63: -15.5, 64: -16.0, 255: -15.5}
    for e, v in hand.items():
        assert w[e] == v, (e, w[e], v)


def test_nvfp4_handbuilt():
    K = 32
    codes = bytearray(K // 2)
    for e in range(K):
        codes[e // 2] |= (e % 16) << (4 * (e & 1))
    scales = bytes([0x38, 0x40])                       # 1.0, 2.0
    canon = bytes(codes) + scales + np.float32(0.5).tobytes()
    w = oracle.block_to_float("nvfp4", np.frombuffer(canon, np.uint8), 1, K)[0]
    table = [0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.0, -0.5, -1, -1.5, -2, -3, -4, -6]
    assert list(w[:16]) == [v * 0.5 for v in table]   # s_b = 1, s_T = 0.5
    assert list(w[16:]) == table                        # s_b = 2, s_T = 0.5


def test_fp8_row_handbuilt():
    K = 256
    codes = bytes(range(256))
    canon = codes + np.float32(2.0).tobytes()
    w = oracle.block_to_float("fp8_row", np.frombuffer(canon, np.uint8), 1, K)[0]
    for c in range(256):
        v = _e4m3_closed_form(c)
        if math.isnan(v):
            assert math.isnan(w[c])
        else:
            assert w[c] == 2.0 * v


# ---------------------------------------------------------------------------
# IQ4_XS: 136-byte blocks, a weight is a codebook entry times its sub-block scale
# ---------------------------------------------------------------------------
CB_HAND = [-127, -100, -60, -33, -20, -9, -2, 0, 1, 5, 11, 25, 40, 66, 90, 127]


def _iq4xs_block(d16, ls, q):
    """IQ4_XS as read: fp16 d, u16 of scale high bits, 4 bytes of scale low nibbles,
    128 bytes of index nibbles (element 2b low, 2b+1 high)."""
    blk = bytearray(136)
    blk[0:2] = d16.to_bytes(2, "little")
    sh = 0
    for j in range(8):
        sh |= ((ls[j] >> 4) & 3) << (2 * j)
        blk[4 + j // 2] |= (ls[j] & 15) << (4 * (j & 1))
    blk[2:4] = sh.to_bytes(2, "little")
    for b in range(128):
        blk[8 + b] = q[2 * b] | (q[2 * b + 1] << 4)
    return bytes(blk)


def _iq4xs_decode(blocks, cb, rows, K):
    canon = b"".join(blocks) + bytes(np.array(cb, dtype=np.int8).view(np.uint8))
    return oracle.block_to_float("iq4_xs", np.frombuffer(canon, np.uint8), rows, K)


def test_iq4_xs_sizes_match_pages():
    g = _golden()
    assert oracle.canon_bytes("iq4_xs", 1, 256) - 16 == g["iq4_xs_block_bytes"] == 136
    assert (oracle.canon_bytes("iq4_xs", 1, 256) - 16) * 8 / 256 == g["iq4_xs_bits_per_weight"]
    assert oracle.canon_bytes("iq4_xs", 1, 32 * 256) - 16 == g["fixture_iq4_xs_bytes"]   # 32 blocks


def test_iq4_xs_handbuilt_values():
    # d = 0.5; ls = 33, 31, 0, 63, then 32 (scale 0); q = e % 16
    blk = _iq4xs_block(0x3800, [33, 31, 0, 63, 32, 32, 32, 32], [e % 16 for e in range(256)])
    w = _iq4xs_decode([blk], CB_HAND, 1, 256)[0]
    # e=0: a = 0.5 * 1, C[0] = -127 -> -63.5        e=1: 0.5 * -100 -> -50
    # e=33: a = 0.5 * -1, C[1] = -100 -> 50         e=47: a = -0.5, C[15] = 127 -> -63.5
    # e=64: a = 0.5 * -32 = -16, C[0] -> 2032       e=79: -16 * 127 -> -2032
    # e=111: a = 0.5 * 31 = 15.5, C[15] -> 1968.5    e=103: 15.5 * C[7] = 0 -> 0
    # e=200: a = 0 -> 0
    hand = {0: -63.5, 1: -50.0, 33: 50.0, 47: -63.5, 64: 2032.0, 79: -2032.0, 111: 1968.5, 103: 0.0,
            200: 0.0}
    for e, v in hand.items():
        assert w[e] == v, (e, w[e], v)


def test_iq4_xs_every_index_reads_its_entry():
    """d = 1, ls = 33 (scale 1): the decoded values are the codebook itself, in index order."""
    blk = _iq4xs_block(0x3C00, [33] * 8, [e % 16 for e in range(256)])
    cb = synth.codebook(5)
    w = _iq4xs_decode([blk], cb, 1, 256)[0]
    assert np.array_equal(w, np.tile(cb.astype(np.float32), 16))


@pytest.mark.parametrize("j", range(8))
def test_iq4_xs_scale_bit_positions(j):
    """Only sub-block j gets ls = 48 (low nibble 0, high bits 3 -> scale 16); the low
    nibble alone (ls = 15 -> -17) is checked the same way."""
    for ls_hot, a in ((48, 16.0), (15, -17.0)):
        ls = [32] * 8
        ls[j] = ls_hot
        w = _iq4xs_decode([_iq4xs_block(0x3C00, ls, [15] * 256)], CB_HAND, 1, 256)[0]
        want = np.zeros(256, np.float32)
        want[32 * j:32 * j + 32] = a * 127
        assert np.array_equal(w, want), (j, ls_hot)


def test_iq4_xs_codebook_per_matrix_in_a_tower():
    """Two experts back to back, each with its own codebook after its blocks."""
    blk = _iq4xs_block(0x3C00, [33] * 8, [3] * 256)
    cb0, cb1 = synth.codebook(1), synth.codebook(2)
    canon = (blk + bytes(cb0.view(np.uint8))) + (blk + bytes(cb1.view(np.uint8)))
    per = oracle.canon_bytes("iq4_xs", 1, 256)
    w0 = oracle.block_to_float("iq4_xs", np.frombuffer(canon[:per], np.uint8), 1, 256)[0]
    w1 = oracle.block_to_float("iq4_xs", np.frombuffer(canon[per:], np.uint8), 1, 256)[0]
    assert np.all(w0 == float(cb0[3])) and np.all(w1 == float(cb1[3]))


# ---------------------------------------------------------------------------
# IQ3_S, IQ2_S: a group of weights is one grid entry with per-weight sign bits
# ---------------------------------------------------------------------------
def test_grid_formats_sizes_match_pages():
    g = _golden()
    for fmt, gw, ne in (("iq3_s", 4, 512), ("iq2_s", 8, 1024)):
        gb = oracle.grid_bytes(fmt)
        assert gb == ne * gw
        blk = oracle.canon_bytes(fmt, 1, 256) - gb
        assert blk == g[f"{fmt}_block_bytes"]
        assert blk * 8 / 256 == g[f"{fmt}_bits_per_weight"]
        assert oracle.canon_bytes(fmt, 1, 32 * 256) - gb == g[f"fixture_{fmt}_bytes"]   # 32 blocks
    assert oracle.grid_bytes("iq2_s") == g["iq2_s_grid_entries"] * g["iq2_s_grid_width"]
    assert oracle.grid_bytes("iq3_s") // 512 == g["iq3_s_group_width"]


def _iq3s_block(d16, sc, idx, neg):
    """IQ3_S as read: fp16 d | idx low bytes of 64 groups | idx bit 8 of group i at bit
    i | sign of element e at bit e | 4-bit scales of the 8 sub-blocks."""
    blk = bytearray(110)
    blk[0:2] = d16.to_bytes(2, "little")
    qh, sg = 0, 0
    for g in range(64):
        blk[2 + g] = idx[g] & 255
        qh |= ((idx[g] >> 8) & 1) << g
    for e in range(256):
        sg |= (1 if e in neg else 0) << e
    blk[66:74] = qh.to_bytes(8, "little")
    blk[74:106] = sg.to_bytes(32, "little")
    for j in range(8):
        blk[106 + j // 2] |= sc[j] << (4 * (j & 1))
    return bytes(blk)


def _iq2s_block(d16, sc, idx, neg):
    """IQ2_S as read: fp16 d | idx low bytes of 32 groups | sign byte of each group |
    idx bits 8..9 of group i at bits 2i, 2i+1 | 4-bit scales of the 16 sub-blocks."""
    blk = bytearray(82)
    blk[0:2] = d16.to_bytes(2, "little")
    qh = 0
    for g in range(32):
        blk[2 + g] = idx[g] & 255
        qh |= ((idx[g] >> 8) & 3) << (2 * g)
        for i in range(8):
            if 8 * g + i in neg:
                blk[34 + g] |= 1 << i
    blk[66:74] = qh.to_bytes(8, "little")
    for k in range(16):
        blk[74 + k // 2] |= sc[k] << (4 * (k & 1))
    return bytes(blk)


def _grid_decode(fmt, G, blocks, rows=1):
    canon = bytes(np.ascontiguousarray(G, dtype=np.uint8).reshape(-1)) + b"".join(blocks)
    return oracle.block_to_float(fmt, np.frombuffer(canon, np.uint8), rows, 256 * len(blocks) // rows)


def test_iq3_s_handbuilt_values():
    G = np.zeros((512, 4), np.uint8)
    G[0] = [1, 2, 3, 4]
    G[300] = [10, 20, 30, 40]
    G[511] = [255, 0, 7, 128]
    idx = [0] * 64
    idx[0], idx[8], idx[63] = 300, 0, 511
    sc = [1, 15, 0, 0, 0, 0, 0, 7]
    w = _grid_decode("iq3_s", G, [_iq3s_block(0x3800, sc, idx, {1, 253})])[0]
    # d = 0.5. Group 0 (sub-block 0, a = 0.5 * 3 = 1.5), entry 300, element 1 negative:
    # 15, -30, 45, 60. Group 8 = elements 32..35 (sub-block 1, a = 0.5 * 31 = 15.5), entry 0:
    # 15.5, 31, 46.5, 62. Group 1 (elements 4..7), entry 0: 1.5, 3, 4.5, 6.
    # Group 63 = elements 252..255 (sub-block 7, a = 0.5 * 15 = 7.5), entry 511, element 253
    # negative: 1912.5, -0, 52.5, 960. Group 40 (elements 160..163, sub-block 5, a = 0.5): 0.5, 1, 1.5, 2.
    hand = {0: 15.0, 1: -30.0, 2: 45.0, 3: 60.0, 32: 15.5, 33: 31.0, 34: 46.5, 35: 62.0, 4: 1.5, 7: 6.0,
            252: 1912.5, 253: -0.0, 254: 52.5, 255: 960.0, 160: 0.5, 163: 2.0}
    for e, v in hand.items():
        assert w[e] == v, (e, w[e], v)
    assert np.signbit(w[253])


def test_iq2_s_handbuilt_values():
    G = np.zeros((1024, 8), np.uint8)
    G[1000] = [1, 2, 3, 4, 5, 6, 7, 8]
    G[5] = [9, 9, 9, 9, 9, 9, 9, 9]
    G[256] = [100, 0, 0, 0, 0, 0, 0, 200]
    idx = [5] * 32
    idx[0], idx[3], idx[31] = 1000, 256, 1000
    sc = [2] + [0] * 14 + [15]
    w = _grid_decode("iq2_s", G, [_iq2s_block(0x3400, sc, idx, {0, 7, 255})])[0]
    # d = 0.25. Group 0 (sub-block 0, a = 0.25 * 5 = 1.25), entry 1000, elements 0 and 7
    # negative: -1.25, 2.5, 3.75, 5, 6.25, 7.5, 8.75, -10. Group 1 (elements 8..15, same
    # sub-block), entry 5: 11.25. Group 3 (elements 24..31, sub-block 1, a = 0.25), entry
    # 256: 25, 0, ..., 50. Group 31 (elements 248..255, sub-block 15, a = 0.25 * 31 = 7.75),
    # entry 1000, element 255 negative: 7.75, ..., -62.
    hand = {0: -1.25, 1: 2.5, 2: 3.75, 6: 8.75, 7: -10.0, 8: 11.25, 15: 11.25, 24: 25.0, 25: 0.0, 31: 50.0,
            16: 2.25, 248: 7.75, 254: 54.25, 255: -62.0}
    for e, v in hand.items():
        assert w[e] == v, (e, w[e], v)


@pytest.mark.parametrize("g", [0, 7, 8, 37, 63])
def test_iq3_s_index_high_bit_and_sign_positions(g):
    """Only group g takes entry 256 + 1 (its bit 8 set) and only its third element is
    negative: just those four values change."""
    G = np.zeros((512, 4), np.uint8)
    G[1] = [1, 1, 1, 1]
    G[257] = [2, 3, 4, 5]
    idx = [1] * 64
    idx[g] = 257
    w = _grid_decode("iq3_s", G, [_iq3s_block(0x3C00, [0] * 8, idx, {4 * g + 2})])[0]
    want = np.ones(256, np.float32)
    want[4 * g:4 * g + 4] = [2, 3, -4, 5]
    assert np.array_equal(w, want)


@pytest.mark.parametrize("g", [0, 3, 4, 17, 31])
def test_iq2_s_index_high_bits_and_sign_positions(g):
    """Only group g takes entry 512 + 256 + 1 (bits 8 and 9 set) and only its element 6
    is negative."""
    G = np.zeros((1024, 8), np.uint8)
    G[1] = 1
    G[769] = [2, 3, 4, 5, 6, 7, 8, 9]
    idx = [1] * 32
    idx[g] = 769
    w = _grid_decode("iq2_s", G, [_iq2s_block(0x3C00, [0] * 16, idx, {8 * g + 6})])[0]
    want = np.ones(256, np.float32)
    want[8 * g:8 * g + 8] = [2, 3, 4, 5, 6, 7, -8, 9]
    assert np.array_equal(w, want)


@pytest.mark.parametrize("fmt,k", [("iq3_s", 0), ("iq3_s", 5), ("iq2_s", 0), ("iq2_s", 9), ("iq2_s", 15)])
def test_grid_scale_nibble_positions(fmt, k):
    """Only sub-block k gets sc = 6 (scale 13); every weight is entry 0 = all ones."""
    ne, gw = (512, 4) if fmt == "iq3_s" else (1024, 8)
    sbs = 32 if fmt == "iq3_s" else 16
    G = np.ones((ne, gw), np.uint8)
    sc = [0] * (256 // sbs)
    sc[k] = 6
    mk = _iq3s_block if fmt == "iq3_s" else _iq2s_block
    w = _grid_decode(fmt, G, [mk(0x3C00, sc, [0] * (256 // gw), set())])[0]
    want = np.ones(256, np.float32)
    want[k * sbs:(k + 1) * sbs] = 13.0
    assert np.array_equal(w, want)


def test_grid_is_one_table_for_a_tower():
    """A tower is one grid, then the blocks of all its rows (as one [E*N, K] matrix)."""
    G = synth.grid(4, 512, 4, 8)
    W = synth.weights(9, 6, 512).numpy()
    c_all = oracle.encode("iq3_s", W, codebook=G)
    gb = oracle.grid_bytes("iq3_s")
    c_top = oracle.encode("iq3_s", W[:2], codebook=G)
    assert np.array_equal(c_all[:gb], G.reshape(-1)) and np.array_equal(c_top[gb:], c_all[gb:gb + 2 * 2 * 110])


@pytest.mark.parametrize("fmt", ["iq3_s", "iq2_s"])
def test_grid_encoder_takes_the_nearest_entry(fmt):
    """Brute force over the whole grid (fp64): each group's chosen entry is the nearest
    one to the group's magnitudes at the scale the block carries; signs follow the
    weights; decoded magnitudes are a * G[idx]."""
    ne, gw, lv = (512, 4, 8) if fmt == "iq3_s" else (1024, 8, 4)
    sbs = 32 if fmt == "iq3_s" else 16
    G = synth.grid(11, ne, gw, lv)
    W = synth.weights(12, 2, 512).numpy()
    c = oracle.encode(fmt, W, codebook=G)
    D = oracle.block_to_float(fmt, c, 2, 512)
    assert np.all((D < 0) <= (W < 0)) and np.all((W > 0) <= (D >= 0))
    Gf = G.astype(np.float64)
    for r in range(2):
        for g in range(512 // gw):
            k = (g * gw) // sbs
            seg = np.abs(W[r, g * gw:(g + 1) * gw]).astype(np.float64)
            got = np.abs(D[r, g * gw:(g + 1) * gw]).astype(np.float64)
            # the scale a = d (2 sc + 1) of this sub-block, read from the block's bytes
            blk = c[oracle.grid_bytes(fmt) + (r * 2 + (g * gw) // 256) * (110 if fmt == "iq3_s" else 82):]
            d = float(np.frombuffer(bytes(blk[:2]), np.float16)[0])
            kk = k % (256 // sbs)
            off = 106 if fmt == "iq3_s" else 74
            sc = (blk[off + kk // 2] >> (4 * (kk & 1))) & 15
            a = d * (2 * int(sc) + 1)
            errs = ((seg[None, :] - a * Gf) ** 2).sum(1)
            mine = ((seg - got) ** 2).sum()
            assert mine <= errs.min() * (1 + 1e-5) + 1e-12, (r, g)


# ---------------------------------------------------------------------------
# encode -> decode round trips on N(0, 0.02) data and edge blocks
# ---------------------------------------------------------------------------
def _data(rows, K, seed=0):
    W = synth.weights(seed, rows, K).numpy()
    W[0, :] = 0.0                                       # all-zero row
    W[1, :] = -np.abs(W[1, :])                          # all-negative row
    W[2, :256] = 0.0123                                 # constant block
    return W


def _f16(a):
    return np.asarray(a, dtype=np.uint16).view(np.float16).astype(np.float32)


def test_roundtrip_q8_0():
    W = _data(8, 1024)
    c = oracle.encode("q8_0", W)
    D = oracle.block_to_float("q8_0", c, 8, 1024)
    blocks = c.reshape(8, 32, 34)
    d = _f16(blocks[:, :, 0].astype(np.uint16) | (blocks[:, :, 1].astype(np.uint16) << 8))
    amax = np.abs(W.reshape(8, 32, 32)).max(-1)
    bound = 0.5 * d + 127 * np.abs(d - amax / 127) + 1e-7
    err = np.abs(W - D).reshape(8, 32, 32).max(-1)
    assert np.all(err <= bound)
    assert np.all(D[0] == 0)


def test_roundtrip_q4_k():
    W = _data(8, 1024)
    c = oracle.encode("q4_k", W)
    D = oracle.block_to_float("q4_k", c, 8, 1024)
    Wb = W.reshape(8, 4, 8, 32)
    lo = np.minimum(0, Wb.min(-1))
    hi = Wb.max(-1)
    s = (hi - lo) / 15
    # the block's step and offset after 6-bit/fp16 rounding: within 1/2 of a
    # 6-bit step of the ideal ones (plus fp16 rounding of d, dmin)
    dd = _f16(c.reshape(8, 4, 144)[:, :, 0].astype(np.uint16) | (c.reshape(8, 4, 144)[:, :, 1].astype(np.uint16) << 8))
    dm = _f16(c.reshape(8, 4, 144)[:, :, 2].astype(np.uint16) | (c.reshape(8, 4, 144)[:, :, 3].astype(np.uint16) << 8))
    bound = (0.5 * s + 15 * 0.5 * dd[..., None] + 0.5 * dm[..., None]) * (1 + 2**-9) + 1e-7
    err = np.abs(W - D).reshape(8, 4, 8, 32).max(-1)
    assert np.all(err <= bound)
    assert np.all(D[0] == 0)
    rel = np.linalg.norm(W[3:] - D[3:]) / np.linalg.norm(W[3:])
    assert rel < 0.12          # 4-bit asymmetric rounding on Gaussian data


def test_roundtrip_q5_k():
    W = _data(8, 1024)
    c = oracle.encode("q5_k", W)
    D = oracle.block_to_float("q5_k", c, 8, 1024)
    Wb = W.reshape(8, 4, 8, 32)
    lo = np.minimum(0, Wb.min(-1))
    hi = Wb.max(-1)
    s = (hi - lo) / 31
    cb = c.reshape(8, 4, 176).astype(np.uint16)
    dd = _f16(cb[:, :, 0] | (cb[:, :, 1] << 8))
    dm = _f16(cb[:, :, 2] | (cb[:, :, 3] << 8))
    # half a step of the ideal 31-level grid, plus the 6-bit rounding of sc_j
    # (up to 31 levels of it) and of m_j, plus fp16 rounding of d, dmin
    bound = (0.5 * s + 31 * 0.5 * dd[..., None] + 0.5 * dm[..., None]) * (1 + 2**-9) + 1e-7
    err = np.abs(W - D).reshape(8, 4, 8, 32).max(-1)
    assert np.all(err <= bound)
    assert np.all(D[0] == 0)
    rel5 = np.linalg.norm(W[3:] - D[3:]) / np.linalg.norm(W[3:])
    D4 = oracle.block_to_float("q4_k", oracle.encode("q4_k", W), 8, 1024)
    rel4 = np.linalg.norm(W[3:] - D4[3:]) / np.linalg.norm(W[3:])
    assert rel5 < 0.07 and rel5 < 0.65 * rel4   # one more bit: about half the error


def test_roundtrip_q6_k():
    W = _data(8, 1024)
    c = oracle.encode("q6_k", W)
    D = oracle.block_to_float("q6_k", c, 8, 1024)
    blk = c.reshape(8, 4, 210)
    d = _f16(blk[:, :, 208].astype(np.uint16) | (blk[:, :, 209].astype(np.uint16) << 8))
    sc = blk[:, :, 192:208].view(np.int8).astype(np.float32)
    step = d[..., None] * np.abs(sc)                                 # [8,4,16]
    amax = np.abs(W.reshape(8, 4, 16, 16)).max(-1)
    # rounding to the nearest step, or the clamp of +amax to code 31 (q - 32 <= 31)
    bound = np.maximum(0.5 * step, amax - 31 * step) * (1 + 2**-20) + 1e-7
    err = np.abs(W - D).reshape(8, 4, 16, 16).max(-1)
    assert np.all(err <= bound)
    rel = np.linalg.norm(W[3:] - D[3:]) / np.linalg.norm(W[3:])
    assert rel < 0.03


def test_roundtrip_nvfp4():
    W = _data(8, 1024)
    sT = np.float32(np.abs(W).max()) / np.float32(2688.0)
    c = oracle.encode("nvfp4", W, float(sT))
    D = oracle.block_to_float("nvfp4", c, 8, 1024)
    sb = np.array([oracle.e4m3_to_f32(int(v)) for v in c[8 * 512: 8 * 512 + 8 * 64]],
                  dtype=np.float32).reshape(8, 64)
    unit = sb * sT                                                   # block quantum scale
    amax = np.abs(W.reshape(8, 64, 16)).max(-1)
    # half the widest E2M1 gap (1.0 between 4 and 6) plus saturation plus the final rounding
    bound = unit * 1.0 + np.maximum(0, amax - 6 * unit) + np.abs(W).max() * 2**-23 * 4
    err = np.abs(W - D).reshape(8, 64, 16).max(-1)
    assert np.all(err <= bound + 1e-12)
    rel = np.linalg.norm(W[3:] - D[3:]) / np.linalg.norm(W[3:])
    assert rel < 0.15


def test_roundtrip_fp8_row():
    W = _data(8, 1024)
    c = oracle.encode("fp8_row", W)
    D = oracle.block_to_float("fp8_row", c, 8, 1024)
    s = np.frombuffer(c[8 * 1024:].tobytes(), dtype=np.float32)
    # relative half-ulp of a 3-bit mantissa for normals, 2^-10 s below 2^-6 s
    bound = np.maximum(np.abs(W) * 2**-4, s[:, None] * 2**-10) * (1 + 2**-20)
    assert np.all(np.abs(W - D) <= bound + 1e-12)
    assert np.all(D[0] == 0)


@pytest.mark.parametrize("cb_seed", [0, 7])
def test_roundtrip_iq4_xs(cb_seed):
    """Error of each element <= |a_j| x (half the widest gap of the codebook, or the
    codebook's shortfall on the side opposite its largest entry) + the scale's
    rounding, (d / 2) |C_ext|; all-zero rows decode to zero."""
    W = _data(8, 1024)
    cb = CB_HAND if cb_seed == 0 else list(synth.codebook(cb_seed))
    c = oracle.encode("iq4_xs", W, codebook=cb)
    assert list(c[-16:].view(np.int8)) == list(cb)
    D = oracle.block_to_float("iq4_xs", c, 8, 1024)
    blocks = c[:-16].reshape(8, 4, 136)
    d = _f16(blocks[:, :, 0].astype(np.uint16) | (blocks[:, :, 1].astype(np.uint16) << 8))
    sh = blocks[:, :, 2].astype(np.int64) | (blocks[:, :, 3].astype(np.int64) << 8)
    cbs = np.array(sorted(cb), dtype=np.float64)
    ext = cbs[np.argmax(np.abs(cbs))]
    opp = np.max(np.abs(cbs[np.sign(cbs) == -np.sign(ext)])) if np.any(np.sign(cbs) == -np.sign(ext)) else 0.0
    reach = max(np.max(np.diff(cbs)) / 2, abs(ext) - opp)
    for j in range(8):
        ls = ((blocks[:, :, 4 + j // 2].astype(np.int64) >> (4 * (j & 1))) & 15) | (((sh >> (2 * j)) & 3) << 4)
        a = d * (ls - 32)
        bound = np.abs(a) * reach + d / 2 * abs(ext) + 1e-6
        err = np.abs(W - D).reshape(8, 4, 8, 32)[:, :, j, :].max(-1)
        assert np.all(err <= bound), j
    assert np.all(D[0] == 0)
    rel = np.linalg.norm(W[3:] - D[3:]) / np.linalg.norm(W[3:])
    assert rel < 0.25


# ---------------------------------------------------------------------------
# the dot products
# ---------------------------------------------------------------------------
def test_gemv_exact_rationals_tiny():
    W = synth.weights(5, 3, 64).numpy()
    x = synth.bf16_bits(synth.activations(5, 2, 64))
    y, den = oracle.gemv_f64(W, x)
    xf = np.array([[oracle.bf16_to_f32(int(v)) for v in row] for row in x], dtype=np.float32)
    for m in range(2):
        for n in range(3):
            exact = sum(Fraction(float(W[n, k])) * Fraction(float(xf[m, k])) for k in range(64))
            ab = sum(abs(Fraction(float(W[n, k])) * Fraction(float(xf[m, k]))) for k in range(64))
            assert abs(Fraction(y[m, n]) - exact) <= ab * Fraction(64, 2**53)
            assert abs(Fraction(den[m, n]) - ab) <= ab * Fraction(64, 2**53)


@pytest.mark.parametrize("M,N,K", [(1, 256, 256), (8, 64, 256), (3, 17, 96)])
def test_gemv_vs_numpy_f64(M, N, K):
    W = synth.weights(7, N, K).numpy()
    xb = synth.activations(7, M, K)
    y, den = oracle.gemv_f64(W, synth.bf16_bits(xb))
    ref = xb.float().numpy().astype(np.float64) @ W.astype(np.float64).T
    assert np.allclose(y, ref, rtol=0, atol=1e-13 * np.abs(ref).max())
    assert np.allclose(den, np.abs(xb.float().numpy().astype(np.float64))
                       @ np.abs(W.astype(np.float64)).T, rtol=1e-12)


def test_q4_k_factored_identity_exact():
    """sum_k w_k x_k == sum_j (d sc_j) sum q x - (dmin m_j) sum x, exactly (rationals)."""
    W = synth.weights(9, 1, 256).numpy()
    c = oracle.encode("q4_k", W)
    D = oracle.block_to_float("q4_k", c, 1, 256)[0]
    x = synth.activations(9, 1, 256).float().numpy()[0]
    blk = c.tobytes()
    d = float(_f16(int.from_bytes(blk[0:2], "little")))
    dmin = float(_f16(int.from_bytes(blk[2:4], "little")))
    bits = int.from_bytes(blk[4:16], "little")
    lhs = sum(Fraction(float(D[k])) * Fraction(float(x[k])) for k in range(256))
    rhs = Fraction(0)
    for j in range(8):
        sc = (bits >> (6 * j)) & 63
        m = (bits >> (6 * (8 + j))) & 63
        sq = sum(Fraction(((blk[16 + e // 2] >> (4 * (e & 1))) & 15)) * Fraction(float(x[e]))
                 for e in range(32 * j, 32 * j + 32))
        sx = sum(Fraction(float(x[e])) for e in range(32 * j, 32 * j + 32))
        rhs += Fraction(d) * sc * sq - Fraction(dmin) * m * sx
    # the decoded w differs from (d sc) q - dmin m only by its one fp32 rounding
    tol = sum(abs(Fraction(float(x[k]))) for k in range(256)) * Fraction(float(np.abs(D).max())) * Fraction(1, 2**23)
    assert abs(lhs - rhs) <= tol


def test_q5_k_factored_identity_exact():
    """The Q5_K sum factors like Q4_K's with q = lo | hi << 4 (rationals)."""
    W = synth.weights(10, 1, 256).numpy()
    c = oracle.encode("q5_k", W)
    D = oracle.block_to_float("q5_k", c, 1, 256)[0]
    x = synth.activations(10, 1, 256).float().numpy()[0]
    blk = c.tobytes()
    d = float(_f16(int.from_bytes(blk[0:2], "little")))
    dmin = float(_f16(int.from_bytes(blk[2:4], "little")))
    bits = int.from_bytes(blk[4:16], "little")
    qh = int.from_bytes(blk[16:48], "little")
    assert qh != 0                                      # the fifth bits are in use
    lhs = sum(Fraction(float(D[k])) * Fraction(float(x[k])) for k in range(256))
    rhs = Fraction(0)
    for j in range(8):
        sc = (bits >> (6 * j)) & 63
        m = (bits >> (6 * (8 + j))) & 63
        sq = sum(Fraction(((blk[48 + e // 2] >> (4 * (e & 1))) & 15) | (((qh >> e) & 1) << 4))
                 * Fraction(float(x[e])) for e in range(32 * j, 32 * j + 32))
        sx = sum(Fraction(float(x[e])) for e in range(32 * j, 32 * j + 32))
        rhs += Fraction(d) * sc * sq - Fraction(dmin) * m * sx
    tol = sum(abs(Fraction(float(x[k]))) for k in range(256)) * Fraction(float(np.abs(D).max())) * Fraction(1, 2**23)
    assert abs(lhs - rhs) <= tol


# ---------------------------------------------------------------------------
# routing
# ---------------------------------------------------------------------------
def test_unique_experts_vs_numpy():
    ids = synth.expert_ids(0, 8, 8, 288)
    assert np.array_equal(oracle.unique_experts(ids), np.unique(ids))
    for t in range(8):
        assert len(set(ids[t].tolist())) == 8          # distinct within a token


def test_distinct_expert_formula():
    g = _golden()
    E, k = 288, 8
    expect = lambda M: E * (1 - (1 - k / E) ** M)
    assert round(expect(3), 1) == g["distinct_experts_3tok_top8_of_288"]
    assert 3 * k == g["distinct_experts_3tok_pairs"]
    assert expect(1) == pytest.approx(8.0)
    for M, tol in ((3, 0.15), (4, 0.2), (8, 0.35)):
        counts = [len(oracle.unique_experts(synth.expert_ids(s, M, k, E))) for s in range(400)]
        assert abs(np.mean(counts) - expect(M)) < tol, (M, np.mean(counts), expect(M))


def test_grouped_reference_vs_numpy():
    E, N, K, M, topk = 6, 16, 256, 3, 2
    W = synth.weights(11, E * N, K).numpy()
    canon = oracle.encode("q4_k", W)
    D = oracle.block_to_float("q4_k", canon, E * N, K)
    ids = synth.expert_ids(11, M, topk, E)
    x = synth.activations(11, M * topk, K)
    xb = synth.bf16_bits(x)
    Y, _ = oracle.grouped_f64(lambda e: D[e * N:(e + 1) * N], ids, xb, x_per_pair=True)
    xf = x.float().numpy().astype(np.float64)
    for t in range(M):
        for j in range(topk):
            e = ids[t, j]
            ref = D[e * N:(e + 1) * N].astype(np.float64) @ xf[t * topk + j]
            assert np.allclose(Y[t, j], ref, rtol=0, atol=1e-13 * np.abs(ref).max())


# ---------------------------------------------------------------------------
# NVFP4 activation quantizer
# ---------------------------------------------------------------------------
def test_quant_act_nvfp4_brute_force():
    M, K = 4, 256
    x = synth.activations(13, M, K)
    xb = synth.bf16_bits(x)
    xf = x.float().numpy()
    xf[1, 16:32] = 0.0                                  # a zero block
    xb[1, 16:32] = 0
    xs = np.float32(np.abs(xf).max()) / np.float32(2688.0)
    codes, scales = oracle.quant_act_nvfp4(xb, float(xs))
    table = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    t = np.float32(6.0) * xs
    for m in range(M):
        for b in range(K // 16):
            blk = xf[m, 16 * b:16 * b + 16]
            amax = np.float32(np.abs(blk).max())
            sb_ref = torch.tensor([amax / t], dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).item()
            assert scales[m, b] == sb_ref
            sbf = np.float32(oracle.e4m3_to_f32(int(sb_ref)))
            for i in range(16):
                e = 16 * b + i
                c = (codes[m, e // 2] >> (4 * (e & 1))) & 15
                if sb_ref == 0:
                    assert c == 0
                    continue
                v = np.float32(blk[i]) / np.float32(sbf * xs)
                d = np.abs(abs(float(v)) - table)
                best = np.flatnonzero(d == d.min())
                mag = best[0] if len(best) == 1 else [q for q in best if q % 2 == 0][0]
                if abs(float(v)) > 6:
                    mag = 7
                assert (c & 7) == mag and (c >> 3) == (1 if np.signbit(v) else 0)
    assert np.all(codes[1, 8:16] == 0) and scales[1, 1] == 0


# ---------------------------------------------------------------------------
# SwiGLU: closed forms and the identity silu(x) - silu(-x) = x
# ---------------------------------------------------------------------------
def test_swiglu_closed_forms():
    import math
    ln3 = math.log(3.0)
    # sigmoid(ln 3) = 3/4, sigmoid(-ln 3) = 1/4, sigmoid(0) = 1/2
    g = np.array([0.0, ln3, -ln3, 2 * math.log(2.0), 40.0, -40.0])
    u = np.array([5.0, 2.0, 2.0, 1.0, 0.5, 3.0])
    h = oracle.swiglu_f64(g, u)
    want = np.array([0.0, ln3 * 0.75 * 2.0, -ln3 * 0.25 * 2.0, 2 * math.log(2.0) * 0.8, 20.0, 0.0])
    assert np.allclose(h, want, rtol=1e-15, atol=1e-15)


def test_swiglu_odd_part_is_identity():
    rng = np.random.default_rng(3)
    x = rng.normal(size=1000) * 4.0
    ones = np.ones_like(x)
    d = oracle.swiglu_f64(x, ones) - oracle.swiglu_f64(-x, ones)
    assert np.allclose(d, x, rtol=1e-14, atol=1e-14)
    # linear in u
    u = rng.normal(size=1000)
    assert np.allclose(oracle.swiglu_f64(x, 3.0 * u), 3.0 * oracle.swiglu_f64(x, u), rtol=1e-15, atol=1e-15)


# ---------------------------------------------------------------------------
# W4A4: the activation quantized (static x_scale), dequantized, fp64 dots
# ---------------------------------------------------------------------------
def _bf16_bits_of(vals):
    return synth.bf16_bits(torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).reshape(1, -1))


def _bf16_of(vals):
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_quant_act_q8_handbuilt():
    """Block 0: amax = 127/16 = 7.9375, so d = 1/16 exactly and on-grid values give their
    own codes; x/d = 2.5 and 3.5 round to the even 2 and 4; -127/16 gives -127. Block 1
    is all zero: d = 0 and every code 0."""
    k = [127, -127, 0, 1, -1, 64, -64, 100] + [3] * 24
    vals = [v / 16 for v in k]
    vals[8], vals[9] = 2.5 / 16, 3.5 / 16
    x = np.concatenate([_bf16_of(vals), _bf16_of([0.0] * 32)])[None, :]
    codes, scales = oracle.quant_act_q8(x)
    assert scales[0, 0] == 0.0625 and scales[0, 1] == 0.0
    assert list(codes[0, :10]) == [127, -127, 0, 1, -1, 64, -64, 100, 2, 4]
    assert np.all(codes[0, 10:32] == 3) and np.all(codes[0, 32:] == 0)


def test_quant_act_q8_roundtrip_bound():
    x = synth.bf16_bits(synth.activations(8, 3, 1024))
    codes, scales = oracle.quant_act_q8(x)
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64).reshape(3, 32, 32)
    d = scales.astype(np.float64)[:, :, None]
    err = np.abs(xf - d * codes.astype(np.float64).reshape(3, 32, 32))
    # half a step, plus the fp32 rounding of x / d (|x / d| <= 127) that decides a near-tie
    assert np.all(err <= d * (0.5 + 128 * 2.0**-24) + 1e-30)
    assert np.all(np.abs(codes).reshape(3, 32, 32).max(-1) == 127)      # the block's largest reaches 127


def test_int8dot_on_grid_reduces_to_gemv():
    """Activations that are exact multiples of their block's d (amax = 127 d) quantize
    without error, so the int8-dot reference equals the plain GEMV on the same x."""
    rng = np.random.default_rng(5)
    q = rng.integers(-127, 128, size=(2, 256))
    q[:, ::32] = 127
    x = _bf16_of((q / 16.0).reshape(-1).tolist()).reshape(2, 256)
    W = synth.weights(6, 40, 256).numpy()
    y1, d1 = oracle.int8dot_f64(W, x)
    y2, d2 = oracle.gemv_f64(W, x)
    assert np.array_equal(y1, y2) and np.array_equal(d1, d2)


def test_int8dot_handbuilt_literal():
    """W = one row of 32 ones and 32 twos; x block 0 = 127/16 everywhere (d = 1/16, codes
    127), block 1 = -127/8 (d = 1/8, codes -127): y = 32 * 7.9375 - 2 * 32 * 15.875 =
    254 - 1016 = -762, and sum |terms| = 1270."""
    x = np.concatenate([_bf16_of([127 / 16] * 32), _bf16_of([-127 / 8] * 32)])[None, :]
    W = np.array([[1.0] * 32 + [2.0] * 32], dtype=np.float32)
    y, den = oracle.int8dot_f64(W, x)
    assert y[0, 0] == -762.0 and den[0, 0] == 1270.0
    # off the grid: x = (127/16, 1.5/16, 0, ...): d = 1/16, 1.5 rounds to 2, so the second
    # element enters as 2/16 = 0.125, not as its own 0.09375
    x2 = _bf16_of([127 / 16, 1.5 / 16] + [0.0] * 30)[None, :]
    W2 = np.array([[0.0, 1.0] + [0.0] * 30], dtype=np.float32)
    y2, _ = oracle.int8dot_f64(W2, x2)
    assert y2[0, 0] == 0.125


def test_w4a4_handbuilt_literal():
    """One token, two 16-value blocks, x_scale = 1. Block 0 has amax 6 -> block scale
    1.0; 2.59375 (bf16 of 2.6) rounds to the E2M1 value 3. Block 1 has amax 12 -> block
    scale 2.0, and 0.75 / 2 = 0.375 rounds to 0.5 -> 1.0. Worked by hand:
    y = 6*0.5 - 3*2 + 1.5*(-1) + 0*4 + 3*1 + 0.5*8 + 12*0.25 + 1*(-2) = 3.5,
    sum |terms| = 3 + 6 + 1.5 + 0 + 3 + 4 + 3 + 2 = 22.5."""
    x = np.zeros(32, dtype=np.float32)
    x[:6] = [6.0, -3.0, 1.5, 0.0, 2.6, 0.5]
    x[16:18] = [12.0, 0.75]
    W = np.zeros((1, 32), dtype=np.float32)
    W[0, :6] = [0.5, 2.0, -1.0, 4.0, 1.0, 8.0]
    W[0, 16:18] = [0.25, -2.0]
    y, den = oracle.w4a4_f64(W, _bf16_bits_of(x), 1.0)
    assert y[0, 0] == 3.5 and den[0, 0] == 22.5


def test_w4a4_handbuilt_static_scale():
    """x_scale = 0.25: block amax 1.5 -> scale e4m3(1.5 / (6 * 0.25)) = 1.0; 1.5 ->
    code 6 -> 6 * 1 * 0.25 = 1.5; bf16(0.3) = 0.30078125 -> 1.203125 -> E2M1 1 -> 0.25.
    y = 1.5 * 2 + 0.25 * 4 = 4."""
    x = np.zeros(16, dtype=np.float32)
    x[:2] = [1.5, 0.3]
    W = np.zeros((2, 16), dtype=np.float32)
    W[0, :2] = [2.0, 4.0]
    W[1, :2] = [-1.0, 0.0]
    y, den = oracle.w4a4_f64(W, _bf16_bits_of(x), 0.25)
    assert y[0].tolist() == [4.0, -1.5]
    assert den[0].tolist() == [4.0, 1.5]


def test_w4a4_on_grid_activations_reduce_to_gemv():
    """Activations already on the NVFP4 grid (E2M1 values times a power of two per
    block, each block holding its 6 * 2^k) quantize without error, so the W4A4 result
    equals the plain fp64 GEMV of the same weights."""
    rng = np.random.default_rng(17)
    M, N, K = 3, 40, 128
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=np.float32)
    x = grid[rng.integers(0, 8, size=(M, K))] * np.where(rng.random((M, K)) < 0.5, -1, 1).astype(np.float32)
    x = x.reshape(M, K // 16, 16)
    x[:, :, 0] = 6.0
    x = x * np.float32(2.0) ** rng.integers(-2, 3, size=(M, K // 16, 1)).astype(np.float32)
    x = x.reshape(M, K)
    xb = synth.bf16_bits(torch.from_numpy(x).to(torch.bfloat16))
    W = synth.weights(19, N, K).numpy()
    y, den = oracle.w4a4_f64(W, xb, 1.0)
    ref, dref = oracle.gemv_f64(W, xb)
    assert np.array_equal(y, ref) and np.array_equal(den, dref)
