#!/usr/bin/env python
"""Benchmark of the block-quantized decode GEMV on GB300.

Metric: effective weight-stream GB/s (and the fraction of HBM peak) of the M = 1
quantized GEMV. Effective GB/s = algorithmic bytes / time, where the algorithmic
bytes of a call are the canonical packed bytes of the weight rows it needs plus
the bytes of x and y (and the expert ids of a grouped call); GB = 1e9 B.

Default workload (one "step"): the Q4_K decode MLP at Qwen3.8-27B geometry, M = 1:
gate and up W[17408, 5120] and down W[5120, 17408], three GEMV calls. Other
configurations are selectable with --workload and print their own line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Inputs are seeded and synthetic (weights N(0, 0.02) quantized by the library's
quantizer, bf16 activations N(0, 1)). Every step reads its weights from HBM: the
packed weights are rotated over enough copies that the bytes between two uses of
one copy exceed 4x the L2 cache. Steps are captured in CUDA graphs (the library's
kernels only; several steps per graph when a step is small) and exactly K steps
are timed with CUDA events between a barrier and a synchronize on both sides. With N > 1 (torchrun) every rank runs the same
workload on its own GPU (replicas: the GEMV has no data-path exchange) and the
maximum time over ranks is used.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

NVFP4_TS = float(np.float32(0.12) / np.float32(2688.0))   # static per-tensor scale (generator bound)
L2_BYTES = 129 * 10**6

QWEN_HIDDEN, QWEN_MLP, QWEN_VOCAB = 5120, 17408, 248320

WORKLOADS = {
    "q4k_mlp_m1": dict(fmt="q4_k", M=1, mats=[("gate", QWEN_MLP, QWEN_HIDDEN), ("up", QWEN_MLP, QWEN_HIDDEN),
                                              ("down", QWEN_HIDDEN, QWEN_MLP)],
                       desc="Q4_K decode MLP, Qwen3.8-27B geometry: gate+up [17408,5120], down [5120,17408], M=1"),
    "q4k_mlp_fused_m1": dict(fmt="q4_k", M=1, fused=True,
                             mats=[("gate|up", QWEN_MLP, QWEN_HIDDEN), ("down", QWEN_HIDDEN, QWEN_MLP)],
                             desc="Q4_K decode MLP, Qwen3.8-27B geometry, M=1: fused gate|up [2 x 17408, 5120] "
                                  "with the SwiGLU epilogue, then down [5120,17408]"),
    "q4k_mlp_layer_m1": dict(fmt="q4_k", M=1, fused=True, layer=True,
                             mats=[("gate|up", QWEN_MLP, QWEN_HIDDEN), ("down", QWEN_HIDDEN, QWEN_MLP)],
                             desc="Q4_K decode MLP layer in one launch (qmv_mlp_layer), Qwen3.8-27B geometry, M=1: "
                                  "fused gate|up [2 x 17408, 5120] with SwiGLU, h in bf16, then down [5120,17408]"),
    "q4k_mlp_layer_m8": dict(fmt="q4_k", M=8, fused=True, layer=True,
                             mats=[("gate|up", QWEN_MLP, QWEN_HIDDEN), ("down", QWEN_HIDDEN, QWEN_MLP)],
                             desc="Q4_K decode MLP layer in one launch, Qwen3.8-27B geometry, M=8"),
    "q4k_mlp_m8": dict(fmt="q4_k", M=8, mats=[("gate", QWEN_MLP, QWEN_HIDDEN), ("up", QWEN_MLP, QWEN_HIDDEN),
                                              ("down", QWEN_HIDDEN, QWEN_MLP)],
                       desc="Q4_K decode MLP, Qwen3.8-27B geometry, M=8 (speculative verify block)"),
    "q5k_mlp_m1": dict(fmt="q5_k", M=1, mats=[("gate", QWEN_MLP, QWEN_HIDDEN), ("up", QWEN_MLP, QWEN_HIDDEN),
                                              ("down", QWEN_HIDDEN, QWEN_MLP)],
                       desc="Q5_K decode MLP, Qwen3.8-27B geometry: gate+up [17408,5120], down [5120,17408], M=1"),
    "q5k_mlp_m8": dict(fmt="q5_k", M=8, mats=[("gate", QWEN_MLP, QWEN_HIDDEN), ("up", QWEN_MLP, QWEN_HIDDEN),
                                              ("down", QWEN_HIDDEN, QWEN_MLP)],
                       desc="Q5_K decode MLP, Qwen3.8-27B geometry, M=8"),
    "q6k_head_m1": dict(fmt="q6_k", M=1, mats=[("head", QWEN_VOCAB, QWEN_HIDDEN)],
                        desc="Q6_K untied output head [248320,5120], M=1"),
    "q6k_head_m8": dict(fmt="q6_k", M=8, mats=[("head", QWEN_VOCAB, QWEN_HIDDEN)],
                        desc="Q6_K untied output head [248320,5120], M=8"),
    "q6k_qkv_m1": dict(fmt="q6_k", M=1, mats=[("attn_qkv", 10240, QWEN_HIDDEN)],
                       desc="Q6_K fused attn_qkv [10240,5120], M=1"),
    "q6k_qkv_m8": dict(fmt="q6_k", M=8, mats=[("attn_qkv", 10240, QWEN_HIDDEN)],
                       desc="Q6_K fused attn_qkv [10240,5120], M=8"),
    "nvfp4_mlp_m1": dict(fmt="nvfp4", M=1, mats=[("up", QWEN_MLP, QWEN_HIDDEN), ("down", QWEN_HIDDEN, QWEN_MLP)],
                         desc="NVFP4 MLP [17408,5120] + [5120,17408], M=1"),
    "nvfp4_mlp_m8": dict(fmt="nvfp4", M=8, mats=[("up", QWEN_MLP, QWEN_HIDDEN), ("down", QWEN_HIDDEN, QWEN_MLP)],
                         desc="NVFP4 MLP [17408,5120] + [5120,17408], M=8"),
    "fp8_m1": dict(fmt="fp8_row", M=1, mats=[("proj", 6144, QWEN_HIDDEN)],
                   desc="row-scaled FP8 projection [6144,5120], M=1"),
    "fp8_m8": dict(fmt="fp8_row", M=8, mats=[("proj", 6144, QWEN_HIDDEN)],
                   desc="row-scaled FP8 projection [6144,5120], M=8"),
    "q8_0_tiny": dict(fmt="q8_0", M=1, mats=[("tiny", 512, 1024)],
                      desc="Q8_0 tiny [512,1024], M=1"),
    "nvfp4_w4a4_m512": dict(fmt="nvfp4", M=512, w4a4=True,
                            mats=[("up", QWEN_MLP, QWEN_HIDDEN), ("down", QWEN_HIDDEN, QWEN_MLP)],
                            desc="NVFP4 W4A4 prefill, M=512: activation quantized to NVFP4, tcgen05 block-scaled "
                                 "MMA, [17408,5120] + [5120,17408]"),
    "q4k_prefill_m512": dict(fmt="q4_k", M=512, kquant=True,
                             mats=[("up", QWEN_MLP, QWEN_HIDDEN), ("down", QWEN_HIDDEN, QWEN_MLP)],
                             desc="Q4_K prefill, M=512: tcgen05 kind::f16 GEMM over exactly decoded Q4_K weights, "
                                  "[17408,5120] + [5120,17408]"),
    "q5k_prefill_m512": dict(fmt="q5_k", M=512, kquant=True,
                             mats=[("up", QWEN_MLP, QWEN_HIDDEN), ("down", QWEN_HIDDEN, QWEN_MLP)],
                             desc="Q5_K prefill, M=512: tcgen05 kind::f16 GEMM over exactly decoded Q5_K weights, "
                                  "[17408,5120] + [5120,17408]"),
    "q6k_prefill_m512": dict(fmt="q6_k", M=512, kquant=True, mats=[("attn_qkv", 10240, QWEN_HIDDEN)],
                             desc="Q6_K prefill, M=512: tcgen05 kind::f16 GEMM over exactly decoded Q6_K weights "
                                  "(scale split into two exact f16 terms), fused attn_qkv [10240,5120]"),
    "tower_m1": dict(fmt="q4_k", M=1, tower=True, E=288, topk=8,
                     mats=[("gate", 2048, 4096), ("up", 2048, 4096), ("down", 4096, 2048)],
                     desc="grouped Q4_K tower, 288 experts x (gate,up [2048,4096], down [4096,2048]), top-8, M=1"),
    "tower_m4": dict(fmt="q4_k", M=4, tower=True, E=288, topk=8,
                     mats=[("gate", 2048, 4096), ("up", 2048, 4096), ("down", 4096, 2048)],
                     desc="grouped Q4_K tower, 288 experts, top-8, M=4"),
    "tower_m8": dict(fmt="q4_k", M=8, tower=True, E=288, topk=8,
                     mats=[("gate", 2048, 4096), ("up", 2048, 4096), ("down", 4096, 2048)],
                     desc="grouped Q4_K tower, 288 experts, top-8, M=8"),
    "tower_fused_m1": dict(fmt="q4_k", M=1, tower=True, fused=True, E=288, topk=8,
                           mats=[("gate|up", 2048, 4096), ("down", 4096, 2048)],
                           desc="grouped Q4_K tower, 288 experts, top-8, M=1: fused gate|up [2 x 2048, 4096] "
                                "with the SwiGLU epilogue, then down [4096,2048]"),
    "tower_fused_m8": dict(fmt="q4_k", M=8, tower=True, fused=True, E=288, topk=8,
                           mats=[("gate|up", 2048, 4096), ("down", 4096, 2048)],
                           desc="grouped Q4_K tower, 288 experts, top-8, M=8: fused gate|up with the SwiGLU "
                                "epilogue, then down"),
    "iq4xs_tower_down_m1": dict(fmt="iq4_xs", M=1, tower=True, E=288, topk=8, mats=[("down", 4096, 2048)],
                                desc="grouped IQ4_XS down-projection tower, 288 experts [4096,2048], a 16-entry "
                                     "codebook per expert, top-8, one x row per pair, M=1"),
    "iq4xs_tower_down_m8": dict(fmt="iq4_xs", M=8, tower=True, E=288, topk=8, mats=[("down", 4096, 2048)],
                                desc="grouped IQ4_XS down-projection tower, 288 experts [4096,2048], top-8, M=8"),
    "iq2s_tower_gateup_m1": dict(fmt="iq2_s", M=1, tower=True, E=288, topk=8, pair_last=False,
                                 mats=[("gate", 2048, 4096), ("up", 2048, 4096)],
                                 desc="grouped IQ2_S gate and up towers, 288 experts [2048,4096], one grid "
                                      "(1024 x 8) per tower, top-8, M=1"),
    "iq3s_tower_down_m1": dict(fmt="iq3_s", M=1, tower=True, E=288, topk=8, mats=[("down", 4096, 2048)],
                               desc="grouped IQ3_S down-projection tower, 288 experts [4096,2048], one grid "
                                    "(512 x 4) per tower, top-8, one x row per pair, M=1"),
    "iq4xs_mlp_m1": dict(fmt="iq4_xs", M=1, mats=[("gate", QWEN_MLP, QWEN_HIDDEN), ("up", QWEN_MLP, QWEN_HIDDEN),
                                                  ("down", QWEN_HIDDEN, QWEN_MLP)],
                         desc="IQ4_XS codebook GEMV at the Qwen3.8-27B MLP shapes (gate, up [17408,5120], "
                              "down [5120,17408]), M=1"),
    "q4k_int8dot_mlp_m1": dict(fmt="q4_k", M=1, int8dot=True,
                               mats=[("gate", QWEN_MLP, QWEN_HIDDEN), ("up", QWEN_MLP, QWEN_HIDDEN),
                                     ("down", QWEN_HIDDEN, QWEN_MLP)],
                               desc="Q4_K int8-dot decode MLP (x quantized to int8 per 32 values, dp4a), "
                                    "Qwen3.8-27B geometry: gate+up [17408,5120], down [5120,17408], M=1"),
    "q4k_int8dot_mlp_m8": dict(fmt="q4_k", M=8, int8dot=True,
                               mats=[("gate", QWEN_MLP, QWEN_HIDDEN), ("up", QWEN_MLP, QWEN_HIDDEN),
                                     ("down", QWEN_HIDDEN, QWEN_MLP)],
                               desc="Q4_K int8-dot decode MLP, Qwen3.8-27B geometry, M=8"),
    "q8_0_int8dot_mlp_m1": dict(fmt="q8_0", M=1, int8dot=True,
                                mats=[("gate", QWEN_MLP, QWEN_HIDDEN), ("up", QWEN_MLP, QWEN_HIDDEN),
                                      ("down", QWEN_HIDDEN, QWEN_MLP)],
                                desc="Q8_0 int8-dot decode MLP (int8 weight codes x int8 activation codes, "
                                     "dp4a), Qwen3.8-27B geometry, M=1"),
}
DEFAULT_WORKLOAD = "q4k_mlp_m1"
DEFAULT_STEPS = {"q4k_mlp_m1": 20000, "q4k_mlp_m8": 20000, "q6k_head_m1": 2000, "q6k_head_m8": 2000,
                 "q6k_qkv_m1": 40000, "q6k_qkv_m8": 40000, "nvfp4_mlp_m1": 20000, "nvfp4_mlp_m8": 20000,
                 "fp8_m1": 40000, "fp8_m8": 40000, "q8_0_tiny": 20000, "tower_m1": 20000,
                 "tower_m4": 10000, "tower_m8": 5000, "nvfp4_w4a4_m512": 2000,
                 "q4k_mlp_fused_m1": 20000, "q4k_mlp_layer_m1": 20000, "q4k_mlp_layer_m8": 20000, "q5k_mlp_m1": 20000, "q5k_mlp_m8": 20000,
                 "tower_fused_m1": 20000, "tower_fused_m8": 5000, "q4k_prefill_m512": 2000,
                 "q5k_prefill_m512": 2000, "q6k_prefill_m512": 2000, "iq4xs_tower_down_m1": 20000, "iq4xs_tower_down_m8": 5000,
                 "iq4xs_mlp_m1": 20000, "iq2s_tower_gateup_m1": 20000, "iq3s_tower_down_m1": 20000,
                 "q4k_int8dot_mlp_m1": 20000, "q4k_int8dot_mlp_m8": 20000, "q8_0_int8dot_mlp_m1": 10000}

METRIC = "effective weight-stream GB/s and % of HBM peak for M=1 quantized GEMV"
CANON_PER_VALUE = {"q8_0": 34 / 32, "q4_k": 144 / 256, "q5_k": 176 / 256, "q6_k": 210 / 256,
                   "nvfp4": 18 / 32, "fp8_row": 1.0, "iq4_xs": 136 / 256, "iq3_s": 110 / 256, "iq2_s": 82 / 256}
# the grid formats' table (uint8 magnitudes): entries, width, levels of the seeded grid;
# read once per call on top of the routed experts' blocks
GRIDS = {"iq3_s": (512, 4, 8), "iq2_s": (1024, 8, 4)}


def canon_bytes(fmt, N, K):
    if fmt == "nvfp4":
        return N * K // 2 + N * K // 16 + 4
    if fmt == "fp8_row":
        return N * K + 4 * N
    if fmt == "iq4_xs":
        return N * (K // 256) * 136 + 16
    return int(round(N * K * CANON_PER_VALUE[fmt]))


def measured_fp4_peak():
    """Dense FP4 tensor peak: the measured bf16 GEMM rate times the nominal FP4/bf16
    ratio of the part (13.5 / 2.25 PFLOP/s)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d.get("bf16_tflops", 1900.0)) * 6.0, "measured bf16 x 6 (nominal fp4/bf16 ratio)"
    return 1900.0 * 6.0, "fallback bf16 x 6 (nominal fp4/bf16 ratio)"


def measured_f16_peak():
    """Dense f16 tensor peak: the measured bf16 GEMM rate (the part's f16 and bf16
    rates are the same)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d.get("bf16_tflops", 1900.0)), "measured bf16 (= dense f16 rate)"
    return 1900.0, "fallback bf16 (= dense f16 rate)"


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d.get("hbm_gbs", 6800.0)), "measured"
    return 6800.0, "fallback"


def kernel_unit(workload):
    """The translation unit that holds the workload's dominant kernel."""
    w = WORKLOADS[workload]
    if w.get("w4a4"):
        return "qmv_w4a4.cu"
    if w.get("int8dot"):
        return "qmv_int8.cu"
    return "qmv_kq.cu" if w.get("kquant") else "qmv_stream.cu"


def kernel_source_hash(unit):
    """Hash of what one kernel is built from: its translation unit, the host launch code
    and every header. A recorded traffic figure is used only while it matches."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_quantized_weight_fly_gb300", "csrc")
    files = [os.path.join(csrc, n) for n in sorted(os.listdir(csrc))
             if n in (unit, "qmv_api.cu") or n.endswith((".cuh", ".h"))]
    files.append(os.path.join(ROOT, "include", "qmv.h"))
    for path in files:
        with open(path, "rb") as f:
            h.update(os.path.basename(path).encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    rec = d.get(workload)
    if not rec or rec.get("kernel_hash") != kernel_source_hash(kernel_unit(workload)):
        return None
    return rec.get("dram_bytes_per_launch")


# ----------------------------------------------------------------------------
# N > 1: replicas, one per rank; the job's rate is the units of all ranks over the
# slowest rank's time
# ----------------------------------------------------------------------------
def slowest_rank_ms(ms, dev):
    """The maximum over ranks of a rank's timed-region milliseconds (every rank calls it)."""
    t = torch.tensor([float(ms)], dtype=torch.float64, device=dev)
    if torch.distributed.is_available() and torch.distributed.is_initialized() and \
            torch.distributed.get_world_size() > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_step, steps, world, ms_max):
    """Units (bytes or FLOPs) of all ranks' steps per second, over the slowest rank's time."""
    return units_per_step * steps * world / (ms_max * 1e-3)


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, smax, reasons = [], None, set()
        for line in (self.out or "").strip().splitlines():
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                smax = float(p[2])
            except ValueError:
                continue
            for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"),
                               p[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------
# device workload
# ----------------------------------------------------------------------------
def codebook_of(seed, e):
    """The IQ4_XS codebook of expert e of a seeded matrix (16 int8 values)."""
    return synth.codebook(seed + 7919 * e)


def grid_of(fmt, seed):
    """The grid of a seeded IQ3_S / IQ2_S tower (uint8 [entries, width])."""
    ne, gw, lv = GRIDS[fmt]
    return synth.grid(seed, ne, gw, lv)


def build_packed(q, fmt, seed, N, K, E, dev):
    """Seeded weights -> library quantizer -> packed device tower (load phase, untimed)."""
    chunk_rows = max(1, (1 << 26) // K)
    canon_parts = []
    if fmt in GRIDS:
        # one grid for the tower, then the blocks of all its rows
        G = grid_of(fmt, seed)
        canon_parts.append(torch.from_numpy(G.reshape(-1).copy()).to(dev))
        for r0 in range(0, E * N, chunk_rows):
            n = min(chunk_rows, E * N - r0)
            W = synth.weights(seed, n, K, device=dev, row0=r0, chunk_rows=n)
            canon_parts.append(q.qmv_quantize_codebook(fmt, W, G)[G.size:])
            del W
    for e in range(E if fmt not in GRIDS else 0):
        if fmt in ("nvfp4", "fp8_row"):
            W = synth.weights(seed, N, K, device=dev, row0=e * N, chunk_rows=chunk_rows)
            canon_parts.append(q.qmv_quantize(fmt, W, NVFP4_TS if fmt == "nvfp4" else 0.0))
            del W
        elif fmt == "iq4_xs":
            # each expert's stream: its blocks, then its own codebook
            cb = codebook_of(seed, e)
            for r0 in range(0, N, chunk_rows):
                n = min(chunk_rows, N - r0)
                W = synth.weights(seed, n, K, device=dev, row0=e * N + r0, chunk_rows=n)
                canon_parts.append(q.qmv_quantize_codebook(fmt, W, cb)[:n * (K // 256) * 136])
                del W
            canon_parts.append(torch.from_numpy(cb.view(np.uint8).copy()).to(dev))
        else:
            for r0 in range(0, N, chunk_rows):
                n = min(chunk_rows, N - r0)
                W = synth.weights(seed, n, K, device=dev, row0=e * N + r0, chunk_rows=n)
                canon_parts.append(q.qmv_quantize(fmt, W))
                del W
    canon = torch.cat(canon_parts)
    del canon_parts
    packed = q.qmv_pack(fmt, canon, N, K, E)
    del canon
    return packed


class DeviceWorkload:
    def __init__(self, q, name, dev):
        self.q, self.name, self.dev = q, name, dev
        w = WORKLOADS[name]
        self.fmt, self.M = w["fmt"], w["M"]
        self.tower = w.get("tower", False)
        self.w4a4 = w.get("w4a4", False)
        self.kquant = w.get("kquant", False)
        self.int8dot = w.get("int8dot", False)  # x quantized to int8 per 32 values (qmv_gemv_int8dot)
        self.fused = w.get("fused", False)
        self.layer = w.get("layer", False)      # the MLP layer in one launch (qmv_mlp_layer)
        self.E = w.get("E", 1)
        self.topk = w.get("topk", 1)
        self.mats = w["mats"]
        torch.cuda.synchronize()
        # fused gate|up: a tower of both matrices (gate experts first, then up)
        base = [build_packed(q, self.fmt, 100 + i, N, K, self.E * (2 if (self.fused and i == 0) else 1), dev)
                for i, (_, N, K) in enumerate(self.mats)]
        torch.cuda.synchronize()
        # bytes a step streams, to size the rotation
        if self.tower:
            per_expert = [canon_bytes(self.fmt, N, K) * (2 if (self.fused and i == 0) else 1)
                          for i, (_, N, K) in enumerate(self.mats)]
            step_w = sum(per_expert) * min(self.E, self.M * self.topk)
        else:
            step_w = sum(canon_bytes(self.fmt, N, K) * (2 if (self.fused and i == 0) else 1)
                         for i, (_, N, K) in enumerate(self.mats))
        self.copies = rotation_copies(name)
        assert self.copies == max(2, math.ceil(4 * L2_BYTES / max(step_w, 1)) + 1)
        self.packed = [base] + [[b.clone() for b in base] for _ in range(self.copies - 1)]
        # activations, outputs, workspaces
        self.x, self.y, self.ws = [], [], []
        for i, (_, N, K) in enumerate(self.mats):
            rows = self.M * self.topk if self.pair_x(i) else self.M
            self.x.append(synth.activations(200 + i, rows, K, device=dev))
            ysh = (self.M, self.topk, N) if self.tower else (self.M, N)
            self.y.append(torch.empty(ysh, dtype=torch.float32, device=dev))
            entry = q.QMV_ENTRY_GROUPED if self.tower else (q.QMV_ENTRY_W4A4 if self.w4a4 else q.QMV_ENTRY_GEMV)
            if self.kquant:
                entry = q.QMV_ENTRY_KQUANT
            if self.int8dot:
                entry = q.QMV_ENTRY_INT8DOT
            if self.fused and i == 0:
                entry = q.QMV_ENTRY_GROUPED_SWIGLU if self.tower else q.QMV_ENTRY_SWIGLU
            if self.layer:
                entry = q.QMV_ENTRY_MLP_LAYER       # one workspace, sized by gate|up's [N_ff, K_h]
                N, K = self.mats[0][1], self.mats[0][2]
            self.ws.append(q.workspace(entry, self.fmt, self.M, N, K, self.E, self.topk, device=dev))
        # W4A4: the static activation scale of each x (amax / (448 * 6)), computed once
        self.x_scale = [float(x.float().abs().max()) / 2688.0 for x in self.x] if self.w4a4 else []
        # routing: a different id set every step (cycled), like consecutive decode steps
        self.ids = []
        self.unique = []
        if self.tower:
            for s in range(64):
                ids = synth.expert_ids(1000 + s, self.M, self.topk, self.E)
                self.ids.append(torch.from_numpy(ids).to(dev))
                self.unique.append(len(np.unique(ids)))
        # W4A4 runs the activation quantizer and the GEMM per matrix
        self.launches_per_step = 1 if self.layer else len(self.mats) * (2 if (self.w4a4 or self.kquant or
                                                                              self.int8dot) else 1)

    def pair_x(self, i):
        """Tower matrices whose x has one row per (token, slot): the down projection
        (the last matrix of a layer), unless the workload holds no down projection."""
        return self.tower and i == len(self.mats) - 1 and WORKLOADS[self.name].get("pair_last", True)

    def step_flops(self):
        return sum(2.0 * self.M * N * K for _, N, K in self.mats)

    def step_bytes(self, s=0):
        """algorithmic bytes of step s (weights of the rows needed + x + y (+ ids))."""
        tot = 0
        for i, (_, N, K) in enumerate(self.mats):
            xb = self.x[i].numel() * 2
            yb = self.y[i].numel() * 4
            gb = GRIDS[self.fmt][0] * GRIDS[self.fmt][1] if self.fmt in GRIDS else 0   # the grid, once per call
            if self.tower:
                u = self.unique[s % len(self.unique)]
                wb = canon_bytes(self.fmt, N, K) * (2 if (self.fused and i == 0) else 1)
                tot += u * wb + xb + yb + self.M * self.topk * 4 + gb
            else:
                tot += canon_bytes(self.fmt, N, K) * (2 if (self.fused and i == 0) else 1) + xb + yb + gb
        return tot

    def launch_step(self, s):
        q = self.q
        c = s % self.copies
        if self.layer:
            (_, N_ff, K_h) = self.mats[0]
            q.qmv_mlp_layer(self.fmt, self.packed[c][0], self.packed[c][1], self.x[0], N_ff, K_h, self.ws[0],
                            y=self.y[1])
            return
        for i, (_, N, K) in enumerate(self.mats):
            if self.tower and self.fused and i == 0:
                q.qmv_grouped_swiglu(self.fmt, self.packed[c][i], self.ids[s % len(self.ids)], self.x[i], N, K,
                                     self.E, self.ws[i], h=self.y[i])
            elif self.tower:
                q.qmv_grouped(self.fmt, self.packed[c][i], self.ids[s % len(self.ids)], self.x[i], N, K, self.E,
                              self.ws[i], x_per_pair=self.pair_x(i), y=self.y[i])
            elif self.fused and i == 0:
                q.qmv_gemv_swiglu(self.fmt, self.packed[c][i], self.x[i], N, K, self.ws[i], h=self.y[i])
            elif self.kquant:
                q.qmv_gemm_kquant(self.fmt, self.packed[c][i], self.x[i], N, K, self.ws[i], y=self.y[i])
            elif self.int8dot:
                q.qmv_gemv_int8dot(self.fmt, self.packed[c][i], self.x[i], N, K, self.ws[i], y=self.y[i])
            elif self.w4a4:
                q.qmv_gemm_nvfp4_w4a4(self.packed[c][i], self.x[i], self.x_scale[i], N, K, self.ws[i], y=self.y[i])
            else:
                q.qmv_gemv(self.fmt, self.packed[c][i], self.x[i], N, K, self.ws[i], y=self.y[i])

    def steps_per_graph(self):
        """Steps captured per CUDA graph: about 1 GB of weights per graph (at most
        256 steps), so that consecutive calls stay inside one graph, where each
        call's prologue overlaps the previous call (programmatic launch edges),
        and replaying graphs is never host-bound."""
        return max(1, min(256, math.ceil(1e9 / max(self.step_bytes(0), 1))))

    def graphs(self, K):
        """CUDA graphs of `u` consecutive steps each (copy index = step % copies,
        routing index = step % 64), and one graph of the K % u remaining steps."""
        period = self.copies if not self.tower else math.lcm(self.copies, len(self.ids))
        period = min(period, 256)
        # whole rotation periods per graph, so that graph boundaries keep the
        # distance between two uses of one weight copy
        u = min(256, period * -(-self.steps_per_graph() // period))
        ngraphs = max(1, -(-period // u))
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for i in range(min(period, 64)):
                self.launch_step(i)       # warm (kernel attributes, module load)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        gs = []
        for k in range(ngraphs):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for j in range(u):
                    self.launch_step(k * u + j)
            gs.append(g)
        rem = None
        if K % u:
            rem = torch.cuda.CUDAGraph()
            with torch.cuda.graph(rem):
                for j in range(K % u):
                    self.launch_step(ngraphs * u + j)
        torch.cuda.synchronize()
        return gs, rem, u


def run_device(args, rank, world, dev):
    import block_quantized_weight_fly_gb300 as q
    wl = DeviceWorkload(q, args.workload, dev)
    K, W = args.steps, args.warmup
    graphs, rem_graph, u = wl.graphs(K)
    period = len(graphs)
    for i in range(max(1, -(-W // u))):
        graphs[i % period].replay()
    torch.cuda.synchronize()
    if q.qmv_device_status() != 0:
        raise RuntimeError("device status error during warm-up")
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        start.record()
        for i in range(K // u):
            graphs[(W + i) % period].replay()
        if rem_graph is not None:
            rem_graph.replay()
        end.record()
        end.synchronize()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms = start.elapsed_time(end)
    status = q.qmv_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    ms_max = slowest_rank_ms(ms, dev)
    step_bytes = [wl.step_bytes(W + i) for i in range(min(K, period))]
    bytes_per_step = sum(step_bytes) / len(step_bytes)
    value = whole_job_rate(bytes_per_step, K, world, ms_max) / 1e9
    launches = K * wl.launches_per_step
    avg_launch_s = (ms * 1e-3) / launches
    achieved = (bytes_per_step / wl.launches_per_step) / avg_launch_s / 1e9
    peak, peak_kind = measured_peaks()
    traffic = recorded_traffic(args.workload)
    if wl.int8dot:
        # one unit per matrix: the x quantizer (a few KB) and the GEMV it feeds
        avg_launch_s = (ms * 1e-3) / (K * len(wl.mats))
        achieved = (bytes_per_step / len(wl.mats)) / avg_launch_s / 1e9
    if wl.w4a4 or wl.kquant:
        # a dense contraction: TFLOP/s against the tensor roofline; each matrix's
        # time includes its activation quantizer (the GEMM's share is in profiles/)
        flops = wl.step_flops()
        value = whole_job_rate(flops, K, world, ms_max) / 1e12
        gemm_s = (ms * 1e-3) / (K * len(wl.mats))
        achieved = (flops / len(wl.mats)) / gemm_s / 1e12
        peak, peak_kind = measured_fp4_peak() if wl.w4a4 else measured_f16_peak()

    # ---- end to end through the public API, host buffers -------------------
    e2e_steps = min(K, 2000)
    hx = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in wl.x]
    for h, x in zip(hx, wl.x):
        h.copy_(x.cpu())
    hy = [torch.empty(y.shape, dtype=y.dtype, pin_memory=True) for y in wl.y]
    h2d = sum(h.numel() * h.element_size() for h in hx)
    d2h = sum(h.numel() * h.element_size() for h in hy)
    stream = torch.cuda.current_stream()
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e_start.record()
    for i in range(e2e_steps):
        for h, x in zip(hx, wl.x):
            x.copy_(h, non_blocking=True)
        wl.launch_step(W + i)
        for h, y in zip(hy, wl.y):
            h.copy_(y, non_blocking=True)
        stream.synchronize()
    e_end.record()
    e_end.synchronize()
    e2e_ms = e_start.elapsed_time(e_end)
    e2e_bytes = sum(wl.step_bytes(W + i) for i in range(e2e_steps))
    e2e_value = e2e_bytes * world / (e2e_ms * 1e-3) / 1e9

    result = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(ms_max / K, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16" if wl.fmt in ("nvfp4", "fp8_row") else "bf16",
        "data": "synthetic (seeded N(0,0.02) weights quantized by the library, bf16 N(0,1) activations)",
        "config": workload_config(args.workload),
        "details": {
            "bytes_per_step": int(bytes_per_step),
            "rotation": f"{wl.copies} copies x {int(bytes_per_step / 1e6)} MB per cycle",
            "graph": f"CUDA graphs of {u} step(s) each",
            "arithmetic": "weights decoded exactly to " + ("f16" if wl.fmt in ("nvfp4", "fp8_row") else "bf16")
                          + ", products on mma.sync, fp32 accumulation",
            "parallelism": "replicas" if world > 1 else "single-gpu",
        },
        "pct_of_peak": round(100.0 * value / world / peak, 2),
        "pct_of_nominal_8000": round(100.0 * value / world / 8000.0, 2),
        "roofline": {
            "bound": "hbm",
            "kernel": (f"qmv::layer_kernel<{wl.fmt}, M={wl.M}>" if wl.layer else
                       f"qmv::stream_kernel<{wl.fmt}, M={wl.M}>" + (" (grouped)" if wl.tower else "")),
            "achieved": round(achieved, 2),
            "peak": peak,
            "peak_kind": peak_kind,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic,
            "avg_launch_us": round(avg_launch_s * 1e6, 3),
            "algorithmic_bytes_per_launch": int(bytes_per_step / (len(wl.mats) if wl.int8dot
                                                                  else wl.launches_per_step)),
        },
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "steps": e2e_steps,
                "ms_per_step": round(e2e_ms / e2e_steps, 6)},
        "gpu_launches": launches,
        "clocks": clk.summary(),
    }
    if wl.w4a4:
        result["metric"] = "NVFP4 W4A4 prefill throughput (M=512)"
        result["unit"] = "TFLOP/s"
        result["dtype"] = "fp4 (e2m1 x e2m1, ue4m3 block scales, fp32 accumulation)"
        result["details"]["arithmetic"] = "tcgen05.mma kind::mxf4nvf4 block_scale scale_vec::4X, TMEM fp32 accumulators"
        del result["pct_of_nominal_8000"]
        result["pct_of_peak"] = round(100.0 * value / world / peak, 2)
        result["roofline"].update({
            "bound": "tensor", "kernel": "qmv::w4a4_kernel (+ its activation quantizer)", "unit": "TFLOP/s",
            "achieved": round(achieved, 2), "peak": round(peak, 1), "frac": round(achieved / peak, 4),
            "avg_launch_us": round(gemm_s * 1e6, 3),
            "algorithmic_flops_per_launch": wl.step_flops() / len(wl.mats)})
        del result["roofline"]["algorithmic_bytes_per_launch"]
        result["e2e"]["unit"] = "TFLOP/s"
        result["e2e"]["value"] = round(wl.step_flops() * e2e_steps * world / (e2e_ms * 1e-3) / 1e12, 2)
    if wl.kquant:
        result["metric"] = f"{wl.fmt.upper()} prefill GEMM throughput (M=512)"
        result["unit"] = "TFLOP/s"
        result["dtype"] = f"f16 (exactly decoded {wl.fmt.upper()} sc*q x f16 x, fp32 accumulation)"
        result["details"]["arithmetic"] = ("tcgen05.mma kind::f16, per-superblock TMEM accumulators folded with "
                                           "d and dmin in fp32")
        del result["pct_of_nominal_8000"]
        result["pct_of_peak"] = round(100.0 * value / world / peak, 2)
        result["roofline"].update({
            "bound": "tensor", "kernel": "qmv::kq_kernel (+ its x pre-pass)", "unit": "TFLOP/s",
            "achieved": round(achieved, 2), "peak": round(peak, 1), "frac": round(achieved / peak, 4),
            "avg_launch_us": round(gemm_s * 1e6, 3),
            "algorithmic_flops_per_launch": wl.step_flops() / len(wl.mats)})
        del result["roofline"]["algorithmic_bytes_per_launch"]
        result["e2e"]["unit"] = "TFLOP/s"
        result["e2e"]["value"] = round(wl.step_flops() * e2e_steps * world / (e2e_ms * 1e-3) / 1e12, 2)
    if wl.int8dot:
        result["dtype"] = "int8 (weight codes x int8 activation codes, int32 dp4a, fp32 scaling)"
        result["details"]["arithmetic"] = ("x quantized to int8 per 32 values (d = amax/127); dp4a int32 dots "
                                           "of the weight codes, scaled in fp32 by the block scales and d")
        result["roofline"]["kernel"] = f"qmv::int8dot_kernel<{wl.fmt}, M={wl.M}> (+ its x quantizer)"
    if wl.tower:
        result["details"]["unique_experts_mean"] = round(float(np.mean(wl.unique)), 2)
    return result


# ----------------------------------------------------------------------------
# CPU oracle
# ----------------------------------------------------------------------------
def oracle_sample(workload, rows_per_mat):
    """Canonical bytes of the first rows of each matrix of the workload (oracle
    encoder), x rows, and the canonical bytes they hold. Untimed preparation."""
    import oracle
    w = WORKLOADS[workload]
    fmt = w["fmt"]
    items = []
    for i, (_, N, K) in enumerate(w["mats"]):
        r = min(rows_per_mat[i], N)
        W = synth.weights_rows(100 + i, np.arange(r), K).numpy()
        table = codebook_of(100 + i, 0) if fmt == "iq4_xs" else (grid_of(fmt, 100 + i) if fmt in GRIDS else None)
        canon = oracle.encode(fmt, W, NVFP4_TS if fmt == "nvfp4" else 0.0, codebook=table)
        x = synth.bf16_bits(synth.activations(200 + i, w["M"], K))
        items.append((fmt, canon, r, K, x, bool(w.get("int8dot"))))
    return items


def rotation_copies(workload):
    """Packed weight copies the GPU arm rotates over: the bytes between two uses of one
    copy exceed 4x the L2 cache (a function of the workload only)."""
    w = WORKLOADS[workload]
    fused, E = w.get("fused", False), w.get("E", 1)
    per = [canon_bytes(w["fmt"], N, K) * (2 if (fused and i == 0) else 1) for i, (_, N, K) in enumerate(w["mats"])]
    step_w = sum(per) * (min(E, w["M"] * w.get("topk", 1)) if w.get("tower") else 1)
    return max(2, math.ceil(4 * L2_BYTES / max(step_w, 1)) + 1)


def workload_config(workload):
    """The `config` of both arms' JSON lines: what names the workload (its shapes,
    format, batch) and how the timed region defeats L2; nothing about one arm's
    implementation, so that the two arms' configs compare equal."""
    w = WORKLOADS[workload]
    cfg = {"workload": w["desc"], "workload_id": workload, "weights": w["fmt"], "M": w["M"],
           "matrices": [f"{n}[{N},{K}]" + (f"x{w.get('E', 1)}" if w.get("tower") else "") for n, N, K in w["mats"]],
           "l2": f"inputs larger than L2: weights rotated over {rotation_copies(workload)} copies"}
    if w.get("tower"):
        cfg["topk"] = w["topk"]
    if tensor_workload(workload):
        cfg["flops_per_step"] = sum(2.0 * w["M"] * N * K for _, N, K in w["mats"])
    return cfg


def tensor_workload(workload):
    w = WORKLOADS[workload]
    return bool(w.get("w4a4") or w.get("kquant"))


def metric_of(workload):
    """(metric, unit) of the workload's JSON line (both arms)."""
    w = WORKLOADS[workload]
    if w.get("w4a4"):
        return "NVFP4 W4A4 prefill throughput (M=512)", "TFLOP/s"
    if w.get("kquant"):
        return f"{w['fmt'].upper()} prefill GEMM throughput (M=512)", "TFLOP/s"
    return METRIC, "GB/s"


def time_oracle(items, min_seconds):
    """Runs the oracle over the sample until min_seconds have passed: (bytes, flops,
    seconds, passes)."""
    import oracle
    done_bytes, done_flops, reps = 0, 0, 0
    t0 = time.perf_counter()
    while True:
        for fmt, canon, r, K, x, int8 in items:
            D = oracle.block_to_float(fmt, canon, r, K)
            (oracle.int8dot_f64 if int8 else oracle.gemv_f64)(D, x)
            done_bytes += canon.size + x.size * 2 + r * x.shape[0] * 4
            done_flops += 2 * r * K * x.shape[0]
        reps += 1
        if time.perf_counter() - t0 >= min_seconds:
            break
    return done_bytes, done_flops, time.perf_counter() - t0, reps


def cpu_baseline(workload, seconds=10.0):
    w = WORKLOADS[workload]
    # about the same canonical bytes from each matrix (~4.4 MB each for the MLP)
    rows = [max(1, int(4.4e6 / canon_bytes(w["fmt"], 1, K))) for _, _, K in w["mats"]]
    if tensor_workload(workload):
        # M = 512 rows of x: fewer weight rows for the same CPU time
        rows = [max(1, r // 64) for r in rows]
    items = oracle_sample(workload, rows)
    nbytes, nflops, secs, reps = time_oracle(items, seconds)
    sample = ", ".join(f"{n}: first {r} rows" for (n, _, _), r in zip(w["mats"], rows))
    _, unit = metric_of(workload)
    value = nflops / secs / 1e12 if unit == "TFLOP/s" else nbytes / secs / 1e9
    return {"value": round(value, 6), "unit": unit, "cores": 1, "kind": "oracle",
            "sample": f"{sample} (BlockToFloat + fp64 dot, {reps} passes, {secs:.1f} s)"}


def run_reference(args):
    """--impl reference: the CPU oracle as it stands, one bounded sample per step."""
    w = WORKLOADS[args.workload]
    K, W = args.steps, args.warmup
    budget = 150.0                                 # seconds for the whole run
    probe = oracle_sample(args.workload, [16] * len(w["mats"]))
    nb, nf, secs, _ = time_oracle(probe, 0.0)
    per_row_s = secs / (16 * len(w["mats"]))
    rows = max(1, int(budget / max(K + W, 1) / max(per_row_s * len(w["mats"]), 1e-9)))
    items = oracle_sample(args.workload, [rows] * len(w["mats"]))
    import oracle
    for _ in range(W):
        for fmt, canon, r, K_, x, int8 in items:
            (oracle.int8dot_f64 if int8 else oracle.gemv_f64)(oracle.block_to_float(fmt, canon, r, K_), x)
    nbytes, nflops = 0, 0
    t0 = time.perf_counter()
    for _ in range(K):
        for fmt, canon, r, K_, x, int8 in items:
            (oracle.int8dot_f64 if int8 else oracle.gemv_f64)(oracle.block_to_float(fmt, canon, r, K_), x)
            nbytes += canon.size + x.size * 2 + r * x.shape[0] * 4
            nflops += 2 * r * K_ * x.shape[0]
    secs = time.perf_counter() - t0
    metric, unit = metric_of(args.workload)
    value = nflops / secs / 1e12 if unit == "TFLOP/s" else nbytes / secs / 1e9
    sample = "per step: " + ", ".join(f"{n}: first {min(rows, N)} rows" for n, N, _ in w["mats"])
    return {
        "metric": metric, "value": round(value, 6), "unit": unit, "n_gpus": args.gpus, "steps": K, "warmup": W,
        "ms_per_step": round(secs * 1e3 / max(K, 1), 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args.workload),
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def read_ceiling(dev, gib=4, reps=10):
    """Read-side HBM ceiling: a PyTorch sum over a bf16 buffer of `gib` GiB (larger than
    L2), timed with CUDA events after warm-up. A library reduction, not this library's
    kernel: context for the roofline, whose peak stays the measured copy bandwidth."""
    n = gib * (1 << 30) // 2
    buf = torch.ones(n, dtype=torch.bfloat16, device=dev)
    for _ in range(3):
        buf.sum(dtype=torch.float32)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        buf.sum(dtype=torch.float32)
    e1.record()
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / reps
    nbytes = n * 2
    del buf
    return {"read_probe": "torch bf16 sum", "bytes": nbytes, "ms": round(ms, 4),
            "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1)}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--read-probe", action="store_true",
                    help="print the read-only HBM ceiling (a PyTorch sum over 4 GiB) and exit")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = DEFAULT_STEPS[args.workload]
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus and world > 1:
        args.gpus = world

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args)), flush=True)
        return

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if args.read_probe:
        print(json.dumps(read_ceiling(dev)), flush=True)
        return
    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group("nccl", device_id=dev)
    try:
        result = run_device(args, rank, world, dev)
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            result["cpu_baseline"] = cpu_baseline(args.workload)
        if rank == 0:
            print(json.dumps(result), flush=True)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
