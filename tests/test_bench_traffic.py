"""Host-side parts of the benchmark's roofline and clock records: each recorded DRAM
traffic figure is keyed by the sources of its own kernel, so editing one kernel
invalidates that kernel's record and no other; the SM clock summary is parsed from
nvidia-smi's CSV lines."""
import importlib.util
import json
import os
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_every_workload_maps_to_a_kernel_source(bench):
    csrc = os.path.join(ROOT, "block_quantized_weight_fly_gb300", "csrc")
    for name, w in bench.WORKLOADS.items():
        unit = bench.kernel_unit(name)
        assert os.path.exists(os.path.join(csrc, unit)), (name, unit)
        if w.get("w4a4"):
            assert unit == "qmv_w4a4.cu"
        elif w.get("kquant"):
            assert unit == "qmv_kq.cu"
        elif w.get("int8dot"):
            assert unit == "qmv_int8.cu"
        else:
            assert unit == "qmv_stream.cu"


def _tree(tmp_path):
    pkg = tmp_path / "block_quantized_weight_fly_gb300"
    shutil.copytree(os.path.join(ROOT, "block_quantized_weight_fly_gb300", "csrc"), pkg / "csrc")
    shutil.copytree(os.path.join(ROOT, "include"), tmp_path / "include")
    return pkg / "csrc"


def test_hash_follows_its_own_sources(bench, tmp_path, monkeypatch):
    csrc = _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    units = ("qmv_stream.cu", "qmv_kq.cu", "qmv_w4a4.cu")
    before = {u: bench.kernel_source_hash(u) for u in units}
    assert len(set(before.values())) == 3
    with open(csrc / "qmv_kq.cu", "a") as f:             # one kernel's translation unit
        f.write("\n")
    after = {u: bench.kernel_source_hash(u) for u in units}
    assert after["qmv_kq.cu"] != before["qmv_kq.cu"]
    assert after["qmv_stream.cu"] == before["qmv_stream.cu"]
    assert after["qmv_w4a4.cu"] == before["qmv_w4a4.cu"]
    with open(csrc / "qmv_api.cu", "a") as f:            # the host launch code: every kernel
        f.write("\n")
    again = {u: bench.kernel_source_hash(u) for u in units}
    assert all(again[u] != after[u] for u in units)
    with open(tmp_path / "include" / "qmv.h", "a") as f:  # the public header: every kernel
        f.write("\n")
    last = {u: bench.kernel_source_hash(u) for u in units}
    assert all(last[u] != again[u] for u in units)


def test_stale_record_is_not_reported(bench, tmp_path, monkeypatch):
    csrc = _tree(tmp_path)
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec = {"q4k_mlp_m1": {"kernel_hash": bench.kernel_source_hash("qmv_stream.cu"),
                          "dram_bytes_per_launch": 123},
           "q4k_prefill_m512": {"kernel_hash": bench.kernel_source_hash("qmv_kq.cu"),
                                "dram_bytes_per_launch": 456}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.recorded_traffic("q4k_mlp_m1") == 123
    assert bench.recorded_traffic("q4k_prefill_m512") == 456
    assert bench.recorded_traffic("tower_m1") is None         # no record
    with open(csrc / "qmv_stream.cu", "a") as f:
        f.write("\n")
    assert bench.recorded_traffic("q4k_mlp_m1") is None       # its kernel changed
    assert bench.recorded_traffic("q4k_prefill_m512") == 456  # another kernel's record stands


def test_committed_records_name_known_workloads(bench):
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        d = json.load(f)
    for name, rec in d.items():
        assert name in bench.WORKLOADS, name
        assert rec["dram_bytes_per_launch"] > 0
        assert len(rec["kernel_hash"]) == 16
        # the full command: the plain run, then the same command under ncu
        src = rec["source"]
        assert " && ncu " in src and "--clock-control none" in src, src
        plain, profiled = src.split(" && ", 1)
        assert plain.startswith("python bench.py ") and plain.split(" > ")[0] in profiled


def test_clock_summary_parses_nvidia_smi_lines(bench):
    s = bench.ClockSampler(0)
    s.out = "\n".join([
        "0, 2070, 2070, 812.40, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1390.10, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1401.00, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "garbage line",
        "0, [N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ])
    d = s.summary()
    assert d["sm_mhz"] == 2070.0 and d["sm_max_mhz"] == 2070.0 and d["samples"] == 3
    assert d["reasons"] == ["sw_power_cap"]
    s.out = "0, 1500, 2070, 900, 0x8, Active, Not Active, Active, Not Active"
    assert bench.ClockSampler.summary(s)["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    s.out = ""
    assert s.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
