"""Host-side pieces of bench.py on CPU (no GPU): the traffic records that tie
committed ncu DRAM counters to the kernel source they were taken on, and the
sweep roofline's flop accounting."""
import hashlib
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench   # noqa: E402
import kvgen   # noqa: E402


def _write_record(tmp_path, src_text, workload, nbytes, key="k_src_sha256"):
    src = tmp_path / "kernel.cu"
    src.write_text(src_text)
    h = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    prof = tmp_path / "profile.md"
    rec = {"workload": workload, "dram_bytes_per_launch": nbytes, key: h}
    prof.write_text("# summary\n\n| a | b |\n\ntraffic_record: " + json.dumps(rec) + "\n")
    return str(prof), str(src)


def test_traffic_record_matches_source_and_workload(tmp_path):
    prof, src = _write_record(tmp_path, "__global__ void k() {}\n", "mistral_t1024", 123456789)
    get = lambda wl: bench.traffic_record(prof, src, "k_src_sha256", "dram_bytes_per_launch", wl)
    assert get("mistral_t1024") == 123456789
    assert get("llama_t1024") is None                    # counters of another workload


def test_traffic_record_is_dropped_when_the_source_changes(tmp_path):
    prof, src = _write_record(tmp_path, "__global__ void k() {}\n", "mistral_t1024", 5)
    with open(src, "a") as f:
        f.write("// edited\n")
    assert bench.traffic_record(prof, src, "k_src_sha256", "dram_bytes_per_launch",
                                "mistral_t1024") is None


def test_traffic_record_missing_files_or_keys(tmp_path):
    prof, src = _write_record(tmp_path, "x", "mistral_t1024", 5)
    assert bench.traffic_record(str(tmp_path / "none.md"), src, "k_src_sha256",
                                "dram_bytes_per_launch", "mistral_t1024") is None
    assert bench.traffic_record(prof, str(tmp_path / "none.cu"), "k_src_sha256",
                                "dram_bytes_per_launch", "mistral_t1024") is None
    # a record keyed for another kernel's source never matches
    assert bench.traffic_record(prof, src, "other_src_sha256", "dram_bytes_per_launch",
                                "mistral_t1024") is None


@pytest.mark.parametrize("path,key,bkey", [
    (bench.DECODE_PROFILE, "decode_src_sha256", "dram_bytes_per_launch"),
    (bench.ATTEND_PROFILE, "attend_src_sha256", "dram_bytes_per_call"),
    (bench.SWEEP_PROFILE, "sweep_src_sha256", "dram_bytes_per_launch"),
])
def test_committed_profiles_carry_one_well_formed_record(path, key, bkey):
    lines = [l for l in open(path).read().splitlines() if l.startswith("traffic_record:")]
    assert len(lines) == 1
    rec = json.loads(lines[0].split(":", 1)[1])
    assert rec["workload"] in kvgen.WORKLOADS
    assert len(rec[key]) == 16 and int(rec[key], 16) >= 0
    assert int(rec[bkey]) > 0


def test_sweep_roofline_counts_650_flops_per_element_on_the_5x5x4_grid():
    w = kvgen.WORKLOADS["mistral_t1024"]
    assert (len(w.rT), len(w.rd), tuple(w.bits)) == (5, 5, (0, 2, 4, 8))
    r = bench.roofline(w, 1e-3, 6500.0, "measured", {"sm_max_mhz": 2032.0})
    # per rank pair: residual 2, max 1, b = 0 square 2, and 7 for each b > 0
    assert r["flops_per_element"] == 25 * (2 + 1 + 2 + 3 * 7) == 650
    assert r["peak"] == pytest.approx(148 * 128 * 2 * 2.032e9 / 1e12)
    elems = w.n_units * w.elems_per_unit
    assert r["achieved"] == pytest.approx(650 * elems / 1e-3 / 1e12)
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"])
    assert r["bound"] == "alu" and r["unit"] == "TFLOP/s"
