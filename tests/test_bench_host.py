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


def _write_record(tmp_path, src_text, workload, nbytes, kernel="k", units=None,
                  kind="traffic_record"):
    src = tmp_path / "kernel.cu"
    src.write_text(src_text)
    h = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    prof = tmp_path / "profiles"
    prof.mkdir(exist_ok=True)
    rec = {"kernel": kernel, "workload": workload, "dram_bytes_per_launch": nbytes,
           "src_sha256": h}
    if units is not None:
        rec["units"] = units
    (prof / "k_profile.md").write_text("# summary\n\n| a | b |\n\n" + kind + ": " +
                                       json.dumps(rec) + "\n")
    return str(prof), str(src)


def _get(prof, src, wl, kernel="k"):
    return bench.traffic_record(kernel, src, "dram_bytes_per_launch", wl, prof)


def test_traffic_record_matches_source_kernel_and_workload(tmp_path):
    prof, src = _write_record(tmp_path, "__global__ void k() {}\n", "mistral_t1024", 123456789)
    assert _get(prof, src, kvgen.WORKLOADS["mistral_t1024"]) == 123456789
    assert _get(prof, src, kvgen.WORKLOADS["llama_t1024"]) is None    # another workload
    assert _get(prof, src, kvgen.WORKLOADS["mistral_t1024"], "other") is None


def test_traffic_record_scales_a_smaller_capture_by_units(tmp_path):
    prof, src = _write_record(tmp_path, "x", "llama_t1024", 1000, units=4)
    w = kvgen.WORKLOADS["llama_t1024"]
    assert _get(prof, src, w) == 1000 * w.n_units // 4
    assert _get(prof, src, kvgen.custom_workload("llama_t1024", n_groups=2)) == 1000


def test_traffic_record_is_dropped_when_the_source_changes(tmp_path):
    prof, src = _write_record(tmp_path, "__global__ void k() {}\n", "mistral_t1024", 5)
    with open(src, "a") as f:
        f.write("// edited\n")
    assert _get(prof, src, kvgen.WORKLOADS["mistral_t1024"]) is None


def test_traffic_record_missing_files(tmp_path):
    prof, src = _write_record(tmp_path, "x", "mistral_t1024", 5)
    w = kvgen.WORKLOADS["mistral_t1024"]
    assert _get(str(tmp_path / "none"), src, w) is None
    assert _get(prof, str(tmp_path / "none.cu"), w) is None


def test_tensor_records_are_read_by_kind(tmp_path):
    prof, src = _write_record(tmp_path, "x", "llama_t1024", 5, kernel="gram_tok_tc_kernel",
                              kind="tensor_record")
    recs = bench.profile_records("tensor_record", src, "llama_t1024", prof)
    assert [r["kernel"] for r in recs] == ["gram_tok_tc_kernel"]
    assert bench.profile_records("traffic_record", src, "llama_t1024", prof) == []


def test_committed_profile_records_are_well_formed():
    import glob
    n = 0
    for f in glob.glob(os.path.join(ROOT, "profiles", "*.md")):
        for line in open(f).read().splitlines():
            kind = line.split(":", 1)[0]
            if kind not in ("traffic_record", "tensor_record"):
                continue
            rec = json.loads(line.split(":", 1)[1])
            assert rec["workload"] in kvgen.WORKLOADS, f
            assert isinstance(rec["kernel"], str) and rec["kernel"], f
            assert len(rec["src_sha256"]) == 16 and int(rec["src_sha256"], 16) >= 0, f
            if kind == "traffic_record":
                key = "dram_bytes_per_call" if "dram_bytes_per_call" in rec else \
                    "dram_bytes_per_launch"
                assert int(rec[key]) > 0, f
            else:
                assert 0.0 <= float(rec["tensor_pipe_active_pct"]) <= 100.0, f
            n += 1
    assert n >= 1


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
