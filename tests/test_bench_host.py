"""bench.py's host-side logic, without a GPU: the stream rotation that keeps a
step's inputs out of L2, the clock summary and its throttle reasons, the
recorded DRAM traffic (present exactly while the kernel sources match the
capture), and the reference arm's one JSON line (the CPU oracle)."""
import json
import os
import subprocess
import sys

import pytest

import bench
import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_stream_rotation_reads_every_step_from_hbm():
    # a decode step's 16.8 MB of streams (in and out twice that) and 25.2 MB of rows fit
    # in L2: rotate input sets until they exceed it twice
    dec = W.by_name("decode_fp8")
    n = bench.stream_rotation(dec)
    assert bench.step_footprint(dec) == 512 * 4 * 4096 * 2 * 2 + 512 * 12 * 4100
    assert n > 1 and n * bench.step_footprint(dec) >= 2 * bench.L2_BYTES
    assert (n - 1) * bench.step_footprint(dec) < 2 * bench.L2_BYTES   # no more sets than needed
    for name in ("mid_prefill_fp8", "full_prefill_fp8", "release_layout_fp8"):
        assert bench.stream_rotation(W.by_name(name)) == 1
    assert "rotation" in bench.l2_note(dec) and "no flush" in bench.l2_note(W.by_name("mid_prefill_fp8"))


def test_clock_summary_median_and_reasons():
    cs = object.__new__(bench.ClockSampler)
    cs.samples = [(1.0, "2070, 2070, 900.5, Not Active, Not Active, Not Active, Not Active"),
                  (2.0, "1950, 2070, 1370.0, Not Active, Not Active, Not Active, Active"),
                  (3.0, "1800, 2070, 1380.0, Not Active, Not Active, Not Active, Active"),
                  (9.0, "300, 2070, 100.0, Active, Not Active, Not Active, Not Active")]
    s = cs.summary(0.5, 3.5)     # the last sample is outside the timed region
    assert s["sm_mhz"] == 1950 and s["sm_max_mhz"] == 2070 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"] and s["power_w_max"] == 1380.0
    assert cs.summary(10, 11)["samples"] == 0


def test_recorded_traffic_matches_the_current_sources():
    """Every committed DRAM-traffic record was taken (or re-confirmed) on the
    kernel sources as they are now: bench.py reports it instead of null."""
    with open(bench.TRAFFIC_FILE) as f:
        recs = {k: v for k, v in json.load(f).items() if not k.startswith("_")}
    assert recs
    for name, rec in recs.items():
        cfg = W.by_name(name)
        kernel = "gemm" if cfg.hidden else "auto"
        got = bench.recorded_traffic(cfg, kernel)
        assert got == pytest.approx(rec["dram_bytes_per_token"] * cfg.T), name
        assert bench.recorded_traffic(cfg, "gather") is None   # another kernel than the captured one


def test_recorded_traffic_null_when_sources_differ(tmp_path, monkeypatch):
    with open(bench.TRAFFIC_FILE) as f:
        d = json.load(f)
    d["mid_prefill_fp8"]["kernel_sources_sha256"] = "0" * 64
    p = tmp_path / "traffic.json"
    p.write_text(json.dumps(d))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(p))
    assert bench.recorded_traffic(W.by_name("mid_prefill_fp8"), "auto") is None


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_fp8_d256", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["metric"] == bench.METRIC and d["higher_is_better"] is True
    assert d["config"]["workload"] == "tiny_fp8_d256"
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
