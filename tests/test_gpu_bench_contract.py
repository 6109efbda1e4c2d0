"""bench.py's native arm on the GPU, as a subprocess on a small workload: exactly
one JSON line with every key of the output contract, a roofline that stays
physical, clocks sampled during the timed region, the end-to-end figure through
host buffers with its byte counts, and the oracle's CPU baseline."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def line():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload",
                        "mid_prefill_fp8", "--rows", "20000", "--steps", "5", "--warmup", "3",
                        "--e2e-steps", "2", "--cpu-sample-tokens", "512", "--min-timed-s", "0.3"],
                       capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def test_contract_keys(line):
    d = line
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "roofline",
              "clocks", "e2e", "cpu_baseline", "gpu_launches"):
        assert k in d, k
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True and d["n_gpus"] == 1
    assert d["steps"] == 5 and d["warmup"] == 3 and d["scaling"] == "weak"
    assert d["config"]["workload"] == "mid_prefill_fp8" and "l2" in d["config"]
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert abs(d["value"] - d["config"]["tokens_per_step"] / (d["ms_per_step"] * 1e-3)) \
        <= 1e-6 * d["value"]


def test_roofline_is_physical(line):
    r = line["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in r, k
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert 0.05 < r["frac"] < 1.4                      # of a measured copy bandwidth
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    # the lookup's duration fits inside a step
    assert r["kernel_ms"] <= line["ms_per_step"] * 1.01


def test_clocks_e2e_and_baseline(line):
    c = line["clocks"]
    assert c["samples"] >= 1 and c["sm_mhz"] > 0 and c["sm_max_mhz"] > 0
    assert isinstance(c["reasons"], list)
    e = line["e2e"]
    cfg = line["config"]
    T, D = cfg["tokens_per_step"], cfg["D"]
    assert e["unit"] == "tokens/s" and e["value"] > 0 and e["matches_device_step"] is True
    assert e["d2h_bytes_per_step"] == T * 4 * D * 2      # the streams out
    assert e["h2d_bytes_per_step"] >= T * 4 * D * 2      # the streams (and ids) in
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0 and cb["sample"]
    assert line["gpu_launches"] >= line["steps"]
