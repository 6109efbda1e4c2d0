"""The NVTX ranges around the C-ABI calls, seen by a profiler: a minimal NVTX tool
(tests/c/nvtx_probe.c) is injected through NVTX_INJECTION64_PATH into a fresh
process, which makes calls that fail their host-side argument checks (no GPU
needed); every call must push a range named after it and pop it, with the
calls an entry point makes of its own nested inside."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_INCLUDE = "/usr/local/cuda/include"

CHILD = r"""
import ctypes as C, sys
sys.path.insert(0, sys.argv[1])
import hashed_gram_memory_gb300 as eg
L = eg.lib
L.engram_lookup_fused(None, 4, 2, None, None, None, None, 1e-6, None, None, None, None)
L.engram_compress(None, 4, None, 8, 7, None, None, None)
L.engram_forward(None, 1, 4, None, 8, 7, None, None, 2, None, None, None, None, None, 1e-6,
                 None, 0, None, None)
probe = C.CDLL(sys.argv[2])
probe.nvtx_probe_log.restype = C.c_char_p
print(probe.nvtx_probe_log().decode())
"""


def test_every_call_is_one_named_range(tmp_path):
    if not os.path.exists(os.path.join(CUDA_INCLUDE, "nvtx3", "nvToolsExt.h")):
        pytest.skip("no NVTX3 headers")
    import hashed_gram_memory_gb300  # noqa: F401  (the library is built)
    probe = tmp_path / "libnvtx_probe.so"
    subprocess.run(["gcc", "-std=c99", "-O1", "-shared", "-fPIC", "-fvisibility=hidden",
                    "-I", CUDA_INCLUDE, os.path.join(ROOT, "tests", "c", "nvtx_probe.c"),
                    "-o", str(probe)], check=True)
    env = dict(os.environ, NVTX_INJECTION64_PATH=str(probe))
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT, str(probe)], capture_output=True,
                       text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr
    log = r.stdout.strip().splitlines()[-1]
    # engram_compress is engram_compress_masked without a mask: its range nests
    assert log == ("+engram_lookup_fused;-;+engram_compress;+engram_compress_masked;-;-;"
                   "+engram_forward;-;"), log
