"""The oracle reproduces its recorded results on the tiny FP8 workload on this
machine (the fixture was written by tests/golden/make_golden.py, which calls only
the oracle and the seeded input generators).  A mismatch in the input digests
means the generators drifted; in the output digests, that the oracle build does
(for instance a compiler that fuses multiply-adds)."""
import json
import os

import pytest

from tests.golden import make_golden

FIXTURE = os.path.join(os.path.dirname(__file__), "golden", "tiny_fp8_d256_oracle.json")


@pytest.fixture(scope="module")
def recorded():
    with open(FIXTURE) as f:
        return json.load(f)


def test_inputs_reproduce(recorded):
    now = make_golden.summary()
    assert now["inputs_sha256"] == recorded["inputs_sha256"]


def test_oracle_outputs_reproduce(recorded):
    now = make_golden.summary()
    assert now["flags"] == recorded["flags"] == [0, 0, 0]
    assert now["sha256"] == recorded["sha256"]
    assert now["first_rows"] == recorded["first_rows"]
    assert now["gate_first4"] == recorded["gate_first4"]
