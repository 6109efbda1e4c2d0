"""Write tests/golden/tiny_fp8_d256_oracle.json: digests of the oracle's results on
the tiny FP8 workload (batch 1, seq 256, D 256, H 2, 3 x 4096-row tables).

Calls only the CPU oracle and the seeded input generators.  The fixture lets a
fresh machine (x86-64 or AArch64) confirm that its oracle build reproduces the
same bytes.  Run: python tests/golden/make_golden.py
"""
import hashlib
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import workloads as W  # noqa: E402


def tiny_results():
    cfg = W.by_name("tiny_fp8_d256")
    ids = W.token_ids(cfg)
    eids, f1 = oracle.compress(ids, W.tid2eid(cfg), cfg.n_eids)
    rows, f2 = oracle.hash_ids(eids, cfg.H, cfg.rows)
    tabs, scales = W.tables_host(cfg)
    x = W.streams_host(cfg)
    y, g, m, f3 = oracle.lookup(rows.reshape(cfg.T, -1), cfg.H, oracle.FP8, tabs, scales,
                                x.reshape(cfg.T, 4, cfg.D), W.alpha(cfg), cfg.eps, aux=True)
    return dict(eids=eids, rows=rows, streams_out=y, gate=g, flags=[f1, f2, f3],
                inputs=dict(ids=ids, tables=np.concatenate([t.ravel() for t in tabs]),
                            scales=np.concatenate(scales), streams=x))


def digest(a) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


def summary():
    r = tiny_results()
    return {
        "workload": W.by_name("tiny_fp8_d256").name,
        "flags": r["flags"],
        "sha256": {k: digest(r[k]) for k in ("eids", "rows", "streams_out")},
        "inputs_sha256": {k: digest(v) for k, v in r["inputs"].items()},
        "first_rows": r["rows"][0, :2].tolist(),
        "gate_first4": [float(v) for v in r["gate"][:4]],
        "gate_mean": float(np.mean(r["gate"])),
    }


if __name__ == "__main__":
    out = os.path.join(HERE, "tiny_fp8_d256_oracle.json")
    with open(out, "w") as f:
        json.dump(summary(), f, indent=1)
    print(out)
