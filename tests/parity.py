"""Shared pieces of the GPU parity tests: run a workload through the C ABI and
through the CPU oracle on the same seeded inputs, and compare.

Tolerances (the streams are bf16 outputs of fp32 arithmetic):
* compressed ids, row ids, history: bit-exact;
* streams: |y - y_ref| <= 2e-2 + 1e-2 |y_ref| elementwise (the stated max-abs
  2e-2 / rel 1e-2 bar, read as an allclose), and in addition within one bf16
  ulp of the oracle's once-rounded value plus the fp32 rounding of the operands
  (2^-23 |x| + 2^-16 |y - x|), and at most 0.1% of elements not bit-identical
  (the fp32 path rounds twice: fp32, then bf16);
* m (fp32, sum of 3H products): within 1e-5 relative + 1e-6 of max |m|;
* g (fp32 sigmoid of a 4096-term fp32 reduction): within 1e-5 absolute.
"""
from __future__ import annotations

import dataclasses

import numpy as np

import oracle
import workloads as W

STREAM_ATOL, STREAM_RTOL = 2e-2, 1e-2
MAX_MISMATCH_FRAC = 1e-3


@dataclasses.dataclass
class HostInputs:
    cfg: W.EngramConfig
    ids: np.ndarray
    tid2eid: np.ndarray
    history: np.ndarray | None
    tables: list
    scales: list
    streams: np.ndarray
    alpha: np.ndarray
    positions: np.ndarray | None = None   # packed samples: index within the sample
    dead: np.ndarray | None = None        # packed samples: image-span positions


def host_inputs(cfg: W.EngramConfig, rank: int = 0) -> HostInputs:
    tabs, scales = W.tables_host(cfg)
    pos, dead = W.packed_layout(cfg, rank) if cfg.packed else (None, None)
    return HostInputs(cfg, W.token_ids(cfg, rank), W.tid2eid(cfg), W.history(cfg, rank), tabs,
                      scales, W.streams_host(cfg, rank), W.alpha(cfg), pos, dead)


def layer_primes(cfg: W.EngramConfig):
    """The bucket sizes [3][H] of one layer's table (the oracle's draw)."""
    return oracle.bucket_primes(1, 4, cfg.H, cfg.hash_vocab)[0]


def oracle_dtype(cfg: W.EngramConfig) -> int:
    """The oracle's table type: rows carrying their exponents are read, like the
    separate layout, as bytes plus e8m0 blocks (oracle_tables splits them)."""
    return {W.FP8: oracle.FP8, W.FP8_E8M0: oracle.FP8_E8M0, W.FP8_E8M0_ROWS: oracle.FP8_E8M0,
            W.BF16: oracle.BF16}[cfg.dtype]


def oracle_tables(cfg: W.EngramConfig, tables, scales):
    """The tables and scales as the oracle takes them: a table whose rows carry
    their exponents is split into its bytes [rows, D] and exponents [rows, D/32]
    (slices of each row, no arithmetic)."""
    if cfg.dtype != W.FP8_E8M0_ROWS:
        return tables, scales
    D = cfg.D
    return ([np.ascontiguousarray(t[:, :D]) for t in tables],
            [np.ascontiguousarray(t[:, D:D + D // 32]) for t in tables])


def oracle_path(inp: HostInputs):
    cfg = inp.cfg
    if inp.dead is not None:
        eids, f1 = oracle.compress_masked(inp.ids, inp.tid2eid, cfg.n_eids, inp.dead)
    else:
        eids, f1 = oracle.compress(inp.ids, inp.tid2eid, cfg.n_eids)
    if cfg.hash_vocab:
        rows, hist, f2 = oracle.hash_bucketed(eids, cfg.H, layer_primes(cfg), history=inp.history,
                                              positions=inp.positions, want_history=True)
    else:
        rows, hist, f2 = oracle.hash_ids(eids, cfg.H, cfg.rows, history=inp.history,
                                         want_history=True, positions=inp.positions)
    tabs, scs = oracle_tables(cfg, inp.tables, inp.scales)
    y, g, m, f3 = oracle.lookup(rows.reshape(cfg.T, -1), cfg.H, oracle_dtype(cfg), tabs, scs,
                                inp.streams.reshape(cfg.T, 4, cfg.D), inp.alpha, cfg.eps,
                                aux=True)
    return dict(eids=eids, rows=rows, history=hist, streams=y.reshape(inp.streams.shape), gate=g,
                mem=m, flags=f1 | f2 | f3)


def to_device(inp: HostInputs, device="cuda"):
    import torch
    import hashed_gram_memory_gb300 as eg
    cfg = inp.cfg
    dev = dict(
        ids=torch.from_numpy(inp.ids).to(device),
        tid2eid=torch.from_numpy(inp.tid2eid).to(device),
        history=None if inp.history is None else torch.from_numpy(inp.history).to(device),
        streams=torch.from_numpy(inp.streams.view(np.int16)).to(device),
        alpha=torch.from_numpy(inp.alpha).to(device),
        positions=None if inp.positions is None else torch.from_numpy(inp.positions).to(device),
        dead=None if inp.dead is None else torch.from_numpy(inp.dead).to(device),
    )
    if cfg.dtype in (W.FP8, W.FP8_E8M0):
        tabs = [torch.from_numpy(t).to(device) for t in inp.tables]
        scs = [torch.from_numpy(s).to(device) for s in inp.scales]
        dt = eg.TABLE_FP8_E4M3FN if cfg.dtype == W.FP8 else eg.TABLE_FP8_E8M0
        dev["tables"] = eg.Tables(dt, tabs, scs)
    elif cfg.dtype == W.FP8_E8M0_ROWS:
        tabs = [torch.from_numpy(t).to(device) for t in inp.tables]
        dev["tables"] = eg.Tables(eg.TABLE_FP8_E8M0_ROWS, tabs, None)
    else:
        tabs = [torch.from_numpy(t.view(np.int16)).to(device) for t in inp.tables]
        dev["tables"] = eg.Tables(eg.TABLE_BF16, tabs, None)
    return dev


def gpu_path(cfg: W.EngramConfig, dev: dict, aux: bool = True, in_place: bool = False):
    """compress -> hash -> fused lookup through the C ABI; returns host arrays."""
    import torch
    import hashed_gram_memory_gb300 as eg
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    eids = eg.engram_compress(dev["ids"], dev["tid2eid"], cfg.n_eids, status=status,
                              dead=dev.get("dead"))
    hist_out = None
    if dev["history"] is not None:
        hist_out = torch.empty_like(dev["history"])
    primes = eg.engram_bucket_primes(1, 4, cfg.H, cfg.hash_vocab)[0] if cfg.hash_vocab else None
    rows = eg.engram_hash(eids, cfg.H, cfg.rows, history=dev["history"], history_out=hist_out,
                          status=status, positions=dev.get("positions"), primes=primes)
    gate = torch.full((cfg.T,), float("nan"), device="cuda") if aux else None
    mem = torch.full((cfg.T, cfg.D), float("nan"), device="cuda") if aux else None
    x = dev["streams"]
    out = x.clone() if in_place else torch.empty_like(x)
    src = out if in_place else x
    eg.engram_lookup_fused(rows, cfg.H, dev["tables"], src, dev["alpha"], cfg.eps, streams_out=out,
                           gate_out=gate, mem_out=mem, status=status)
    code, flags = eg.engram_read_status(status)
    res = dict(eids=eids.cpu().numpy(), rows=rows.cpu().numpy(), x=x.cpu().numpy().view(np.uint16),
               history=None if hist_out is None else hist_out.cpu().numpy(),
               streams=out.cpu().numpy().view(np.uint16), flags=flags, code=code)
    if aux:
        res["gate"] = gate.cpu().numpy()
        res["mem"] = mem.cpu().numpy()
    return res


def bf16_ulp(y: np.ndarray) -> np.ndarray:
    a = np.abs(y.astype(np.float64))
    e = np.frexp(np.maximum(a, 2.0 ** -126))[1]
    return np.ldexp(1.0, e - 8)


def compare_streams(y_gpu_bits: np.ndarray, y_ref_bits: np.ndarray, x_bits: np.ndarray,
                    what: str = "streams"):
    """The stated allclose bar, then a tight one: one bf16 ulp of the oracle's
    value plus the fp32 path's own error, which scales with its operands (x and
    the update g*alpha*m ~ y - x), not with y: near cancellation the ulp of y is
    far below fp32's rounding of x."""
    yg = oracle.bf16_bits_to_float(y_gpu_bits).astype(np.float64)
    yr = oracle.bf16_bits_to_float(y_ref_bits).astype(np.float64)
    x = oracle.bf16_bits_to_float(x_bits).astype(np.float64)
    assert np.isfinite(yg).all(), f"{what}: non-finite output"
    err = np.abs(yg - yr)
    bound = STREAM_ATOL + STREAM_RTOL * np.abs(yr)
    worst = float(np.max(err / bound)) if err.size else 0.0
    assert np.all(err <= bound), f"{what}: allclose bar exceeded, worst err/bound {worst:.3g}"
    tight = bf16_ulp(yr) + 2.0 ** -23 * np.abs(x) + 2.0 ** -16 * np.abs(yr - x)
    worst = float(np.max(err / tight)) if err.size else 0.0
    assert np.all(err <= tight), f"{what}: tight bound exceeded by {worst:.3g}x"
    mism = float(np.mean(y_gpu_bits != y_ref_bits)) if err.size else 0.0
    assert mism <= MAX_MISMATCH_FRAC, f"{what}: {mism:.2e} of elements not bit-identical"
    return dict(max_abs=float(err.max()) if err.size else 0.0, mismatch_frac=mism)


def compare_mem(m_gpu, m_ref):
    scale = float(np.max(np.abs(m_ref))) if m_ref.size else 0.0
    np.testing.assert_allclose(m_gpu, m_ref, rtol=1e-5, atol=1e-6 * scale + 1e-30)


def compare_gate(g_gpu, g_ref):
    np.testing.assert_allclose(g_gpu, g_ref, rtol=0, atol=1e-5)


def compare_all(res: dict, ref: dict, aux: bool = True):
    assert res["flags"] == ref["flags"] == 0, (res["flags"], ref["flags"])
    assert np.array_equal(res["eids"], ref["eids"])
    assert np.array_equal(res["rows"], ref["rows"])
    if ref["history"] is not None and res["history"] is not None:
        assert np.array_equal(res["history"], ref["history"])
    stats = compare_streams(res["streams"], ref["streams"], res["x"])
    if aux:
        compare_mem(res["mem"], ref["mem"])
        compare_gate(res["gate"], ref["gate"])
    return stats
