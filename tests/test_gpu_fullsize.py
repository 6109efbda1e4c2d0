"""Parity at the full workload sizes, in the launch configuration the benchmark
times (engram_compress_hash then engram_lookup_fused, no aux outputs,
out-of-place streams; a decode step as the one fused launch of engram_forward):
tables and streams are generated on the GPU, token ids on the host.  Every
compressed id and every row id is checked against the oracle; the streams are
checked on a seeded sample of tokens, for which the oracle gets exactly the
table rows and stream values the GPU read (copied back from the device: inputs,
not results).  A decode step's streams are checked on every slot; a
prefill's on 4096 sampled tokens (the first, the last and a seeded draw),
handed to the oracle in batches of 1024."""
import numpy as np
import pytest

import oracle
import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu

N_SAMPLE = 4096
ORACLE_BATCH = 1024


@pytest.fixture(scope="module")
def eg():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import hashed_gram_memory_gb300 as eg
    return eg


def run_full(eg, cfg, device_inputs):
    """The step as bench.py launches it: engram_compress_hash (with the compressed
    ids kept for the check) then engram_lookup_fused; a decode step's streams and
    history come from engram_forward's fused launch, its ids from
    engram_compress_hash."""
    import torch
    d = device_inputs
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    eids = torch.empty_like(d["ids"])
    hist_out = torch.empty_like(d["history"]) if d["history"] is not None else None
    primes = eg.engram_bucket_primes(1, 4, cfg.H, cfg.hash_vocab)[0] if cfg.hash_vocab else None
    rows = eg.engram_compress_hash(d["ids"], d["tid2eid"], cfg.n_eids, cfg.H, cfg.rows,
                                   history=d["history"], history_out=hist_out, eids_out=eids,
                                   status=st, positions=d["positions"], dead=d["dead"],
                                   primes=primes)
    out = torch.empty_like(d["streams"])
    if cfg.decode:
        hist_fused = torch.empty_like(d["history"])
        eg.engram_forward(d["ids"], d["tid2eid"], cfg.n_eids, cfg.H, d["tables"], d["streams"],
                          d["alpha"], cfg.eps, history=d["history"], history_out=hist_fused,
                          streams_out=out, status=st, positions=d["positions"], dead=d["dead"],
                          primes=primes)
        torch.cuda.synchronize()
        assert torch.equal(hist_fused, hist_out)
    else:
        eg.engram_lookup_fused(rows, cfg.H, d["tables"], d["streams"], d["alpha"], cfg.eps,
                               streams_out=out, status=st)
    code, flags = eg.engram_read_status(st)
    return eids, rows, hist_out, out, flags


def device_inputs(eg, cfg):
    import torch
    tabs, scales = W.tables_device(cfg, "cuda")
    dt = {W.FP8: eg.TABLE_FP8_E4M3FN, W.FP8_E8M0: eg.TABLE_FP8_E8M0, W.BF16: eg.TABLE_BF16,
          W.FP8_E8M0_ROWS: eg.TABLE_FP8_E8M0_ROWS}[cfg.dtype]
    hist = W.history(cfg)
    pos, dead = W.packed_layout(cfg) if cfg.packed else (None, None)
    return dict(ids=torch.from_numpy(W.token_ids(cfg)).cuda(),
                positions=None if pos is None else torch.from_numpy(pos).cuda(),
                dead=None if dead is None else torch.from_numpy(dead).cuda(),
                tid2eid=torch.from_numpy(W.tid2eid(cfg)).cuda(),
                history=None if hist is None else torch.from_numpy(hist).cuda(),
                streams=W.streams_device(cfg, "cuda"),
                alpha=torch.from_numpy(W.alpha(cfg)).cuda(),
                tables=eg.Tables(dt, tabs, scales))


def check_streams(cfg, d, out, r_all, toks):
    """The oracle's streams for tokens `toks`, from exactly the table rows and
    stream values the GPU read (copied back), against the GPU's."""
    import torch
    T = cfg.T
    rr = r_all[toks]                                      # [K, 3H]
    tabs, scs, remap = [], [], np.empty_like(rr)
    for n in range(3):
        cols = slice(n * cfg.H, (n + 1) * cfg.H)
        live = rr[:, cols] != oracle.DEAD
        uniq, inv = np.unique(np.where(live, rr[:, cols], 0), return_inverse=True)
        remap[:, cols] = np.where(live, inv.reshape(rr[:, cols].shape), oracle.DEAD)
        idx = torch.from_numpy(uniq.astype(np.int64)).cuda()
        t = d["tables"].tables[n].index_select(0, idx).cpu().numpy()
        tabs.append(t.view(np.uint16) if cfg.dtype == W.BF16 else t.view(np.uint8))
        scs.append(d["tables"].scales[n].index_select(0, idx).cpu().numpy()
                   if cfg.dtype in (W.FP8, W.FP8_E8M0) else None)
    tabs, scs = P.oracle_tables(cfg, tabs, scs)
    sel = torch.from_numpy(np.ascontiguousarray(toks)).cuda()
    x = d["streams"].view(T, 4, cfg.D)[sel].cpu().numpy().view(np.uint16)
    y_ref, f3 = oracle.lookup(remap, cfg.H, P.oracle_dtype(cfg), tabs, scs, x,
                              d["alpha"].cpu().numpy(), cfg.eps)
    assert f3 == 0
    y = out.view(T, 4, cfg.D)[sel].cpu().numpy().view(np.uint16)
    P.compare_streams(y, y_ref, x, what=f"{cfg.name} streams of tokens {toks[0]}..{toks[-1]}")


@pytest.mark.parametrize("name", ["mid_prefill_fp8", "decode_fp8", "full_prefill_fp8", "bf16_tables",
                                  "packed_mm_fp8", "full_prefill_fp8_e8m0",
                                  "full_prefill_fp8_e8m0_rows", "release_layout_fp8",
                                  "release_layout_fp8_rows"])
def test_full_size_sampled(eg, name):
    import torch
    cfg = W.by_name(name)
    free = torch.cuda.mem_get_info()[0]
    need = cfg.table_bytes() + 2 * cfg.T * 4 * cfg.D * 2 + (4 << 30)
    if free < need:
        pytest.skip(f"needs {need / 2**30:.1f} GiB of device memory, {free / 2**30:.1f} free")
    d = device_inputs(eg, cfg)
    eids, rows, hist_out, out, flags = run_full(eg, cfg, d)
    assert flags == 0

    # every index, bit-exact
    ids_h = d["ids"].cpu().numpy()
    if d["dead"] is not None:
        e_ref, f1 = oracle.compress_masked(ids_h, d["tid2eid"].cpu().numpy(), cfg.n_eids,
                                           d["dead"].cpu().numpy())
    else:
        e_ref, f1 = oracle.compress(ids_h, d["tid2eid"].cpu().numpy(), cfg.n_eids)
    hist_h = None if d["history"] is None else d["history"].cpu().numpy()
    pos_h = None if d["positions"] is None else d["positions"].cpu().numpy()
    if cfg.hash_vocab:
        r_ref, h_ref, f2 = oracle.hash_bucketed(e_ref, cfg.H, P.layer_primes(cfg), history=hist_h,
                                                positions=pos_h, want_history=True)
    else:
        r_ref, h_ref, f2 = oracle.hash_ids(e_ref, cfg.H, cfg.rows, history=hist_h,
                                           want_history=True, positions=pos_h)
    assert f1 == f2 == 0
    assert np.array_equal(eids.cpu().numpy(), e_ref)
    assert np.array_equal(rows.cpu().numpy(), r_ref)
    if hist_out is not None:
        assert np.array_equal(hist_out.cpu().numpy(), h_ref)

    # streams: every slot of a decode step, else a seeded sample of tokens
    # (first, last, random), in batches the oracle finishes quickly
    T = cfg.T
    if cfg.decode:
        toks = np.arange(T)
    else:
        g = np.random.default_rng(1000 + cfg.seed)
        toks = np.unique(np.concatenate([[0, T - 1], g.choice(np.arange(1, T - 1),
                                                             size=min(N_SAMPLE - 2, T - 2),
                                                             replace=False)]))
    assert len(toks) >= min(N_SAMPLE, T)
    r_all = r_ref.reshape(T, -1)
    for b0 in range(0, len(toks), ORACLE_BATCH):
        check_streams(cfg, d, out, r_all, toks[b0:b0 + ORACLE_BATCH])
    del d, out, rows, eids
    torch.cuda.empty_cache()
