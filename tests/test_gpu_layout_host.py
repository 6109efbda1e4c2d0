"""The whole-path calls with a batch layout (packed samples: positions and a dead
mask; the released prime-bucket table) and the host-buffer connection.

* engram_forward with a layout equals compress_masked -> hash_packed /
  hash_bucketed -> lookup bit for bit, and the oracle within the stated
  tolerance; for one new token a slot the fused decode launch takes the layout
  too (positions cap the lookback, dead slots pass through, bucket moduli and
  offsets) and equals the three calls.
* engram_forward_host with host positions and dead mask equals engram_forward
  with the same layout on device buffers, for ragged chunk sizes, and for
  decode steps (each chunk of slots one fused launch), history included.
* engram_connection_host (host ids and streams, chunked copies overlapped with
  the connection) equals compress -> hash -> engram_connection on device
  buffers bit for bit: plain and bucketed tables, packed batches with dead
  tokens, ragged chunks, pinned and pageable memory, two calls back to back on
  one workspace.
"""
import numpy as np
import pytest

import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def eg():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import hashed_gram_memory_gb300 as eg
    return eg


def _primes(eg, cfg):
    return eg.engram_bucket_primes(1, 4, cfg.H, cfg.hash_vocab)[0] if cfg.hash_vocab else None


LAYOUT_CASES = {
    "packed_dead": W.by_name("packed_mm_fp8").scaled(B=2, S=300, rows=(6007, 6011, 6029),
                                                     mean_sample_len=40, image_span=8,
                                                     image_frac=0.3),
    "bucketed": W.by_name("release_layout_fp8").scaled(B=2, S=333, rows=(32_000,) * 3,
                                                       hash_vocab=1000),
    "bucketed_packed_dead": W.by_name("release_layout_fp8").scaled(
        B=2, S=211, D=128, rows=(32_000,) * 3, hash_vocab=1000, packed=True,
        mean_sample_len=50, image_span=8, image_frac=0.25),
    "bucketed_d4096_h4": W.by_name("full_prefill_fp8").scaled(B=1, S=150, H=4,
                                                              rows=(16_000,) * 3,
                                                              hash_vocab=1000),
}


def _forward(eg, cfg, dev, **kw):
    import torch
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = eg.engram_forward(dev["ids"], dev["tid2eid"], cfg.n_eids, cfg.H, dev["tables"],
                          dev["streams"], dev["alpha"], cfg.eps, history=dev["history"],
                          status=st, positions=dev.get("positions"), dead=dev.get("dead"),
                          primes=_primes(eg, cfg), **kw)
    return y, eg.engram_read_status(st)[1]


@pytest.mark.parametrize("name", list(LAYOUT_CASES))
def test_forward_with_layout_equals_separate_calls_and_oracle(eg, name):
    cfg = LAYOUT_CASES[name]
    inp = P.host_inputs(cfg)
    dev = P.to_device(inp)
    sep = P.gpu_path(cfg, dev, aux=False)
    y, flags = _forward(eg, cfg, dev)
    assert flags == 0 and sep["flags"] == 0
    assert np.array_equal(y.cpu().numpy().view(np.uint16), sep["streams"])
    ref = P.oracle_path(inp)
    assert np.array_equal(sep["rows"].reshape(ref["rows"].shape), ref["rows"])
    P.compare_streams(sep["streams"], ref["streams"], inp.streams)
    if inp.dead is not None:   # dead tokens copied through
        d = inp.dead.reshape(-1).astype(bool)
        assert d.any()
        assert np.array_equal(sep["streams"].reshape(cfg.T, -1)[d],
                              inp.streams.reshape(cfg.T, -1)[d])


@pytest.mark.parametrize("primes,with_history", [(False, True), (True, True), (True, False)])
def test_fused_decode_with_layout_equals_three_calls(eg, primes, with_history):
    """One new token a slot with positions (0..5: a slot at position p reads back
    at most p ids), a dead mask (about one slot in eight) and, optionally, the
    prime-bucket layout: the fused launch gives the streams and the history of
    compress_masked -> hash -> lookup bit for bit."""
    import torch
    B = 301
    base = W.by_name("decode_fp8").scaled(B=B, H=4, rows=(32_000,) * 3)
    cfg = base.scaled(hash_vocab=1000) if primes else base
    inp = P.host_inputs(cfg)
    dev = P.to_device(inp)
    g = np.random.default_rng(77)
    pos = torch.from_numpy(g.integers(0, 6, size=(B, 1)).astype(np.int32)).cuda()
    dead = torch.from_numpy((g.random((B, 1)) < 0.125).astype(np.uint8)).cuda()
    assert dead.any()
    hist = dev["history"] if with_history else None
    pr = _primes(eg, cfg)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    eids = eg.engram_compress(dev["ids"], dev["tid2eid"], cfg.n_eids, status=st, dead=dead)
    h_sep = torch.empty_like(hist) if hist is not None else None
    rows = eg.engram_hash(eids, cfg.H, cfg.rows, history=hist, history_out=h_sep, status=st,
                          positions=pos, primes=pr)
    y_sep = eg.engram_lookup_fused(rows, cfg.H, dev["tables"], dev["streams"], dev["alpha"],
                                   cfg.eps, status=st)
    h_out = torch.empty_like(hist) if hist is not None else None
    y = eg.engram_forward(dev["ids"], dev["tid2eid"], cfg.n_eids, cfg.H, dev["tables"],
                          dev["streams"], dev["alpha"], cfg.eps, history=hist, history_out=h_out,
                          status=st, positions=pos, dead=dead, primes=pr)
    assert eg.engram_read_status(st)[1] == 0
    assert torch.equal(y, y_sep)
    if hist is not None:
        assert torch.equal(h_out, h_sep)
    d = dead.reshape(-1).bool()
    assert torch.equal(y[d], dev["streams"][d])   # dead slots pass through


@pytest.mark.parametrize("name,chunk", [("packed_dead", 97), ("bucketed", 0),
                                        ("bucketed_packed_dead", 64)])
def test_forward_host_with_layout_equals_forward(eg, name, chunk):
    import torch
    cfg = LAYOUT_CASES[name]
    inp = P.host_inputs(cfg)
    dev = P.to_device(inp)
    y_dev, flags = _forward(eg, cfg, dev)
    assert flags == 0
    ids_h = torch.from_numpy(inp.ids).pin_memory()
    x_h = torch.from_numpy(inp.streams.view(np.int16)).reshape(cfg.T, 4, cfg.D).pin_memory()
    y_h = torch.full_like(x_h, 0x7777).pin_memory()
    pos_h = None if inp.positions is None else torch.from_numpy(inp.positions).pin_memory()
    dead_h = None if inp.dead is None else torch.from_numpy(inp.dead).pin_memory()
    ws = torch.empty(eg.engram_forward_host_workspace_bytes(cfg.B, cfg.S, cfg.H, cfg.D, chunk),
                     dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        eg.engram_forward_host(ids_h, dev["tid2eid"], cfg.n_eids, cfg.H, dev["tables"], x_h, y_h,
                               dev["alpha"], ws, cfg.eps, history=dev["history"],
                               chunk_tokens=chunk, status=st, positions=pos_h, dead=dead_h,
                               primes=_primes(eg, cfg))
    stream.synchronize()
    assert eg.engram_read_status(st)[1] == 0
    assert np.array_equal(y_h.numpy().view(np.uint16).reshape(cfg.T, -1),
                          y_dev.cpu().numpy().view(np.uint16).reshape(cfg.T, -1))


CONN = W.by_name("release_connection_e8m0")
CONN_CASES = {
    "e8m0_h2_d128": CONN.scaled(B=2, S=129, H=2, D=128, rows=(2003, 2011, 2017), hash_vocab=0,
                                hidden=512),
    "bucketed_h8_d256": CONN.scaled(B=2, S=300, H=8, D=256, rows=(32_000,) * 3,
                                    hash_vocab=1000, hidden=1024),
    "packed_dead_bf16": CONN.scaled(B=2, S=150, H=2, D=64, rows=(1009, 1013, 1019),
                                    hash_vocab=0, dtype=W.BF16, hidden=256, packed=True,
                                    mean_sample_len=64, image_span=16, image_frac=0.25),
}


def _connection_device(eg, cfg, dev, wkv):
    """compress -> hash -> engram_connection on device buffers."""
    import torch
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    eids = eg.engram_compress(dev["ids"], dev["tid2eid"], cfg.n_eids, status=st,
                              dead=dev.get("dead"))
    rows = eg.engram_hash(eids, cfg.H, cfg.rows, history=dev["history"], status=st,
                          positions=dev.get("positions"), primes=_primes(eg, cfg))
    x = dev["streams"].view(cfg.T, 4, cfg.hidden)
    y = eg.engram_connection(rows, cfg.H, dev["tables"], wkv, x, dev["alpha"], cfg.eps,
                             status=st)
    assert eg.engram_read_status(st)[1] == 0
    return y.cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("name,chunk,pinned", [("e8m0_h2_d128", 100, True),
                                               ("e8m0_h2_d128", 0, False),
                                               ("bucketed_h8_d256", 128, True),
                                               ("packed_dead_bf16", 77, True)])
def test_connection_host_equals_device_connection(eg, name, chunk, pinned):
    import torch
    cfg = CONN_CASES[name]
    ws = torch.empty(eg.engram_connection_host_workspace_bytes(cfg.B, cfg.S, cfg.H, cfg.D,
                                                               cfg.hidden, chunk),
                     dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    calls = []
    # two calls back to back with different inputs (replicas 0 and 1) on one workspace
    for rank in (0, 1):
        inp = P.host_inputs(cfg, rank=rank)
        dev = P.to_device(inp)
        wkv = torch.from_numpy(W.wkv_host(cfg).view(np.int16)).cuda()
        ref = _connection_device(eg, cfg, dev, wkv)
        ids_h = torch.from_numpy(inp.ids)
        x_h = torch.from_numpy(inp.streams.view(np.int16)).reshape(cfg.T, 4, cfg.hidden)
        y_h = torch.full_like(x_h, 0x7777)
        pos_h = None if inp.positions is None else torch.from_numpy(inp.positions)
        dead_h = None if inp.dead is None else torch.from_numpy(inp.dead)
        if pinned:
            ids_h, x_h, y_h = ids_h.pin_memory(), x_h.pin_memory(), y_h.pin_memory()
            pos_h = None if pos_h is None else pos_h.pin_memory()
            dead_h = None if dead_h is None else dead_h.pin_memory()
        calls.append((ids_h, x_h, y_h, pos_h, dead_h, dev, wkv, ref))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    with torch.cuda.stream(stream):
        for ids_h, x_h, y_h, pos_h, dead_h, dev, wkv, _ in calls:
            eg.engram_connection_host(ids_h, dev["tid2eid"], cfg.n_eids, cfg.H, dev["tables"],
                                      wkv, x_h, y_h, dev["alpha"], ws, cfg.eps,
                                      history=dev["history"], chunk_tokens=chunk, status=st,
                                      positions=pos_h, dead=dead_h, primes=_primes(eg, cfg))
    stream.synchronize()
    assert eg.engram_read_status(st)[1] == 0
    for ids_h, x_h, y_h, pos_h, dead_h, dev, wkv, ref in calls:
        assert np.array_equal(y_h.numpy().view(np.uint16).reshape(ref.shape), ref)


@pytest.mark.parametrize("primes,chunk", [(False, 0), (True, 100)])
def test_forward_host_decode_with_layout_equals_forward(eg, primes, chunk):
    """A decode step through engram_forward_host (each chunk of slots one fused
    launch) with host positions and dead mask, and optionally the bucket layout,
    equals engram_forward on device buffers: streams and history bit for bit."""
    import torch
    B = 301
    base = W.by_name("decode_fp8").scaled(B=B, H=4, rows=(32_000,) * 3)
    cfg = base.scaled(hash_vocab=1000) if primes else base
    inp = P.host_inputs(cfg)
    dev = P.to_device(inp)
    g = np.random.default_rng(78)
    pos = g.integers(0, 6, size=(B, 1)).astype(np.int32)
    dead = (g.random((B, 1)) < 0.125).astype(np.uint8)
    pr = _primes(eg, cfg)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    h_dev = torch.empty_like(dev["history"])
    y_dev = eg.engram_forward(dev["ids"], dev["tid2eid"], cfg.n_eids, cfg.H, dev["tables"],
                              dev["streams"], dev["alpha"], cfg.eps, history=dev["history"],
                              history_out=h_dev, status=st, positions=torch.from_numpy(pos).cuda(),
                              dead=torch.from_numpy(dead).cuda(), primes=pr)
    ids_h = torch.from_numpy(inp.ids).pin_memory()
    x_h = torch.from_numpy(inp.streams.view(np.int16)).reshape(cfg.T, 4, cfg.D).pin_memory()
    y_h = torch.full_like(x_h, 0x7777).pin_memory()
    h_host = torch.empty_like(dev["history"])
    ws = torch.empty(eg.engram_forward_host_workspace_bytes(cfg.B, cfg.S, cfg.H, cfg.D, chunk),
                     dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        eg.engram_forward_host(ids_h, dev["tid2eid"], cfg.n_eids, cfg.H, dev["tables"], x_h, y_h,
                               dev["alpha"], ws, cfg.eps, history=dev["history"],
                               history_out=h_host, chunk_tokens=chunk, status=st,
                               positions=torch.from_numpy(pos).pin_memory(),
                               dead=torch.from_numpy(dead).pin_memory(), primes=pr)
    stream.synchronize()
    assert eg.engram_read_status(st)[1] == 0
    assert np.array_equal(y_h.numpy().view(np.uint16).reshape(cfg.T, -1),
                          y_dev.cpu().numpy().view(np.uint16).reshape(cfg.T, -1))
    assert torch.equal(h_host, h_dev)
