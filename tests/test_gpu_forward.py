"""The one-call entry points: engram_forward (device buffers) must equal the three
separate calls bit for bit (for one new token a slot it runs them as one fused
launch); engram_forward_host (host ids and streams, chunked
copy/compute pipeline) must equal engram_forward bit for bit, for ragged chunk
sizes, pinned and pageable host memory, and back-to-back calls that reuse the
same workspace with different inputs."""
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


CASES = {
    "prefill_h8": W.by_name("full_prefill_fp8").scaled(B=2, S=517, rows=(6007, 6011, 6029)),
    "decode_history": W.by_name("decode_fp8").scaled(B=300, rows=(7001, 7013, 7019)),
    "bf16": W.by_name("bf16_tables").scaled(B=3, S=133, rows=(3001, 3011, 3019)),
    "tiny_d256": W.by_name("tiny_fp8_d256"),
}


@pytest.mark.parametrize("name", list(CASES))
def test_forward_equals_separate_calls_and_oracle(eg, name):
    import torch
    cfg = CASES[name]
    inp = P.host_inputs(cfg)
    dev = P.to_device(inp)
    sep = P.gpu_path(cfg, dev, aux=False)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    hist_out = torch.empty_like(dev["history"]) if dev["history"] is not None else None
    y = eg.engram_forward(dev["ids"], dev["tid2eid"], cfg.n_eids, cfg.H, dev["tables"],
                          dev["streams"], dev["alpha"], cfg.eps, history=dev["history"],
                          history_out=hist_out, status=st)
    code, flags = eg.engram_read_status(st)
    assert flags == 0
    assert np.array_equal(y.cpu().numpy().view(np.uint16), sep["streams"])
    if hist_out is not None:
        assert np.array_equal(hist_out.cpu().numpy(), sep["history"])
    ref = P.oracle_path(inp)
    P.compare_streams(sep["streams"], ref["streams"], inp.streams)


@pytest.mark.parametrize("name,chunk,pinned", [("prefill_h8", 77, True), ("prefill_h8", 0, False),
                                               ("decode_history", 64, True), ("bf16", 128, True),
                                               ("tiny_d256", 1, True)])
def test_forward_host_equals_forward(eg, name, chunk, pinned):
    import torch
    cfg = CASES[name]
    outs_dev, outs_host = [], []
    ws = torch.empty(eg.engram_forward_host_workspace_bytes(cfg.B, cfg.S, cfg.H, cfg.D, chunk),
                     dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    hosts = []
    # two back-to-back calls with different inputs (replica 0 and 1) on one workspace
    for rank in (0, 1):
        inp = P.host_inputs(cfg, rank=rank)
        dev = P.to_device(inp)
        outs_dev.append(eg.engram_forward(dev["ids"], dev["tid2eid"], cfg.n_eids, cfg.H,
                                          dev["tables"], dev["streams"], dev["alpha"], cfg.eps,
                                          history=dev["history"]).cpu().numpy().view(np.uint16))
        ids_h = torch.from_numpy(inp.ids)
        x_h = torch.from_numpy(inp.streams.view(np.int16)).reshape(cfg.T, 4, cfg.D)
        if pinned:
            ids_h, x_h = ids_h.pin_memory(), x_h.pin_memory()
        y_h = torch.full_like(x_h, 0x7777)
        if pinned:
            y_h = y_h.pin_memory()
        hosts.append((ids_h, x_h, y_h, dev))
    with torch.cuda.stream(stream):
        for ids_h, x_h, y_h, dev in hosts:
            eg.engram_forward_host(ids_h, dev["tid2eid"], cfg.n_eids, cfg.H, dev["tables"], x_h,
                                   y_h, dev["alpha"], ws, cfg.eps, history=dev["history"],
                                   chunk_tokens=chunk)
    stream.synchronize()
    for (ids_h, x_h, y_h, dev), ref in zip(hosts, outs_dev):
        assert np.array_equal(y_h.numpy().view(np.uint16).reshape(ref.shape), ref)


def _decode_case(eg, B=257, H=4, D=4096, rows=(7001, 7013, 7019), with_history=True, seed=5,
                 dtype=W.FP8):
    import torch
    cfg = W.by_name("decode_fp8").scaled(B=B, H=H, D=D, rows=rows, dtype=dtype)
    inp = P.host_inputs(cfg)
    dev = P.to_device(inp)
    g = np.random.default_rng(seed)
    hist = None
    if with_history:
        h = inp.history.copy()
        h[g.choice(B, size=B // 8, replace=False), g.integers(0, 3, size=B // 8)] = -1  # dead
        hist = torch.from_numpy(h).cuda()
    return cfg, inp, dev, hist


@pytest.mark.parametrize("B,dtype,with_history,in_place_history", [
    (257, W.FP8, True, False), (257, W.FP8, False, False), (257, W.FP8, True, True),
    (257, W.BF16, True, False), (257, W.FP8_E8M0, True, False),
    (257, W.FP8_E8M0_ROWS, True, False),
    (1500, W.FP8, True, False), (5000, W.FP8_E8M0, True, False)])
def test_fused_decode_equals_three_calls(eg, B, dtype, with_history, in_place_history):
    """One new token a slot: the fused decode launch gives the streams and the
    updated history of compress -> hash -> lookup bit for bit, with dead ids in
    the history (they block the lookback) or no history at all (pad), for every
    table type, and for small and large batches."""
    import torch
    cfg, inp, dev, hist = _decode_case(eg, B=B, with_history=with_history, dtype=dtype)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    # the three calls
    eids = eg.engram_compress(dev["ids"], dev["tid2eid"], cfg.n_eids, status=st)
    h_sep = torch.empty_like(hist) if hist is not None else None
    rows = eg.engram_hash(eids, cfg.H, cfg.rows, history=hist, history_out=h_sep, status=st)
    y_sep = eg.engram_lookup_fused(rows, cfg.H, dev["tables"], dev["streams"], dev["alpha"],
                                   cfg.eps, status=st)
    # the fused launch
    if hist is not None and in_place_history:
        h_in = hist.clone()
        h_out = h_in
    else:
        h_in, h_out = hist, (torch.empty_like(hist) if hist is not None else None)
    y = eg.engram_forward(dev["ids"], dev["tid2eid"], cfg.n_eids, cfg.H, dev["tables"],
                          dev["streams"], dev["alpha"], cfg.eps, history=h_in, history_out=h_out,
                          status=st)
    assert eg.engram_read_status(st)[1] == 0
    assert torch.equal(y, y_sep)
    if hist is not None:
        assert torch.equal(h_out, h_sep)


@pytest.mark.parametrize("D,H,dtype", [(512, 4, W.FP8), (1024, 4, W.FP8), (2048, 8, W.FP8_E8M0),
                                       (3072, 2, W.BF16)])
def test_decode_step_other_widths_match_oracle(eg, D, H, dtype):
    """One new token a slot at other row widths through the fused decode launch:
    one warp a slot (D 512), two (D 1024), 8 heads of e8m0-blocked rows (D 2048),
    BF16 rows of 3072 (six warps): streams and history against the oracle."""
    import torch
    cfg, inp, dev, hist = _decode_case(eg, B=129, H=H, D=D, dtype=dtype, rows=(5003, 5009, 5011))
    ref = P.oracle_path(P.HostInputs(cfg, inp.ids, inp.tid2eid, hist.cpu().numpy(), inp.tables,
                                     inp.scales, inp.streams, inp.alpha))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    h_out = torch.empty_like(hist)
    y = eg.engram_forward(dev["ids"], dev["tid2eid"], cfg.n_eids, cfg.H, dev["tables"],
                          dev["streams"], dev["alpha"], cfg.eps, history=hist, history_out=h_out,
                          status=st)
    assert eg.engram_read_status(st)[1] == 0 and ref["flags"] == 0
    P.compare_streams(y.cpu().numpy().view(np.uint16), ref["streams"], inp.streams,
                      what=f"decode D={D} H={H} {dtype}")
    assert np.array_equal(h_out.cpu().numpy(), ref["history"])


def test_fused_decode_bad_token_leaves_its_slot_unwritten(eg):
    """A token id outside the vocabulary flags ENGRAM_FLAG_BAD_TOKEN and leaves
    that slot's streams and history unwritten; the other slots are exact."""
    import torch
    cfg, inp, dev, hist = _decode_case(eg, B=64)
    ids = dev["ids"].clone()
    ids[10, 0] = cfg.vocab + 5
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full_like(dev["streams"], 0x1234)
    h_out = torch.full_like(hist, 77)
    eg.engram_forward(ids, dev["tid2eid"], cfg.n_eids, cfg.H, dev["tables"], dev["streams"],
                      dev["alpha"], cfg.eps, history=hist, history_out=h_out, streams_out=out,
                      status=st)
    assert eg.engram_read_status(st)[1] & eg.FLAG_BAD_TOKEN
    assert torch.all(out[10] == 0x1234) and torch.all(h_out[10] == 77)
    good = eg.engram_forward(dev["ids"], dev["tid2eid"], cfg.n_eids, cfg.H, dev["tables"],
                             dev["streams"], dev["alpha"], cfg.eps, history=hist,
                             history_out=torch.empty_like(hist))
    keep = [b for b in range(cfg.B) if b != 10]
    assert torch.equal(out[keep], good[keep])


@pytest.mark.parametrize("mode", ["queued", "graph"])
def test_back_to_back_decode_steps_equal_synchronised_steps(eg, mode):
    """Sixteen decode steps chained through one history and one set of streams,
    both updated in place, so that every step reads what the step before wrote.
    The fused decode launch lets the next grid start while the previous one
    finishes (programmatic dependent launch); launched back to back (queued
    behind a sleeping kernel, or replayed from a CUDA graph) the steps must give
    the bits of the same steps with a synchronize after each, and the history
    the oracle's hash chain gives."""
    import torch
    import oracle
    cfg = W.by_name("decode_fp8").scaled(B=77, rows=(7001, 7013, 7019))
    inp = P.host_inputs(cfg)
    dev = P.to_device(inp)
    N = 16
    ids_h = [W.token_ids(cfg, 100 + s) for s in range(N)]
    ids = [torch.from_numpy(a).cuda() for a in ids_h]
    ws = torch.empty(max(eg.engram_forward_workspace_bytes(cfg.B, 1, cfg.H), 16),
                     dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    x = torch.empty_like(dev["streams"])
    h = torch.empty_like(dev["history"])

    def reset():
        x.copy_(dev["streams"])
        h.copy_(dev["history"])

    def steps(sync):
        for s in range(N):
            eg.engram_forward(ids[s], dev["tid2eid"], cfg.n_eids, cfg.H, dev["tables"], x,
                              dev["alpha"], cfg.eps, history=h, history_out=h, streams_out=x,
                              workspace=ws, status=st)
            if sync:
                torch.cuda.synchronize()

    reset()
    torch.cuda.synchronize()
    steps(sync=True)
    x_ref, h_ref = x.clone(), h.clone()

    reset()
    if mode == "queued":
        torch.cuda._sleep(20_000_000)  # every launch below is queued before the first runs
        steps(sync=False)
    else:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            steps(sync=False)
        reset()
        g.replay()
    torch.cuda.synchronize()
    assert eg.engram_read_status(st)[1] == 0
    assert torch.equal(h, h_ref)
    assert torch.equal(x, x_ref)

    hist = inp.history
    for a in ids_h:
        e, f1 = oracle.compress(a, inp.tid2eid, cfg.n_eids)
        _, hist, f2 = oracle.hash_ids(e, cfg.H, cfg.rows, history=hist, want_history=True)
        assert f1 == f2 == 0
    assert np.array_equal(h.cpu().numpy(), hist)
