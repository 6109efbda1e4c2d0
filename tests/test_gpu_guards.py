"""Stray writes and chunked prefill, on the GPU.

Guard bands stand in for a memory checker (closed on this pool): every output
of every entry point is a slice in the middle of a larger buffer whose margins
hold a canary pattern, and after the call the margins must be untouched, the
slice written as the oracle (or engram_forward) says.  A prefill cut into
chunks that carry the three-id history must give the streams and the final
history of the whole sequence, bit for bit."""
import numpy as np
import pytest

import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu

MARGIN = 4096          # bytes on each side of an output (a multiple of 16)
CANARY = 0xA5


@pytest.fixture(scope="module")
def eg():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import hashed_gram_memory_gb300 as eg
    return eg


class Guarded:
    """An output tensor of `shape` and `dtype` carved from the middle of a byte
    buffer whose MARGIN-byte margins hold CANARY."""

    def __init__(self, shape, dtype):
        import torch
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.buf = torch.full((2 * MARGIN + n,), CANARY, dtype=torch.uint8, device="cuda")
        self.t = self.buf[MARGIN:MARGIN + n].view(dtype).view(shape)

    def margins_intact(self) -> bool:
        b = self.buf.cpu().numpy()
        return bool((b[:MARGIN] == CANARY).all() and (b[-MARGIN:] == CANARY).all())


def test_every_output_stays_inside_its_buffer(eg):
    import torch
    cfg = W.by_name("full_prefill_fp8").scaled(B=2, S=301, rows=(6007, 6011, 6029))
    inp = P.host_inputs(cfg)
    ref = P.oracle_path(inp)
    dev = P.to_device(inp)
    B, S, H, T, D = cfg.B, cfg.S, cfg.H, cfg.T, cfg.D
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    eids = Guarded((B, S), torch.int32)
    eg.engram_compress(dev["ids"], dev["tid2eid"], cfg.n_eids, eids_out=eids.t, status=st)
    rows = Guarded((B, S, 3, H), torch.int32)
    eg.engram_hash(eids.t, H, cfg.rows, row_ids_out=rows.t, status=st)
    rows2 = Guarded((B, S, 3, H), torch.int32)
    eids2 = Guarded((B, S), torch.int32)
    eg.engram_compress_hash(dev["ids"], dev["tid2eid"], cfg.n_eids, H, cfg.rows,
                            row_ids_out=rows2.t, eids_out=eids2.t, status=st)
    out = Guarded(tuple(dev["streams"].shape), torch.int16)
    gate = Guarded((T,), torch.float32)
    mem = Guarded((T, D), torch.float32)
    eg.engram_lookup_fused(rows.t, H, dev["tables"], dev["streams"], dev["alpha"], cfg.eps,
                           streams_out=out.t, gate_out=gate.t, mem_out=mem.t, status=st)
    fwd = Guarded(tuple(dev["streams"].shape), torch.int16)
    eg.engram_forward(dev["ids"], dev["tid2eid"], cfg.n_eids, H, dev["tables"], dev["streams"],
                      dev["alpha"], cfg.eps, streams_out=fwd.t, status=st)
    torch.cuda.synchronize()
    assert eg.engram_read_status(st)[1] == 0
    for name, g in (("eids", eids), ("rows", rows), ("rows (compress-hash)", rows2),
                    ("eids (compress-hash)", eids2), ("streams", out), ("gate", gate),
                    ("mem", mem), ("streams (forward)", fwd)):
        assert g.margins_intact(), f"{name}: a write outside the output"
    assert np.array_equal(eids.t.cpu().numpy(), ref["eids"])
    assert np.array_equal(rows.t.cpu().numpy(), ref["rows"])
    assert np.array_equal(rows2.t.cpu().numpy(), ref["rows"])
    P.compare_streams(out.t.cpu().numpy().view(np.uint16), ref["streams"], inp.streams)
    assert np.array_equal(fwd.t.cpu().numpy(), out.t.cpu().numpy())


def test_decode_and_rows_layout_outputs_stay_inside(eg):
    """The fused decode launch's streams and history, the 256-wide small-row
    lookup and the packing of rows with their exponents."""
    import torch
    cfg = W.by_name("decode_fp8").scaled(B=77, rows=(7001, 7013, 7019))
    inp = P.host_inputs(cfg)
    ref = P.oracle_path(inp)
    dev = P.to_device(inp)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = Guarded(tuple(dev["streams"].shape), torch.int16)
    hist = Guarded((cfg.B, 3), torch.int32)
    eg.engram_forward(dev["ids"], dev["tid2eid"], cfg.n_eids, cfg.H, dev["tables"],
                      dev["streams"], dev["alpha"], cfg.eps, history=dev["history"],
                      history_out=hist.t, streams_out=out.t, status=st)
    rl = W.by_name("release_layout_fp8").scaled(B=1, S=300, rows=(32_000,) * 3, hash_vocab=1000)
    rinp = P.host_inputs(rl)
    rref = P.oracle_path(rinp)
    rdev = P.to_device(rinp)
    t, e = rdev["tables"].tables[0], rdev["tables"].scales[0]
    packed = Guarded((t.shape[0], eg.e8m0_row_bytes(rl.D)), torch.uint8)
    eg.engram_pack_e8m0_rows(t, e, packed=packed.t)
    primes = P.layer_primes(rl)
    rows = eg.engram_hash(eg.engram_compress(rdev["ids"], rdev["tid2eid"], rl.n_eids), rl.H,
                          rl.rows, primes=primes)
    rout = Guarded(tuple(rdev["streams"].shape), torch.int16)
    eg.engram_lookup_fused(rows, rl.H, eg.Tables(eg.TABLE_FP8_E8M0_ROWS, [packed.t] * 3, None),
                           rdev["streams"], rdev["alpha"], rl.eps, streams_out=rout.t, status=st)
    torch.cuda.synchronize()
    assert eg.engram_read_status(st)[1] == 0
    for name, g in (("decode streams", out), ("decode history", hist), ("packed rows", packed),
                    ("rows-layout streams", rout)):
        assert g.margins_intact(), f"{name}: a write outside the output"
    P.compare_streams(out.t.cpu().numpy().view(np.uint16), ref["streams"], inp.streams)
    assert np.array_equal(hist.t.cpu().numpy(), ref["history"])
    P.compare_streams(rout.t.cpu().numpy().view(np.uint16), rref["streams"], rinp.streams)


@pytest.mark.parametrize("cuts", [[200], [1, 300], [150, 151], [64, 64, 64]])
def test_chunked_prefill_equals_the_whole_sequence(eg, cuts):
    """A prefill cut into chunks, each engram_forward call taking the previous
    chunk's history_out (and positions continuing the sequence), gives the
    streams and the final history of one call over the whole sequence, bit for
    bit: an n-gram only needs the three ids before a chunk."""
    import torch
    cfg = W.by_name("full_prefill_fp8").scaled(B=2, S=301, rows=(6007, 6011, 6029))
    dev = P.to_device(P.host_inputs(cfg))
    B, S = cfg.B, cfg.S
    whole_hist = torch.empty((B, 3), dtype=torch.int32, device="cuda")
    whole = eg.engram_forward(dev["ids"], dev["tid2eid"], cfg.n_eids, cfg.H, dev["tables"],
                              dev["streams"], dev["alpha"], cfg.eps, history_out=whole_hist)
    x = dev["streams"]
    bounds = [0] + [c for c in np.cumsum(cuts) if c < S] + [S]
    hist = None
    parts = []
    for a, b in zip(bounds[:-1], bounds[1:]):
        ids = dev["ids"][:, a:b].contiguous()
        pos = torch.arange(a, b, dtype=torch.int32, device="cuda").expand(B, -1).contiguous()
        h_out = torch.empty((B, 3), dtype=torch.int32, device="cuda")
        y = eg.engram_forward(ids, dev["tid2eid"], cfg.n_eids, cfg.H, dev["tables"],
                              x[:, a:b].contiguous(), dev["alpha"], cfg.eps, history=hist,
                              history_out=h_out, positions=pos)
        parts.append(y)
        hist = h_out
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(parts, dim=1), whole)
    assert torch.equal(hist, whole_hist)
