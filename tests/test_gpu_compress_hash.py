"""engram_compress_hash (compression and hash in one launch) against the two
calls it replaces, engram_compress_masked then engram_hash_packed /
engram_hash_bucketed, bit for bit: row ids, compressed ids and history_out, for
plain prefills with a history, packed batches with dead tokens, the prime-bucket
layout, decode steps with the history updated in place, and sequences shorter
than the three-id history.  A bad token id flags ENGRAM_FLAG_BAD_TOKEN and
leaves unwritten exactly its own row ids and those of the tokens whose windows
reach it; every other token's ids equal the two calls'."""
import numpy as np
import pytest

import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu

FILL = 0x5A5A5A5A


@pytest.fixture(scope="module")
def eg():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import hashed_gram_memory_gb300 as eg
    return eg


def _primes(eg, cfg):
    return eg.engram_bucket_primes(1, 4, cfg.H, cfg.hash_vocab)[0] if cfg.hash_vocab else None


CASES = {
    "prefill_h8": W.by_name("full_prefill_fp8").scaled(B=2, S=517, rows=(6007, 6011, 6029)),
    "packed_dead": W.by_name("packed_mm_fp8").scaled(B=2, S=300, rows=(6007, 6011, 6029),
                                                     mean_sample_len=40, image_span=8,
                                                     image_frac=0.3),
    "bucketed": W.by_name("release_layout_fp8").scaled(B=2, S=333, rows=(32_000,) * 3,
                                                       hash_vocab=1000),
    "bucketed_packed_dead": W.by_name("release_layout_fp8").scaled(
        B=2, S=211, D=128, rows=(32_000,) * 3, hash_vocab=1000, packed=True,
        mean_sample_len=50, image_span=8, image_frac=0.25),
    "decode_h4": W.by_name("decode_fp8").scaled(B=300, rows=(7001, 7013, 7019)),
    "h32_ragged": W.by_name("full_prefill_fp8").scaled(B=3, S=67, H=32, rows=(997, 991, 983)),
}


def _two_calls(eg, cfg, dev, ids, history, history_out):
    import torch
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    eids = eg.engram_compress(ids, dev["tid2eid"], cfg.n_eids, status=st, dead=dev.get("dead"))
    rows = eg.engram_hash(eids, cfg.H, cfg.rows, history=history, history_out=history_out,
                          status=st, positions=dev.get("positions"), primes=_primes(eg, cfg))
    return eids, rows, eg.engram_read_status(st)[1]


def _fused(eg, cfg, dev, ids, history, history_out, eids_out=None, rows_out=None):
    import torch
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rows = eg.engram_compress_hash(ids, dev["tid2eid"], cfg.n_eids, cfg.H, cfg.rows,
                                   history=history, history_out=history_out, status=st,
                                   eids_out=eids_out, row_ids_out=rows_out,
                                   positions=dev.get("positions"), dead=dev.get("dead"),
                                   primes=_primes(eg, cfg))
    return rows, eg.engram_read_status(st)[1]


@pytest.mark.parametrize("name", list(CASES))
def test_compress_hash_equals_two_calls(eg, name):
    import torch
    cfg = CASES[name]
    inp = P.host_inputs(cfg)
    dev = P.to_device(inp)
    hist = dev["history"]
    h_sep = torch.empty_like(hist) if hist is not None else None
    eids, rows, f1 = _two_calls(eg, cfg, dev, dev["ids"], hist, h_sep)
    e_out = torch.full_like(dev["ids"], FILL)
    if hist is not None and cfg.S == 1:   # the decode step updates its history in place
        h_in = hist.clone()
        h_out = h_in
    else:
        h_in, h_out = hist, (torch.empty_like(hist) if hist is not None else None)
    got, f2 = _fused(eg, cfg, dev, dev["ids"], h_in, h_out, eids_out=e_out)
    assert f1 == 0 and f2 == 0
    assert torch.equal(got, rows)
    assert torch.equal(e_out, eids)
    if hist is not None:
        assert torch.equal(h_out, h_sep)
    ref = P.oracle_path(inp)
    assert np.array_equal(got.cpu().numpy().reshape(ref["rows"].shape), ref["rows"])


@pytest.mark.parametrize("seq", [1, 2, 5])
def test_compress_hash_short_sequences_history(eg, seq):
    """Sequences shorter than, or just over, the three-id history: history_out is
    the last three ids of history ++ eids, as the two calls give, in place too."""
    import torch
    cfg = W.by_name("decode_fp8").scaled(B=40, S=seq, rows=(7001, 7013, 7019))
    inp = P.host_inputs(cfg)
    dev = P.to_device(inp)
    g = np.random.default_rng(seq)
    hist = torch.from_numpy(g.integers(1, cfg.n_eids, size=(cfg.B, 3)).astype(np.int32)).cuda()
    ids = torch.from_numpy(g.integers(0, cfg.vocab, size=(cfg.B, seq)).astype(np.int32)).cuda()
    h_sep = torch.empty_like(hist)
    _, rows, f1 = _two_calls(eg, cfg, dev, ids, hist, h_sep)
    h_inplace = hist.clone()
    got, f2 = _fused(eg, cfg, dev, ids, h_inplace, h_inplace)
    assert f1 == 0 and f2 == 0
    assert torch.equal(got, rows)
    assert torch.equal(h_inplace, h_sep)


def test_compress_hash_bad_token_leaves_its_reach_unwritten(eg):
    import torch
    cfg = CASES["prefill_h8"]
    inp = P.host_inputs(cfg)
    dev = P.to_device(inp)
    ids = dev["ids"].clone()
    b, p = 1, 200
    ids[b, p] = cfg.vocab + 3
    _, rows, f1 = _two_calls(eg, cfg, dev, dev["ids"], None, None)   # the valid ids' rows
    out = torch.full((cfg.B, cfg.S, 3, cfg.H), FILL, dtype=torch.int32, device="cuda")
    e_out = torch.full_like(ids, FILL)
    got, flags = _fused(eg, cfg, dev, ids, None, None, eids_out=e_out, rows_out=out)
    assert flags & eg.FLAG_BAD_TOKEN
    reach = np.zeros((cfg.B, cfg.S), bool)
    reach[b, p:p + 4] = True          # the token and the three whose windows read it
    g = got.cpu().numpy().reshape(cfg.B, cfg.S, -1)
    r = rows.cpu().numpy().reshape(cfg.B, cfg.S, -1)
    assert np.all(g[reach] == FILL)
    assert np.array_equal(g[~reach], r[~reach])
    e = e_out.cpu().numpy()
    others = np.ones_like(e, bool)
    others[b, p] = False
    assert e[b, p] == FILL and np.all(e[others] != FILL)
