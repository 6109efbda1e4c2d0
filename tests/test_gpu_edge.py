"""GPU edge cases through the C ABI: empty inputs, device-detected bad ids (status
flags, the affected outputs left unwritten, every other output still exact),
decode steps with the history updated in place against the prefill, and the
zero-gate invariants."""
import numpy as np
import pytest

import oracle
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


def _t(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def test_empty_inputs(eg):
    import torch
    cfg = W.by_name("tiny_fp8_d256").scaled(S=0)
    inp = P.host_inputs(W.by_name("tiny_fp8_d256"))
    dev = P.to_device(inp)
    e = eg.engram_compress(torch.zeros((1, 0), dtype=torch.int32, device="cuda"), dev["tid2eid"], 800)
    assert e.numel() == 0
    r = eg.engram_hash(e, 2, cfg.rows)
    assert r.shape == (1, 0, 3, 2)
    y = eg.engram_lookup_fused(r, 2, dev["tables"], torch.empty((0, 4, 256), dtype=torch.int16,
                                                                device="cuda"), dev["alpha"])
    assert y.numel() == 0
    # seq == 0 with a history: history_out is the history itself
    h = _t(np.array([[4, 5, 6], [7, 8, 9]], np.int32))
    ho = torch.full_like(h, -1)
    eg.engram_hash(torch.zeros((2, 0), dtype=torch.int32, device="cuda"), 2, cfg.rows, history=h,
                   history_out=ho)
    assert ho.cpu().tolist() == [[4, 5, 6], [7, 8, 9]]
    torch.cuda.synchronize()


def test_compress_flags_and_unwritten(eg):
    import torch
    m = np.array([3, 0, 9, 12, 5], np.int32)          # 12 > n_eids = 10
    ids = np.array([0, 1, 2, 3, 4, 5, -1, 2], np.int32)
    ref, rflags = oracle.compress(ids, m, 10, fill=-7)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full((8,), -7, dtype=torch.int32, device="cuda")
    eg.engram_compress(_t(ids), _t(m), 10, eids_out=out, status=st)
    code, flags = eg.engram_read_status(st)
    assert code == eg.ERR_OUT_OF_RANGE and flags == rflags == (eg.FLAG_BAD_TOKEN | eg.FLAG_BAD_EID)
    assert out.cpu().numpy().tolist() == ref.tolist()


def test_hash_flags_negative_ids_and_unwritten(eg):
    import torch
    eids = np.array([[3, 4, -1, 5, 6, 7, 8, 9], [1, 2, 3, 4, 5, 6, 7, 8]], np.int32)
    hist = np.array([[1, 2, 3], [-4, 5, 6]], np.int32)
    rows = (101, 103, 107)
    ref, rflags = oracle.hash_ids(eids, 2, rows, history=hist, fill=-7)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full((2, 8, 3, 2), -7, dtype=torch.int32, device="cuda")
    eg.engram_hash(_t(eids), 2, rows, history=_t(hist), row_ids_out=out, status=st)
    code, flags = eg.engram_read_status(st)
    assert flags == rflags == eg.FLAG_BAD_EID
    assert np.array_equal(out.cpu().numpy(), ref)


def test_lookup_flags_bad_rows_and_leaves_token_unwritten(eg):
    import torch
    cfg = W.by_name("tiny_fp8_d256").scaled(S=37)
    inp = P.host_inputs(cfg)
    eids, _ = oracle.compress(inp.ids, inp.tid2eid, cfg.n_eids)
    rows, _ = oracle.hash_ids(eids, cfg.H, cfg.rows)
    rows = rows.reshape(cfg.T, -1).copy()
    rows[3, 1] = cfg.rows[0]          # one past the end of the 2-gram table
    rows[20, 5] = -2
    ref, _, _, rflags = oracle.lookup(rows, cfg.H, oracle.FP8, inp.tables, inp.scales,
                                      inp.streams.reshape(cfg.T, 4, cfg.D), inp.alpha, cfg.eps,
                                      aux=True, fill=0x1234)
    dev = P.to_device(inp)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full((cfg.T, 4, cfg.D), 0x1234, dtype=torch.int16, device="cuda")
    eg.engram_lookup_fused(_t(rows), cfg.H, dev["tables"], dev["streams"].view(cfg.T, 4, cfg.D),
                           dev["alpha"], cfg.eps, streams_out=out, status=st)
    code, flags = eg.engram_read_status(st)
    assert code == eg.ERR_OUT_OF_RANGE and flags == rflags == eg.FLAG_BAD_ROW
    got = out.cpu().numpy().view(np.uint16)
    assert (got[3] == 0x1234).all() and (got[20] == 0x1234).all()
    keep = [t for t in range(cfg.T) if t not in (3, 20)]
    P.compare_streams(got[keep], ref[keep], inp.streams.reshape(cfg.T, 4, cfg.D)[keep])


@pytest.mark.parametrize("H", [4, 8])
def test_bad_rows_in_large_tokens_leave_exactly_those_tokens_unwritten(eg, H):
    """4096-wide rows: one token a block (4 heads) and four tokens chained in a
    block (8 heads, 1300 tokens).  Tokens with an id past its table, a negative
    id, or dead ids mixed with live ones -- first, second, third and last in a
    chained block, and the sequence's last token -- flag ENGRAM_FLAG_BAD_ROW and
    stay unwritten; a fully dead token in a chain copies its streams through;
    every other token equals the oracle."""
    import torch
    cfg = W.by_name("full_prefill_fp8").scaled(B=1, S=1300, H=H, rows=(1009, 1013, 1019))
    inp = P.host_inputs(cfg)
    eids, _ = oracle.compress(inp.ids, inp.tid2eid, cfg.n_eids)
    rows, _ = oracle.hash_ids(eids, cfg.H, cfg.rows)
    rows = rows.reshape(cfg.T, -1).copy()
    bad = {4: ("past", 0), 9: ("neg", 7), 14: ("mix", 3), 7: ("past", 3 * H - 1),
           cfg.T - 1: ("neg", 2)}
    for t, (kind, r) in bad.items():
        if kind == "past":
            rows[t, r] = cfg.rows[r // H]
        elif kind == "neg":
            rows[t, r] = -2
        else:
            rows[t, :r] = oracle.DEAD
    rows[21, :] = oracle.DEAD          # a dead token: streams copied through
    ref, _, _, rflags = oracle.lookup(rows, cfg.H, oracle.FP8, inp.tables, inp.scales,
                                      inp.streams.reshape(cfg.T, 4, cfg.D), inp.alpha, cfg.eps,
                                      aux=True, fill=0x1234)
    dev = P.to_device(inp)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full((cfg.T, 4, cfg.D), 0x1234, dtype=torch.int16, device="cuda")
    eg.engram_lookup_fused(_t(rows), cfg.H, dev["tables"], dev["streams"].view(cfg.T, 4, cfg.D),
                           dev["alpha"], cfg.eps, streams_out=out, status=st)
    code, flags = eg.engram_read_status(st)
    assert code == eg.ERR_OUT_OF_RANGE and flags == rflags == eg.FLAG_BAD_ROW
    got = out.cpu().numpy().view(np.uint16)
    for t in bad:
        assert (got[t] == 0x1234).all(), f"bad token {t} was written"
    assert np.array_equal(got[21], inp.streams.reshape(cfg.T, 4, cfg.D)[21])
    keep = [t for t in range(cfg.T) if t not in bad]
    P.compare_streams(got[keep], ref[keep], inp.streams.reshape(cfg.T, 4, cfg.D)[keep])


@pytest.mark.parametrize("split", [0, 1, 2, 3, 9])
def test_decode_steps_in_place_history_equal_prefill(eg, split):
    import torch
    cfg = W.by_name("decode_fp8").scaled(B=5, S=1, rows=(5_040_000,) * 3)
    g = np.random.default_rng(17 + split)
    S = 14
    eids = g.integers(1, 100_000, size=(cfg.B, S)).astype(np.int32)
    full = eg.engram_hash(_t(eids), cfg.H, cfg.rows).cpu().numpy()
    ref, _ = oracle.hash_ids(eids, cfg.H, cfg.rows)
    assert np.array_equal(full, ref)
    hist = torch.empty((cfg.B, 3), dtype=torch.int32, device="cuda")
    parts = [eg.engram_hash(_t(eids[:, :split]), cfg.H, cfg.rows, history_out=hist).cpu().numpy()]
    for s in range(split, S):
        # history and history_out are the same buffer: the decode cache updated in place
        parts.append(eg.engram_hash(_t(eids[:, s:s + 1]), cfg.H, cfg.rows, history=hist,
                                    history_out=hist).cpu().numpy())
    assert np.array_equal(np.concatenate(parts, axis=1), full)
    assert np.array_equal(hist.cpu().numpy(), eids[:, -3:])


def test_two_token_step_in_place_history(eg):
    import torch
    hist0 = np.array([[5, 6, 7], [1, 2, 3]], np.int32)
    eids = np.array([[9, 10], [11, 12]], np.int32)
    rows = (1009, 1013, 1019)
    ref, href, _ = oracle.hash_ids(eids, 3, rows, history=hist0, want_history=True)
    h = _t(hist0)
    got = eg.engram_hash(_t(eids), 3, rows, history=h, history_out=h).cpu().numpy()
    assert np.array_equal(got, ref) and np.array_equal(h.cpu().numpy(), href)
    torch.cuda.synchronize()


@pytest.mark.parametrize("dtype", [W.FP8, W.BF16])
def test_zero_alpha_and_zero_rows_leave_streams_bit_identical(eg, dtype):
    import torch
    base = W.by_name("tiny_fp8_d256") if dtype == W.FP8 else W.by_name("bf16_tables").scaled(B=1, S=64, rows=(97, 89, 83))
    inp = P.host_inputs(base)
    assert not (inp.streams == 0x8000).any()
    dev = P.to_device(inp)
    dev["alpha"] = torch.zeros(4, dtype=torch.float32, device="cuda")
    res = P.gpu_path(base, dev, aux=False)
    assert np.array_equal(res["streams"], inp.streams)
    dev = P.to_device(inp)
    for t in dev["tables"].tables:
        t.zero_()
    res = P.gpu_path(base, dev, aux=True)
    assert np.array_equal(res["streams"], inp.streams)
    assert np.all(res["mem"] == 0) and np.allclose(res["gate"], 0.5)


@pytest.mark.parametrize("shape", ["one_token_a_block", "small_rows"])
def test_bulk_kernel_bounded_wait_times_out_and_context_survives(eg, shape):
    """A withheld row copy (the mbarrier expects bytes that never come) makes the
    consumers' bounded wait run out: the launch ends by itself with
    ENGRAM_FLAG_TIMEOUT, and the next launch on the same context is exact.  Both
    bulk kernels: 4096-wide rows (a token a block) and the released 256-wide rows
    (16 tokens a block)."""
    import torch
    cfg = (W.by_name("full_prefill_fp8").scaled(B=1, S=700, rows=(1009, 1013, 1019)) if shape == "one_token_a_block"
           else W.by_name("release_layout_fp8").scaled(B=1, S=700, rows=(32_000,) * 3, hash_vocab=1000))
    inp = P.host_inputs(cfg)
    ref = P.oracle_path(inp)
    dev = P.to_device(inp)
    prev_k = eg.engram_set_lookup_kernel(eg.LOOKUP_BULK)
    prev_l = eg.engram_set_wait_limit_ns(5_000_000)
    try:
        eg.engram_debug_withhold_copies(1)
        res = P.gpu_path(cfg, dev, aux=False)
        assert res["code"] == eg.ERR_TIMEOUT and res["flags"] & eg.FLAG_TIMEOUT
        torch.cuda.synchronize()
        again = P.gpu_path(cfg, dev, aux=True)
        assert again["flags"] == 0
        P.compare_all(again, ref)
    finally:
        eg.engram_debug_withhold_copies(0)
        eg.engram_set_wait_limit_ns(prev_l)
        eg.engram_set_lookup_kernel(prev_k)


def test_decode_step_bounded_wait_times_out_and_context_survives(eg):
    """The fused decode launch with a withheld row copy in every slot: each
    slot's bounded wait on that row runs out, the launch ends by itself with
    ENGRAM_FLAG_TIMEOUT and leaves every slot's streams unwritten, and the next
    decode step on the same context matches the oracle."""
    import torch
    cfg = W.by_name("decode_fp8").scaled(B=40, rows=(7001, 7013, 7019))
    inp = P.host_inputs(cfg)
    ref = P.oracle_path(inp)
    dev = P.to_device(inp)
    prev_l = eg.engram_set_wait_limit_ns(5_000_000)
    try:
        eg.engram_debug_withhold_copies(1)
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = torch.full_like(dev["streams"], 0x5555)
        eg.engram_forward(dev["ids"], dev["tid2eid"], cfg.n_eids, cfg.H, dev["tables"],
                          dev["streams"], dev["alpha"], cfg.eps, history=dev["history"],
                          streams_out=out, status=st)
        code, flags = eg.engram_read_status(st)
        assert code == eg.ERR_TIMEOUT and flags & eg.FLAG_TIMEOUT
        assert bool((out == 0x5555).all()), "a timed-out slot wrote its streams"
        torch.cuda.synchronize()
        st.zero_()
        hist_out = torch.empty_like(dev["history"])
        again = eg.engram_forward(dev["ids"], dev["tid2eid"], cfg.n_eids, cfg.H, dev["tables"],
                                  dev["streams"], dev["alpha"], cfg.eps, history=dev["history"],
                                  history_out=hist_out, status=st)
        assert eg.engram_read_status(st)[1] == 0
        P.compare_streams(again.cpu().numpy().view(np.uint16), ref["streams"], inp.streams,
                          what="decode step after a timeout")
        assert np.array_equal(hist_out.cpu().numpy(), ref["history"])
    finally:
        eg.engram_debug_withhold_copies(0)
        eg.engram_set_wait_limit_ns(prev_l)


@pytest.mark.parametrize("pos", [0, 1, 2, 3, 40])
def test_decode_positions_and_dead_history_match_oracle(eg, pos):
    """Decode steps of packed requests: the start position bounds how far back the
    history is read, a dead history entry blocks the lookback, dead tokens pass
    through; the history updated in place carries the dead markers."""
    import torch
    g = np.random.default_rng(30 + pos)
    B = 7
    hist = g.integers(1, 100_000, size=(B, 3)).astype(np.int32)
    hist[1, 1] = oracle.DEAD
    hist[4, 2] = oracle.DEAD
    eids = g.integers(1, 100_000, size=(B, 1)).astype(np.int32)
    eids[5, 0] = oracle.DEAD
    positions = np.full((B, 1), pos, np.int32)
    positions[6, 0] = 1
    rows = (10007, 10009, 10037)
    ref, href, flags = oracle.hash_ids(eids, 4, rows, history=hist, want_history=True,
                                       positions=positions)
    assert flags == 0
    h = _t(hist)
    got = eg.engram_hash(_t(eids), 4, rows, history=h, history_out=h, positions=_t(positions))
    assert np.array_equal(got.cpu().numpy(), ref)
    assert np.array_equal(h.cpu().numpy(), href)
    torch.cuda.synchronize()


def test_masked_compress_matches_oracle(eg):
    g = np.random.default_rng(5)
    m = g.integers(1, 50, size=64).astype(np.int32)
    ids = g.integers(-3, 70, size=200).astype(np.int32)
    dead = (g.random(200) < 0.3).astype(np.uint8)
    ref, rflags = oracle.compress_masked(ids, m, 49, dead, fill=-7)
    import torch
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full((200,), -7, dtype=torch.int32, device="cuda")
    eg.engram_compress(_t(ids), _t(m), 49, eids_out=out, status=st, dead=_t(dead))
    assert eg.engram_read_status(st)[1] == rflags
    assert np.array_equal(out.cpu().numpy(), ref)
