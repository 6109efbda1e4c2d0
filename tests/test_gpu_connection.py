"""Parity of engram_connection (a token's 3H rows concatenated, k = wkv e on the
tensor cores, the gate, the add into the four streams) against the oracle's
connection on the same seeded inputs; the row ids come from the GPU hash and are
first checked bit-exact against the oracle's.

Tolerances (derived from the arithmetic, written out below):
* k: the rows are exact in bf16 and every product w*e is exact in fp32; the
  tensor cores add K/16 partial sums of 16 products into an fp32 accumulator,
  each step off by at most one fp32 rounding of a value bounded by
  S_j = sum_i |w_ji e_i|.  Allowing 2^-22 per step and 16 steps more:
  |k_j - k_ref_j| <= (K/16 + 16) 2^-22 S_j.
  On average the errors must look like rounding, not like a wrong term: the rms
  of |k_j - k_ref_j| / S_j stays within sqrt(K/16 + 16) 2^-23.
* g: the gate's logit moved by the measured k errors dk, to first order and
  doubled, times the sigmoid's largest slope 1/4, plus 1e-5 for its fp32
  evaluation.
* streams: the stated allclose bar (max-abs 2e-2 / rel 1e-2) without exception,
  and per element one bf16 ulp of the oracle's value plus the fp32 rounding of
  the operands plus |alpha_s| (g dk_j + |k_j| gb): the update's own error.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu

FILL = 0x1234   # pre-filled output: bad tokens must leave it unwritten

BASE = W.by_name("release_connection_e8m0")
SMALL = {
    # BF16 tables, K = 3*2*64 = 384, hidden 256 (one N tile), 300 tokens (3 M tiles, ragged)
    "bf16_h2_d64": BASE.scaled(B=1, S=300, H=2, D=64, rows=(1009, 1013, 1019), hash_vocab=0,
                               dtype=W.BF16, hidden=256, wkv_std=2.0),
    # e8m0 tables, K = 768, hidden 512 (two N tiles), 2 x 129 tokens
    "e8m0_h2_d128": BASE.scaled(B=2, S=129, H=2, D=128, rows=(2003, 2011, 2017), hash_vocab=0,
                                hidden=512),
    # the released row shape: K = 24 * 256 = 6144 (96 K steps, the stage ring wraps 24 times)
    "e8m0_h8_d256": BASE.scaled(B=1, S=200, H=8, D=256, rows=(3001, 3011, 3019), hash_vocab=0,
                                hidden=1024),
    # the full stream width (16 N tiles), one M tile exactly
    "e8m0_h8_wide": BASE.scaled(B=1, S=128, H=8, D=256, rows=(3001, 3011, 3019), hash_vocab=0,
                                hidden=4096),
    # a single token (the tile is almost all zero fill)
    "one_token": BASE.scaled(B=1, S=1, H=4, D=256, rows=(101, 103, 107), hash_vocab=0,
                             hidden=512),
    # 16,684 tokens: 131 M tiles, about one tile per CTA at the end of the walk
    "many_tiles": BASE.scaled(B=1, S=16384 + 300, H=2, D=64, rows=(1009, 1013, 1019),
                           hash_vocab=0, dtype=W.BF16, hidden=256),
    # the released row shape with each row's exponents stored after it (272-byte rows)
    "rows_h8_d256": BASE.scaled(B=1, S=200, H=8, D=256, rows=(3001, 3011, 3019), hash_vocab=0,
                                hidden=1024, dtype=W.FP8_E8M0_ROWS),
    # packed samples with image spans: dead tokens pass through
    "packed_dead": BASE.scaled(B=2, S=150, H=2, D=128, rows=(1009, 1013, 1019), hash_vocab=0,
                               hidden=256, packed=True, mean_sample_len=64, image_span=16,
                               image_frac=0.25),
}


@pytest.fixture(scope="module")
def eg():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import hashed_gram_memory_gb300 as eg
    return eg


def _e4m3_lut():
    return np.array([oracle.e4m3fn_decode(b) for b in range(256)])


def abs_rows(cfg, tables, scales, rows):
    """|e| [T, K] in fp64 (for the tolerance only): the magnitudes of the
    dequantised rows; dead tokens and tokens with a row outside its table give
    zeros."""
    T = rows.shape[0]
    e = np.zeros((T, cfg.K))
    lut = _e4m3_lut() if cfg.dtype != W.BF16 else None
    for t in range(T):
        ids = rows[t]
        if (ids < 0).any() or any(ids[r] >= len(tables[r // cfg.H]) for r in range(cfg.R)):
            continue
        for r in range(cfg.R):
            n = r // cfg.H
            if cfg.dtype == W.BF16:
                v = oracle.bf16_bits_to_float(tables[n][ids[r]]).astype(np.float64)
            else:
                v = lut[tables[n][ids[r]]] * np.ldexp(
                    1.0, np.repeat(scales[n][ids[r]].astype(np.int64) - 127, 32))
            e[t, r * cfg.D:(r + 1) * cfg.D] = np.abs(v)
    return e


def k_bound(cfg, wkv_bits, e_abs):
    """kb [T, hidden]: the worst-case error of k, as the module docstring derives it."""
    w = np.abs(oracle.bf16_bits_to_float(wkv_bits).astype(np.float64))
    S = e_abs @ w.T
    return (cfg.K / 16 + 16) * 2.0 ** -22 * S, S


def gate_bound(cfg, x_bits, k_ref, dk):
    """gb [T]: how far the gate may move when k is off by dk [T, hidden] (first
    order, doubled), times the sigmoid's largest slope, plus fp32 evaluation."""
    a = oracle.bf16_bits_to_float(x_bits[:, 0, :]).astype(np.float64)
    D = cfg.hidden
    k = np.nan_to_num(k_ref)
    ra = np.sqrt((a * a).sum(-1) / D + cfg.eps)
    rk = np.sqrt((k * k).sum(-1) / D + cfg.eps)
    logit = (a * k).sum(-1) / (ra * rk * np.sqrt(D))
    d_sak = (np.abs(a) * dk).sum(-1)
    d_skk = 2 * (np.abs(k) * dk).sum(-1) + (dk * dk).sum(-1)
    d_logit = d_sak / (ra * rk * np.sqrt(D)) + np.abs(logit) * d_skk / (2 * D * rk * rk)
    return 1e-5 + 0.25 * 2 * d_logit


def compare_connection(cfg, res, ref, x_bits, alpha, kb, S, live):
    """Checks k, g and the streams of the live tokens (mask `live`): k within its
    worst-case bound, and its errors no larger on average than a random walk of
    K/16 + 16 fp32 roundings; g and the streams within what the measured k error
    and their own rounding allow."""
    y_ref, g_ref, k_ref = ref
    dk = np.abs(res["k"][live] - k_ref[live])
    assert np.all(dk <= kb[live]), f"k: worst err/bound {np.max(dk / kb[live]):.3g}"
    rel = dk / np.maximum(S[live], 1e-300)
    rms = float(np.sqrt(np.mean(rel * rel)))
    assert rms <= np.sqrt(cfg.K / 16 + 16) * 2.0 ** -23, f"k: rms error {rms:.3g} of sum |w e|"
    x = x_bits[live]
    gb = gate_bound(cfg, x, k_ref[live], dk)
    g_err = np.abs(res["gate"][live] - g_ref[live])
    assert np.all(g_err <= gb), f"g: worst err/bound {np.max(g_err / gb):.3g}"
    yg = oracle.bf16_bits_to_float(res["streams"][live]).astype(np.float64)
    yr = oracle.bf16_bits_to_float(y_ref[live]).astype(np.float64)
    xf = oracle.bf16_bits_to_float(x).astype(np.float64)
    assert np.isfinite(yg).all()
    err = np.abs(yg - yr)
    bar = P.STREAM_ATOL + P.STREAM_RTOL * np.abs(yr)
    assert np.all(err <= bar), f"streams: allclose bar, worst err/bound {np.max(err / bar):.3g}"
    a = np.abs(alpha.astype(np.float64))[None, :, None]
    upd = a * (g_ref[live][:, None, None] * dk[:, None, :] +
               np.abs(k_ref[live])[:, None, :] * gb[:, None, None])
    tight = P.bf16_ulp(yr) + 2.0 ** -23 * np.abs(xf) + 2.0 ** -16 * np.abs(yr - xf) + upd
    assert np.all(err <= tight), f"streams: tight bound exceeded by {np.max(err / tight):.3g}x"
    return dict(k_rms_rel=rms, max_gate_err=float(g_err.max()),
                mismatch_frac=float(np.mean(res["streams"][live] != y_ref[live])))


def run_gpu(eg, cfg, inp, wkv_bits, in_place=False, with_k=True, rows_override=None):
    import torch
    dev = P.to_device(inp)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    eids = eg.engram_compress(dev["ids"], dev["tid2eid"], cfg.n_eids, status=status,
                              dead=dev.get("dead"))
    rows = eg.engram_hash(eids, cfg.H, cfg.rows, history=dev["history"], status=status,
                          positions=dev.get("positions"))
    if rows_override is not None:
        rows = torch.from_numpy(rows_override).cuda()
    T, Dm = cfg.T, cfg.hidden
    x = dev["streams"].view(T, 4, Dm)
    wkv = torch.from_numpy(wkv_bits.view(np.int16)).cuda()
    gate = torch.full((T,), float("nan"), device="cuda")
    k = torch.full((T, Dm), float("nan"), device="cuda") if with_k else None
    if in_place:
        out = x.clone()
        src = out
    else:
        out = torch.full_like(x, FILL)
        src = x
    eg.engram_connection(rows, cfg.H, dev["tables"], wkv, src, dev["alpha"], cfg.eps,
                         streams_out=out, gate_out=gate, k_out=k, status=status)
    code, flags = eg.engram_read_status(status)
    return dict(rows=rows.cpu().numpy(), streams=out.cpu().numpy().view(np.uint16),
                gate=gate.cpu().numpy(), k=None if k is None else k.cpu().numpy(),
                flags=flags, code=code)


def oracle_rows(cfg, inp):
    if inp.dead is not None:
        eids, _ = oracle.compress_masked(inp.ids, inp.tid2eid, cfg.n_eids, inp.dead)
    else:
        eids, _ = oracle.compress(inp.ids, inp.tid2eid, cfg.n_eids)
    rows, _ = oracle.hash_ids(eids, cfg.H, cfg.rows, history=inp.history,
                              positions=inp.positions)
    return rows.reshape(cfg.T, -1)


def oracle_connection(cfg, inp, rows, wkv_bits):
    x = inp.streams.reshape(cfg.T, 4, cfg.hidden)
    tabs, scs = P.oracle_tables(cfg, inp.tables, inp.scales)
    y, g, k, flags = oracle.connection(rows, cfg.H, P.oracle_dtype(cfg), tabs, scs,
                                       wkv_bits, x, inp.alpha, cfg.eps, rows=cfg.rows, fill=FILL)
    return y, g, k, flags


@pytest.mark.parametrize("name", list(SMALL))
def test_connection_parity(eg, name):
    cfg = SMALL[name]
    inp = P.host_inputs(cfg)
    wkv = W.wkv_host(cfg)
    rows = oracle_rows(cfg, inp)
    res = run_gpu(eg, cfg, inp, wkv)
    assert res["code"] == eg.OK and res["flags"] == 0, res["flags"]
    assert np.array_equal(res["rows"].reshape(cfg.T, -1), rows)
    y_ref, g_ref, k_ref, flags = oracle_connection(cfg, inp, rows, wkv)
    assert flags == 0
    x = inp.streams.reshape(cfg.T, 4, cfg.hidden)
    dead = (rows == oracle.DEAD).all(axis=1)
    live = ~dead
    assert live.any()
    kb, S = k_bound(cfg, wkv, abs_rows(cfg, *P.oracle_tables(cfg, inp.tables, inp.scales), rows))
    compare_connection(cfg, res, (y_ref, g_ref, k_ref), x, inp.alpha, kb, S, live)
    if dead.any():   # copied through, g = 0, k = 0
        assert np.array_equal(res["streams"][dead], x[dead])
        assert np.all(res["gate"][dead] == 0) and np.all(res["k"][dead] == 0)
    if name == "packed_dead":
        assert dead.any()


def test_connection_in_place_and_without_k(eg):
    """In place (streams_out == streams_in) and with k kept in the workspace give
    the same bits as the out-of-place run with k_out."""
    cfg = SMALL["e8m0_h2_d128"]
    inp = P.host_inputs(cfg)
    wkv = W.wkv_host(cfg)
    a = run_gpu(eg, cfg, inp, wkv)
    b = run_gpu(eg, cfg, inp, wkv, in_place=True, with_k=False)
    assert a["flags"] == b["flags"] == 0
    assert np.array_equal(a["streams"], b["streams"])
    assert np.array_equal(a["gate"], b["gate"])


def test_stages_compose_to_connection(eg):
    """engram_concat_rows -> engram_wkv_project -> engram_gate_add give the same
    bits as engram_connection, and E holds exactly the dequantised rows (each
    value exact in bf16: bit-exact against the oracle's decoders)."""
    import torch
    cfg = SMALL["e8m0_h8_d256"]
    inp = P.host_inputs(cfg)
    wkv_h = W.wkv_host(cfg)
    rows_h = oracle_rows(cfg, inp)
    dev = P.to_device(inp)
    rows = torch.from_numpy(rows_h).cuda()
    wkv = torch.from_numpy(wkv_h.view(np.int16)).cuda()
    x = dev["streams"].view(cfg.T, 4, cfg.hidden)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    g1 = torch.empty(cfg.T, device="cuda")
    k1 = torch.empty((cfg.T, cfg.hidden), device="cuda")
    y1 = eg.engram_connection(rows, cfg.H, dev["tables"], wkv, x, dev["alpha"], cfg.eps,
                              gate_out=g1, k_out=k1, status=st)
    E, state = eg.engram_concat_rows(rows, cfg.H, dev["tables"], status=st)
    k2 = eg.engram_wkv_project(E, wkv, status=st)
    g2 = torch.empty(cfg.T, device="cuda")
    y2 = eg.engram_gate_add(k2, state, x, dev["alpha"], cfg.eps, gate_out=g2)
    assert eg.engram_read_status(st)[1] == 0
    assert torch.equal(y1, y2) and torch.equal(g1, g2) and torch.equal(k1, k2)
    assert torch.all(state == 0)
    lut = _e4m3_lut()
    e_ref = np.empty((cfg.T, cfg.K))
    for t in range(cfg.T):
        for r in range(cfg.R):
            n, row = r // cfg.H, rows_h[t, r]
            sc = np.array([oracle.e8m0_decode(int(b)) for b in inp.scales[n][row]])
            e_ref[t, r * cfg.D:(r + 1) * cfg.D] = lut[inp.tables[n][row]] * np.repeat(sc, 32)
    bits = (e_ref.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(oracle.bf16_bits_to_float(bits).astype(np.float64), e_ref)
    assert np.array_equal(E.view(torch.int16).cpu().numpy().view(np.uint16), bits)


@pytest.mark.parametrize("name", ["bf16_h2_d64", "e8m0_h8_wide", "one_token", "many_tiles"])
def test_projection_kernels_identical(eg, name):
    """The CTA-pair projection (256 x 256 tiles, cta_group::2) and the one-CTA
    projection (128 x 256 tiles) add the same products in the same order: the
    same bits, including a lone token and a ragged last pair of tiles."""
    import torch
    cfg = SMALL[name]
    inp = P.host_inputs(cfg)
    dev = P.to_device(inp)
    rows = torch.from_numpy(oracle_rows(cfg, inp)).cuda()
    wkv = torch.from_numpy(W.wkv_host(cfg).view(np.int16)).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    E, _ = eg.engram_concat_rows(rows, cfg.H, dev["tables"], status=st)
    out = {}
    try:
        for which in (eg.PROJECTION_PAIR, eg.PROJECTION_SINGLE):
            eg.engram_set_projection_kernel(which)
            out[which] = eg.engram_wkv_project(E, wkv, status=st)
    finally:
        eg.engram_set_projection_kernel(eg.PROJECTION_AUTO)
    assert eg.engram_read_status(st)[1] == 0
    assert torch.equal(out[eg.PROJECTION_PAIR], out[eg.PROJECTION_SINGLE])


def test_connection_bad_rows(eg):
    """A row id outside its table, or some (not all) ids dead, is a bad row: the
    flag is raised and that token's streams are left unwritten; the others are
    unaffected."""
    cfg = SMALL["bf16_h2_d64"]
    inp = P.host_inputs(cfg)
    wkv = W.wkv_host(cfg)
    rows = oracle_rows(cfg, inp).copy()
    rows[5, 3] = cfg.rows[1]           # one past the 3-gram table
    rows[77, 0] = oracle.DEAD          # partly dead
    rows[150, :] = oracle.DEAD         # wholly dead: passes through
    res = run_gpu(eg, cfg, inp, wkv, rows_override=rows)
    assert res["flags"] & eg.FLAG_BAD_ROW
    y_ref, g_ref, k_ref, flags = oracle_connection(cfg, inp, rows, wkv)
    assert flags & oracle.BAD_ROW
    x = inp.streams.reshape(cfg.T, 4, cfg.hidden)
    for t in (5, 77):
        assert np.all(res["streams"][t] == FILL) and np.all(y_ref[t] == FILL)
    assert np.array_equal(res["streams"][150], x[150])
    live = np.ones(cfg.T, bool)
    live[[5, 77, 150]] = False
    kb, S = k_bound(cfg, wkv, abs_rows(cfg, inp.tables, inp.scales, rows))
    compare_connection(cfg, res, (y_ref, g_ref, k_ref), x, inp.alpha, kb, S, live)


def test_connection_host_errors(eg):
    """Argument errors come back before any launch: per-row-scale FP8 tables,
    a stream width the projection does not tile, a short workspace."""
    import torch
    cfg = SMALL["e8m0_h2_d128"]
    inp = P.host_inputs(cfg)
    dev = P.to_device(inp)
    rows = torch.zeros((cfg.T, cfg.R), dtype=torch.int32, device="cuda")
    wkv = torch.zeros((cfg.hidden, cfg.K), dtype=torch.int16, device="cuda")
    x = dev["streams"].view(cfg.T, 4, cfg.hidden)
    fp8 = eg.Tables(eg.TABLE_FP8_E4M3FN, dev["tables"].tables,
                    [torch.ones(r, device="cuda") for r in cfg.rows])
    with pytest.raises(eg.EngramError) as ei:
        eg.engram_connection(rows, cfg.H, fp8, wkv, x, dev["alpha"])
    assert ei.value.code == eg.ERR_UNSUPPORTED
    x300 = torch.zeros((cfg.T, 4, 320), dtype=torch.int16, device="cuda")
    w300 = torch.zeros((320, cfg.K), dtype=torch.int16, device="cuda")
    with pytest.raises(eg.EngramError) as ei:
        eg.engram_connection(rows, cfg.H, dev["tables"], w300, x300, dev["alpha"])
    assert ei.value.code == eg.ERR_UNSUPPORTED
    short = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(eg.EngramError) as ei:
        eg.engram_connection(rows, cfg.H, dev["tables"], wkv, x, dev["alpha"], workspace=short)
    assert ei.value.code == eg.ERR_INVALID_ARG


def test_connection_full_size_sampled(eg):
    """The released layout at full size (65,536 tokens, 24 rows of 256 from the
    98 GB bucketed table, projected to 4096): every row id against the oracle,
    then k, g and the streams on a seeded sample of tokens, for which the oracle
    gets exactly the rows and stream values the GPU read."""
    import torch
    cfg = BASE
    free = torch.cuda.mem_get_info()[0]
    need = cfg.table_bytes() + 2 * cfg.T * 4 * cfg.hidden * 2 + \
        eg.engram_connection_workspace_bytes(cfg.T, cfg.H, cfg.D, cfg.hidden) + (4 << 30)
    if free < need:
        pytest.skip(f"needs {need / 2**30:.1f} GiB of device memory, {free / 2**30:.1f} free")
    tabs, scales = W.tables_device(cfg, "cuda")
    tables = eg.Tables(eg.TABLE_FP8_E8M0, tabs, scales)
    ids = torch.from_numpy(W.token_ids(cfg)).cuda()
    tid2eid = torch.from_numpy(W.tid2eid(cfg)).cuda()
    x = W.streams_device(cfg, "cuda").view(cfg.T, 4, cfg.hidden)
    wkv = W.wkv_device(cfg, "cuda")
    alpha = torch.from_numpy(W.alpha(cfg)).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    primes = eg.engram_bucket_primes(1, 4, cfg.H, cfg.hash_vocab)[0]
    eids = eg.engram_compress(ids, tid2eid, cfg.n_eids, status=st)
    rows = eg.engram_hash(eids, cfg.H, cfg.rows, status=st, primes=primes)
    out = torch.empty_like(x)
    k = torch.empty((cfg.T, cfg.hidden), dtype=torch.float32, device="cuda")
    gate = torch.empty((cfg.T,), dtype=torch.float32, device="cuda")
    eg.engram_connection(rows, cfg.H, tables, wkv, x, alpha, cfg.eps, streams_out=out,
                         gate_out=gate, k_out=k, status=st)
    code, flags = eg.engram_read_status(st)
    assert flags == 0

    e_ref, _ = oracle.compress(ids.cpu().numpy(), tid2eid.cpu().numpy(), cfg.n_eids)
    r_ref, _ = oracle.hash_bucketed(e_ref, cfg.H, P.layer_primes(cfg))
    r_ref = r_ref.reshape(cfg.T, -1)
    assert np.array_equal(rows.cpu().numpy().reshape(cfg.T, -1), r_ref)

    g = np.random.default_rng(1008)
    toks = np.unique(np.concatenate([[0, cfg.T - 1], g.choice(cfg.T, size=64, replace=False)]))
    rr = r_ref[toks]
    uniq, inv = np.unique(rr, return_inverse=True)
    remap = inv.reshape(rr.shape).astype(np.int32)
    idx = torch.from_numpy(uniq.astype(np.int64)).cuda()
    t_h = tabs[0].index_select(0, idx).cpu().numpy()
    s_h = scales[0].index_select(0, idx).cpu().numpy()
    sub = cfg.scaled(rows=(len(uniq),) * 3, hash_vocab=0)
    tsel = torch.from_numpy(toks).cuda()
    x_h = x[tsel].cpu().numpy().view(np.uint16)
    w_h = wkv.cpu().numpy().view(np.uint16)
    y_ref, g_ref, k_ref, f = oracle.connection(remap, cfg.H, oracle.FP8_E8M0, [t_h] * 3,
                                               [s_h] * 3, w_h, x_h, W.alpha(cfg), cfg.eps)
    assert f == 0
    res = dict(streams=out[tsel].cpu().numpy().view(np.uint16), gate=gate[tsel].cpu().numpy(),
               k=k[tsel].cpu().numpy())
    kb, S = k_bound(sub, w_h, abs_rows(sub, [t_h] * 3, [s_h] * 3, remap))
    compare_connection(sub, res, (y_ref, g_ref, k_ref), x_h, W.alpha(cfg), kb, S,
                       np.ones(len(toks), bool))
    del tabs, scales, tables, x, out, k
    torch.cuda.empty_cache()
