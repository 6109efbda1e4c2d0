"""The synthetic input recipe (workloads.py), without a GPU: the workloads have
the sizes the measurement contract lists for each configuration, their
algorithmic bytes per token are that table's, every generator is seeded and
replica-specific, and the distributions are the stated ones (finite Zipf(1.1)
token ids, planted repeated 4-token spans, packed samples with image spans,
maps and histories onto [1, n_eids])."""
import numpy as np
import pytest

import workloads as W


@pytest.mark.parametrize("name,T,H,D,rows,bytes_tok", [
    ("tiny_fp8_d256", 256, 2, 256, 4096, 5_680),
    ("mid_prefill_fp8", 16_384, 4, 4096, 1_000_000, 114_784),
    ("decode_fp8", 512, 4, 4096, 5_040_000, 114_784),
    ("full_prefill_fp8", 65_536, 8, 4096, 5_040_000, 164_032),
    ("bf16_tables", 32_768, 4, 4096, 5_040_000, 163_888),
])
def test_configs_match_the_contract(name, T, H, D, rows, bytes_tok):
    cfg = W.by_name(name)
    assert (cfg.T, cfg.H, cfg.D, cfg.rows) == (T, H, D, (rows,) * 3)
    assert cfg.algorithmic_bytes_per_token() == bytes_tok


def test_generators_are_seeded_and_per_replica():
    cfg = W.by_name("full_prefill_fp8").scaled(B=2, S=1024)
    a, b = W.token_ids(cfg, 0), W.token_ids(cfg, 0)
    assert np.array_equal(a, b)
    assert not np.array_equal(a, W.token_ids(cfg, 1))
    assert np.array_equal(W.tid2eid(cfg), W.tid2eid(cfg))
    dec = W.by_name("decode_fp8").scaled(B=64)
    assert np.array_equal(W.history(dec, 0), W.history(dec, 0))
    assert not np.array_equal(W.history(dec, 0), W.history(dec, 1))


def test_maps_and_histories_stay_off_the_pad_id():
    cfg = W.by_name("mid_prefill_fp8")
    m = W.tid2eid(cfg)
    assert m.shape == (cfg.vocab,) and m.min() >= 1 and m.max() <= cfg.n_eids
    h = W.history(W.by_name("decode_fp8"))
    assert h.shape == (512, 3) and h.min() >= 1 and h.max() <= 100_000


def test_zipf_token_ids_follow_their_law():
    """Finite Zipf(1.1) over 129,280 ranks: token 0 (rank 1) and token 9 (rank 10)
    appear with the law's probabilities, within five standard deviations."""
    cfg = W.by_name("mid_prefill_fp8")
    ids = W.token_ids(cfg).ravel()
    assert ids.min() >= 0 and ids.max() < cfg.vocab
    k = np.arange(1, cfg.vocab + 1, dtype=np.float64)
    p = k ** -1.1 / np.sum(k ** -1.1)
    n = ids.size
    for tok in (0, 9):
        want = p[tok] * n
        got = np.count_nonzero(ids == tok)
        assert abs(got - want) < 5 * np.sqrt(want * (1 - p[tok])), (tok, got, want)


def test_planted_repeats():
    """The full-size prefill plants round(0.05 * 8192 / 4) = 102 earlier 4-token
    spans per sequence at non-overlapping 4-aligned destinations; each
    destination holds its source's ids."""
    cfg = W.by_name("full_prefill_fp8").scaled(B=2)
    g = W.rng(cfg, 99, 0)
    ids = g.integers(0, 1000, size=(cfg.B, cfg.S)).astype(np.int32)
    planted = W.plant_repeats(ids, cfg.repeat_frac, W.rng(cfg, 98, 0))
    assert len(planted) == 2 * 102
    for b in range(cfg.B):
        dsts = sorted(d for bb, _, d in planted if bb == b)
        assert all(d % 4 == 0 for d in dsts) and all(y - x >= 4 for x, y in zip(dsts, dsts[1:]))
    for b, src, dst in planted:
        assert 0 <= src and src + 4 <= dst
        assert np.array_equal(ids[b, dst:dst + 4], ids[b, src:src + 4])


def test_packed_layout():
    """Samples of U[L/2, 3L/2] tokens (the last one cut at the row's end) whose
    positions count from 0; image spans of exactly image_span dead positions
    inside one sample; about image_frac of the positions dead."""
    cfg = W.by_name("packed_mm_fp8")
    pos, dead = W.packed_layout(cfg)
    assert pos.shape == dead.shape == (cfg.B, cfg.S)
    L, span = cfg.mean_sample_len, cfg.image_span
    for b in range(cfg.B):
        starts = np.flatnonzero(pos[b] == 0)
        assert starts[0] == 0
        ends = np.append(starts[1:], cfg.S)
        for s0, s1 in zip(starts, ends):
            n = s1 - s0
            assert np.array_equal(pos[b, s0:s1], np.arange(n))
            if s1 < cfg.S:
                assert L // 2 <= n <= L + L // 2
            d = dead[b, s0:s1]
            assert d.sum() in (0, span)
            if d.sum():
                first = int(np.flatnonzero(d)[0])
                assert d[first:first + span].all()
    frac = dead.mean()
    assert 0.15 < frac < 0.3, frac
    plain_pos, plain_dead = W.packed_layout(W.by_name("full_prefill_fp8").scaled(B=2, S=64))
    assert np.array_equal(plain_pos[1], np.arange(64)) and not plain_dead.any()


def test_rows_layout_holds_the_blocks_layout_values():
    """The rows-with-exponents workload draws the same bytes and exponents as the
    blocks layout and stores each row, then its exponents, then zeros; its
    algorithmic bytes per token are the same (the padding is not counted)."""
    e8 = W.by_name("release_layout_fp8").scaled(rows=(500,) * 3, hash_vocab=10)
    rw = W.by_name("release_layout_fp8_rows").scaled(rows=(500,) * 3, hash_vocab=10)
    (t,), (e,) = [x[:1] for x in W.tables_host(e8)]
    (p,), _ = [x[:1] for x in W.tables_host(rw)]
    D = rw.D
    assert rw.stored_row_bytes() == 272 and p.shape == (500, 272)
    assert np.array_equal(p[:, :D], t) and np.array_equal(p[:, D:D + D // 32], e)
    assert not p[:, D + D // 32:].any()
    assert rw.algorithmic_bytes_per_token() == e8.algorithmic_bytes_per_token()
    assert W.by_name("release_layout_fp8_rows").table_bytes() == 384_006_168 * 272
