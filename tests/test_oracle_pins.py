"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Every function of the oracle is checked here against published values, library
routines it does not call, closed forms, invariants the pages state, or brute
force, so that a dropped term, a wrong index or sign, or a transposed operand
fails at least one test:

* splitmix64 -- the published output sequence for seed 1234567;
* the n-gram fold -- run backwards from its output with the modular inverse of
  the multiplier and the inverse xorshift, it must land on the published seed;
* window extents and alignment -- changing one id changes exactly the 2/3/4-gram
  rows whose windows contain it;
* pad before the start, history, decode = prefill (VeOmni PR page, commits on
  the n-gram lookup and its incremental decode cache);
* e4m3fn decode -- all 256 bytes against torch's float8_e4m3fn cast and the OCP
  table of special values;
* bf16 rounding -- torch's float32 -> bfloat16 cast, ties, and single rounding
  from fp64;
* gather / mean / gate / add -- closed forms (constant rows, orthogonal and
  parallel stream 0, eps placement) and NumPy restatements of special cases.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
M64 = (1 << 64) - 1
FOLD = 0x9E3779B97F4A7C15


# ----------------------------------------------------------------- splitmix64

def _read_splitmix_golden():
    seed, outs = None, []
    with open(os.path.join(GOLDEN, "splitmix64_seed1234567.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("seed"):
                seed = int(line.split()[1])
            else:
                outs.append(int(line))
    return seed, outs


def test_splitmix64_published_sequence():
    seed, outs = _read_splitmix_golden()
    assert len(outs) == 5
    # The k-th output of a generator started at `seed` is the first output of
    # one started at seed + k * increment.
    got = [oracle.splitmix64((seed + k * 0x9E3779B97F4A7C15) & M64) for k in range(5)]
    assert got == outs


def test_seeds_are_splitmix_of_n16_plus_j():
    for n in (2, 3, 4):
        for j in range(8):
            assert oracle.seed(n, j) == oracle.splitmix64(n * 16 + j)
    seeds = {oracle.seed(n, j) for n in (2, 3, 4) for j in range(16)}
    assert len(seeds) == 48


# ----------------------------------------------------------------- the n-gram fold

def _unxorshift(h, k):
    """Inverse of h ^= h >> k on 64-bit words."""
    x = h
    for _ in range(64 // k + 1):
        x = h ^ (x >> k)
    return x & M64


def _unfold(h, window):
    inv = pow(FOLD, -1, 1 << 64)
    for e in reversed(window):
        h = _unxorshift(h, 29)
        h = (h * inv) & M64
        h ^= e
    return h


@pytest.mark.parametrize("n", [2, 3, 4])
def test_fold_inverts_to_seed(n):
    g = np.random.default_rng(11)
    for trial in range(200):
        window = [int(v) for v in g.integers(0, 2**31 - 1, size=n)]
        j = int(g.integers(0, 8))
        h = oracle.ngram_hash(window, n, j)
        assert _unfold(h, window) == oracle.seed(n, j)


def test_fold_is_order_sensitive_and_zero_extends():
    assert oracle.ngram_hash([1, 2], 2, 0) != oracle.ngram_hash([2, 1], 2, 0)
    # A large non-negative id must be zero-extended (no sign smear into the top word).
    big = 2**31 - 1
    h = oracle.ngram_hash([big, 0], 2, 0)
    assert _unfold(h, [big, 0]) == oracle.seed(2, 0)


def test_row_is_hash_mod_rows():
    g = np.random.default_rng(5)
    eids = g.integers(1, 1000, size=(1, 40)).astype(np.int32)
    for rows in ([1, 1, 1], [7, 4096, 2**31 - 1], [2**20, 3, 5_040_000]):
        ids, flags = oracle.hash_ids(eids, 3, rows)
        assert flags == 0
        if rows == [1, 1, 1]:
            assert (ids == 0).all()
        for s in range(40):
            w = [0] * 3 + list(eids[0])
            for n in (2, 3, 4):
                window = w[s + 4 - n: s + 4]
                for j in range(3):
                    assert ids[0, s, n - 2, j] == oracle.ngram_hash(window, n, j) % rows[n - 2]


# ----------------------------------------------------------------- windows

BIG_ROWS = [2**31 - 1, 2**31 - 19, 2**31 - 61]   # collisions mod rows ~1e-9


def test_window_extent_per_order():
    """Changing the id at p changes the n-gram rows at p .. p+n-1 and nothing else."""
    g = np.random.default_rng(3)
    S = 48
    eids = g.integers(1, 100_000, size=(1, S)).astype(np.int32)
    base, _ = oracle.hash_ids(eids, 4, BIG_ROWS)
    for p in (0, 1, 5, 20, S - 1):
        e2 = eids.copy()
        e2[0, p] += 1
        new, _ = oracle.hash_ids(e2, 4, BIG_ROWS)
        for n in (2, 3, 4):
            changed = (new[0, :, n - 2, :] != base[0, :, n - 2, :]).any(axis=1)
            expect = np.zeros(S, bool)
            expect[p:min(S, p + n)] = True
            assert (changed == expect).all(), (p, n)


def test_pad_before_start_equals_zero_history():
    """Blocked lookback and pad compress to the same id 0 (VeOmni PR page)."""
    g = np.random.default_rng(4)
    eids = g.integers(1, 100_000, size=(3, 9)).astype(np.int32)
    a, _ = oracle.hash_ids(eids, 2, BIG_ROWS)
    b, _ = oracle.hash_ids(eids, 2, BIG_ROWS, history=np.zeros((3, 3), np.int32))
    assert (a == b).all()


def test_history_reaches_only_first_three_positions():
    g = np.random.default_rng(6)
    eids = g.integers(1, 100_000, size=(2, 10)).astype(np.int32)
    a, _ = oracle.hash_ids(eids, 2, BIG_ROWS)
    hist = g.integers(1, 100_000, size=(2, 3)).astype(np.int32)
    b, _ = oracle.hash_ids(eids, 2, BIG_ROWS, history=hist)
    # position s reaches back n-1 ids: s=0 all orders, s=1 orders 3,4, s=2 order 4.
    for s in range(10):
        for n in (2, 3, 4):
            differs = (a[:, s, n - 2] != b[:, s, n - 2]).all()
            same = (a[:, s, n - 2] == b[:, s, n - 2]).all()
            if s - n + 1 < 0:
                assert differs, (s, n)
            else:
                assert same, (s, n)


def test_decode_steps_equal_prefill():
    """Hash ids are integers: token-by-token decode with a three-id history must
    equal the prefill bit for bit, at every split point (VeOmni PR page, the
    incremental decode cache commit)."""
    g = np.random.default_rng(7)
    B, S = 3, 23
    eids = g.integers(1, 100_000, size=(B, S)).astype(np.int32)
    full, hfull, _ = oracle.hash_ids(eids, 4, BIG_ROWS, want_history=True)
    for split in (0, 1, 2, 3, 11):
        ids, hist, _ = oracle.hash_ids(eids[:, :split], 4, BIG_ROWS, want_history=True)
        got = [ids]
        for s in range(split, S):
            step, hist, _ = oracle.hash_ids(eids[:, s:s + 1], 4, BIG_ROWS, history=hist,
                                            want_history=True)
            got.append(step)
        assert (np.concatenate(got, axis=1) == full).all(), split
        assert (hist == hfull).all()
    assert (hfull == eids[:, -3:]).all()


def test_history_out_short_sequences_and_aliasing_safe():
    hist = np.array([[5, 6, 7]], np.int32)
    _, h1, _ = oracle.hash_ids(np.array([[9]], np.int32), 1, BIG_ROWS, history=hist,
                               want_history=True)
    assert h1.tolist() == [[6, 7, 9]]
    _, h2, _ = oracle.hash_ids(np.array([[9, 10]], np.int32), 1, BIG_ROWS, history=hist,
                               want_history=True)
    assert h2.tolist() == [[7, 9, 10]]
    _, h0, _ = oracle.hash_ids(np.array([[9]], np.int32), 1, BIG_ROWS, want_history=True)
    assert h0.tolist() == [[0, 0, 9]]
    _, he, _ = oracle.hash_ids(np.zeros((1, 0), np.int32), 1, BIG_ROWS, history=hist,
                               want_history=True)
    assert he.tolist() == [[5, 6, 7]]


def test_identical_windows_identical_rows_on_planted_repeats():
    cfg = W.by_name("full_prefill_fp8").scaled(B=2, S=512)
    ids = W.token_ids(cfg)
    planted = W.plant_repeats(ids.copy(), cfg.repeat_frac, W.rng(cfg, 7, 0))
    assert len(planted) == 2 * round(0.05 * 512 / 4)
    eids, flags = oracle.compress(ids, W.tid2eid(cfg), cfg.n_eids)
    assert flags == 0
    rows, _ = oracle.hash_ids(eids, cfg.H, cfg.rows)
    for b, src, dst in planted:
        # the 4-gram ending at the span's last id, 3-grams at its last two, 2-grams at its last three
        for n in (2, 3, 4):
            for k in range(n - 1, 4):
                assert (rows[b, dst + k, n - 2] == rows[b, src + k, n - 2]).all()


def test_brute_force_python_ints_tiny():
    """Cross-check of the C oracle against an independent Python-int restatement
    on every window of a tiny input (exact 64-bit arithmetic by masking)."""
    def sm(x):
        z = (x + 0x9E3779B97F4A7C15) & M64
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
        return z ^ (z >> 31)
    g = np.random.default_rng(9)
    B, S, H = 2, 8, 3
    rows = [17, 13, 11]
    eids = g.integers(0, 40, size=(B, S)).astype(np.int32)
    hist = g.integers(0, 40, size=(B, 3)).astype(np.int32)
    for hh in (None, hist):
        got, _ = oracle.hash_ids(eids, H, rows, history=hh)
        for b in range(B):
            pre = [0, 0, 0] if hh is None else list(hh[b])
            seq = pre + list(eids[b])
            for s in range(S):
                for n in (2, 3, 4):
                    for j in range(H):
                        h = sm(n * 16 + j)
                        for e in seq[s + 3 - n + 1: s + 4]:
                            h = ((h ^ int(e)) * FOLD) & M64
                            h ^= h >> 29
                        assert got[b, s, n - 2, j] == h % rows[n - 2]


def test_hash_flags_negative_eids_and_skips_token():
    eids = np.array([[3, 4, -2, 5, 6, 7, 8]], np.int32)   # -1 is the dead marker, -2 invalid
    ids, flags = oracle.hash_ids(eids, 1, [101, 103, 107], fill=-7)
    assert flags == oracle.BAD_EID
    # windows s-3..s containing position 2: s = 2..5 are skipped
    for s in range(7):
        skipped = (ids[0, s] == -7).all()
        assert skipped == (2 <= s <= 5), s


# ----------------------------------------------------------------- compress

def test_compress_gather_and_range_flags():
    m = np.array([0, 5, 9, 2, 11], np.int32)
    out, flags = oracle.compress(np.array([1, 2, 3, 0, 4], np.int32), m, n_eids=10)
    assert out.tolist() == [5, 9, 2, 0, -7] and flags == oracle.BAD_EID
    out, flags = oracle.compress(np.array([1, 5, -1], np.int32), m, n_eids=20)
    assert out.tolist() == [5, -7, -7] and flags == oracle.BAD_TOKEN
    ident = np.arange(100, dtype=np.int32)
    tid = np.random.default_rng(1).integers(0, 100, 57).astype(np.int32)
    out, flags = oracle.compress(tid, ident, n_eids=99)
    assert flags == 0 and (out == tid).all()


# ----------------------------------------------------------------- e4m3fn decode

def test_e4m3fn_all_bytes_match_torch_cast():
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    for b in range(256):
        v = oracle.e4m3fn_decode(b)
        if math.isnan(ref[b]):
            assert math.isnan(v), b
        else:
            assert v == float(ref[b]) and math.copysign(1, v) == math.copysign(1, ref[b]), b


def test_e4m3fn_ocp_special_values():
    with open(os.path.join(GOLDEN, "e4m3fn_ocp.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            b, v = line.split()
            got = oracle.e4m3fn_decode(int(b, 16))
            if v == "nan":
                assert math.isnan(got)
            else:
                assert got == float(v), b


# ----------------------------------------------------------------- bf16 rounding

def test_bf16_round_matches_torch_on_float32_inputs():
    g = np.random.default_rng(2)
    x = np.concatenate([
        g.standard_normal(20000).astype(np.float32),
        (g.standard_normal(5000) * 1e30).astype(np.float32),
        (g.standard_normal(5000) * 1e-39).astype(np.float32),   # bf16 subnormals
        np.array([3.3895314e38, -3.3895314e38, 3.4e38, 1e-45, 0.0, -0.0], np.float32),
    ])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_round(float(v)) for v in x], np.uint16)
    assert (got == ref).all()


def test_bf16_round_ties_even_and_single_rounding():
    one = 0x3F80
    assert oracle.bf16_round(1.0 + 2**-8) == one                 # tie -> even (down)
    assert oracle.bf16_round(1.0 + 3 * 2**-8) == one + 2         # tie -> even (up)
    # Single rounding from fp64: a value just above a tie must round up, although a
    # detour through float32 would land exactly on the tie and round to even.
    assert oracle.bf16_round(1.0 + 2**-8 + 2**-40) == one + 1
    assert oracle.bf16_round(-(1.0 + 2**-8 + 2**-40)) == 0x8000 | (one + 1)
    assert oracle.bf16_round(2.0**128) == 0x7F80
    assert oracle.bf16_round(-0.0) == 0x8000
    for bits in (0x0001, 0x3F81, 0x7F7F, 0xC2F7, 0x8001):
        assert oracle.bf16_round(oracle.bf16_decode(bits)) == bits


# ----------------------------------------------------------------- lookup closed forms

def _const_tables(D, rows, bytes_per_table, dtype=oracle.FP8):
    tabs = [np.full((rows, D), b, np.uint8) for b in bytes_per_table]
    return tabs


def _dec(b):
    return oracle.e4m3fn_decode(b)


def test_mean_is_equal_weight_over_3h_rows():
    """Constant tables c_n with constant scales s_n: m = (c2 s2 + c3 s3 + c4 s4) / 3
    for every token, whatever the row ids and H."""
    D, rows, T = 32, 50, 7
    g = np.random.default_rng(1)
    bytes_ = [0x38, 0x40, 0xB4]      # 1.0, 2.0, -0.75
    sc = [0.5, 0.25, 2.0]
    for H in (1, 2, 5):
        tabs = _const_tables(D, rows, bytes_)
        scales = [np.full(rows, s, np.float32) for s in sc]
        ids = g.integers(0, rows, size=(T, 3 * H)).astype(np.int32)
        x = W._to_bf16_bits(g.standard_normal((T, 4, D)).astype(np.float32))
        y, gate, m, flags = oracle.lookup(ids, H, oracle.FP8, tabs, scales, x, np.zeros(4, np.float32),
                                          1e-6, aux=True)
        assert flags == 0
        expect = sum(_dec(b) * s for b, s in zip(bytes_, sc)) / 3.0
        assert np.all(m == expect)


def test_gate_half_when_stream0_orthogonal_to_m():
    """sum(a*m) = 0 exactly gives g = 1/2, so out_s = x_s + alpha_s * m / 2."""
    D, rows, T, H = 16, 8, 3, 2
    tabs = _const_tables(D, rows, [0x38, 0x38, 0x38])          # m = 1.0 everywhere
    scales = [np.ones(rows, np.float32)] * 3
    ids = np.zeros((T, 3 * H), np.int32)
    a = np.tile(np.array([1.5, -1.5], np.float32), D // 2)       # sums to 0 exactly
    g = np.random.default_rng(3)
    x = g.standard_normal((T, 4, D)).astype(np.float32)
    x[:, 0, :] = a
    xb = W._to_bf16_bits(x)
    alpha = np.array([0.5, -2.0, 0.25, 4.0], np.float32)
    y, gate, m, flags = oracle.lookup(ids, H, oracle.FP8, tabs, scales, xb, alpha, 1e-6, aux=True)
    assert flags == 0 and np.all(gate == 0.5) and np.all(m == 1.0)
    xf = oracle.bf16_bits_to_float(xb)
    ref = torch.from_numpy((xf + 0.5 * alpha[None, :, None] * 1.0).astype(np.float32)).to(
        torch.bfloat16).view(torch.int16).numpy().view(np.uint16)   # exact sums in float32
    assert (y == ref).all()


@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_gate_is_sigmoid_sqrt_d_for_parallel_stream0(sign):
    """Stream 0 constant k and m constant c with eps = 0: the normalised dot product
    is sign(kc) * sqrt(D), so g = sigmoid(+-sqrt(D)).  With eps = 1/4 and k = c = 1:
    logit = D / (1.25 * sqrt(D))."""
    D, rows, T, H = 16, 4, 2, 1
    tabs = _const_tables(D, rows, [0x38] * 3)                    # c = 1
    scales = [np.ones(rows, np.float32)] * 3
    ids = np.zeros((T, 3), np.int32)
    x = np.zeros((T, 4, D), np.float32)
    x[:, 0, :] = 3.0 * sign
    xb = W._to_bf16_bits(x)
    _, gate, _, _ = oracle.lookup(ids, H, oracle.FP8, tabs, scales, xb, np.ones(4, np.float32), 0.0,
                                  aux=True)
    assert np.allclose(gate, 1.0 / (1.0 + math.exp(-sign * 4.0)), rtol=0, atol=1e-15)
    x[:, 0, :] = 1.0
    _, gate, _, _ = oracle.lookup(ids, H, oracle.FP8, tabs, scales, W._to_bf16_bits(x),
                                  np.ones(4, np.float32), 0.25, aux=True)
    logit = D / (1.25 * math.sqrt(D))
    assert np.allclose(gate, 1.0 / (1.0 + math.exp(-logit)), rtol=0, atol=1e-15)


def _random_case(dtype, T=9, H=3, D=48, rows=(31, 37, 41), seed=0):
    g = np.random.default_rng(seed)
    if dtype == oracle.FP8:
        tabs = [W._to_e4m3_bytes(g.standard_normal((r, D)).astype(np.float32) * 8) for r in rows]
        scales = [g.uniform(1e-3, 1e-2, r).astype(np.float32) for r in rows]
    else:
        tabs = [W._to_bf16_bits(g.standard_normal((r, D)).astype(np.float32) * 0.02) for r in rows]
        scales = None
    ids = np.stack([g.integers(0, rows[r // H], size=T) for r in range(3 * H)], 1).astype(np.int32)
    x = W._to_bf16_bits(g.standard_normal((T, 4, D)).astype(np.float32))
    alpha = g.standard_normal(4).astype(np.float32)
    return tabs, scales, ids, x, alpha


@pytest.mark.parametrize("dtype", [oracle.FP8, oracle.BF16])
def test_gather_mean_matches_torch_decode(dtype):
    """m = mean over r of decode(table[n_r][row_r]) * scale[n_r][row_r], with the
    decode done by torch's casts and the gather by NumPy indexing."""
    H = 3
    tabs, scales, ids, x, alpha = _random_case(dtype, H=H)
    _, _, m, flags = oracle.lookup(ids, H, dtype, tabs, scales, x, alpha, 1e-6, aux=True)
    assert flags == 0
    acc = np.zeros(m.shape)
    for r in range(3 * H):
        n = r // H
        if dtype == oracle.FP8:
            dec = torch.from_numpy(tabs[n]).view(torch.float8_e4m3fn).double().numpy()
            acc += dec[ids[:, r]] * scales[n][ids[:, r]].astype(np.float64)[:, None]
        else:
            dec = torch.from_numpy(tabs[n].view(np.int16)).view(torch.bfloat16).double().numpy()
            acc += dec[ids[:, r]]
    assert np.allclose(m, acc / (3 * H), rtol=1e-14, atol=1e-18)


@pytest.mark.parametrize("dtype", [oracle.FP8, oracle.BF16])
def test_gate_is_sigmoid_of_scaled_cosine_when_eps_zero(dtype):
    tabs, scales, ids, x, alpha = _random_case(dtype, seed=4)
    _, gate, m, _ = oracle.lookup(ids, 3, dtype, tabs, scales, x, alpha, 0.0, aux=True)
    a = oracle.bf16_bits_to_float(x[:, 0, :]).astype(np.float64)
    D = a.shape[1]
    cos = np.einsum("td,td->t", a, m) / (np.linalg.norm(a, axis=1) * np.linalg.norm(m, axis=1))
    assert np.allclose(gate, 1.0 / (1.0 + np.exp(-cos * math.sqrt(D))), rtol=1e-13, atol=0)


@pytest.mark.parametrize("dtype", [oracle.FP8, oracle.BF16])
def test_output_is_once_rounded_gated_add(dtype):
    """out_s = round_bf16(x_s + g alpha_s m) for all four streams, checked with
    torch's cast where the fp64 sum is exactly a float32 (almost always a
    float32 here; the rest may differ from torch's cast by the double rounding
    of float32 -> bf16 only)."""
    tabs, scales, ids, x, alpha = _random_case(dtype, seed=8, D=64)
    y, gate, m, _ = oracle.lookup(ids, 3, dtype, tabs, scales, x, alpha, 1e-6, aux=True)
    xf = oracle.bf16_bits_to_float(x).astype(np.float64)
    exact = xf + gate[:, None, None] * alpha.astype(np.float64)[None, :, None] * m[:, None, :]
    as32 = exact.astype(np.float32)
    ref = torch.from_numpy(as32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    representable = as32.astype(np.float64) == exact
    assert (y[representable] == ref[representable]).all()
    yf = oracle.bf16_bits_to_float(y).astype(np.float64)
    ulp = np.ldexp(1.0, np.frexp(np.abs(exact))[1] - 8)
    assert np.all(np.abs(yf - exact) <= 0.5 * ulp + 1e-300)


def test_zero_alpha_or_zero_rows_leave_streams_unchanged():
    tabs, scales, ids, x, alpha = _random_case(oracle.FP8, seed=2)
    assert not (x == 0x8000).any()          # IEEE: -0 + +0 would be +0
    y, _ = oracle.lookup(ids, 3, oracle.FP8, tabs, scales, x, np.zeros(4, np.float32), 1e-6)
    assert (y == x).all()
    zt = [np.zeros_like(t) for t in tabs]
    y, _ = oracle.lookup(ids, 3, oracle.FP8, zt, scales, x, alpha, 1e-6)
    assert (y == x).all()


def test_lookup_flags_bad_rows_and_leaves_token_unwritten():
    tabs, scales, ids, x, alpha = _random_case(oracle.FP8, seed=3)
    ids = ids.copy()
    ids[2, 4] = 37          # table n=3 (r // H = 1) has 37 rows: 37 is out of range
    ids[5, 0] = -1
    y, flags = oracle.lookup(ids, 3, oracle.FP8, tabs, scales, x, alpha, 1e-6, fill=0x1234)
    assert flags == oracle.BAD_ROW
    for t in range(ids.shape[0]):
        assert (y[t] == 0x1234).all() == (t in (2, 5))


def test_lookup_in_place_equals_out_of_place():
    tabs, scales, ids, x, alpha = _random_case(oracle.BF16, seed=5)
    y, _ = oracle.lookup(ids, 3, oracle.BF16, tabs, scales, x, alpha, 1e-6)
    import ctypes as C
    xx = x.copy()
    tp = (C.c_void_p * 3)(*[t.ctypes.data for t in tabs])
    sp = (C.c_void_p * 3)(None, None, None)
    r = (C.c_int64 * 3)(*[t.shape[0] for t in tabs])
    oracle.lib().orc_lookup(ids.ctypes.data, ids.shape[0], 3, oracle.BF16, x.shape[-1], tp, sp, r,
                            xx.ctypes.data, alpha.ctypes.data, 1e-6, xx.ctypes.data, None, None)
    assert (xx == y).all()


# ----------------------------------------------------------------- dead positions, packed samples

def test_compress_masked_marks_dead_whatever_the_token():
    m = np.array([0, 5, 9, 2], np.int32)
    ids = np.array([1, -5, 2, 7, 3], np.int32)
    dead = np.array([0, 1, 0, 1, 0], np.uint8)
    out, flags = oracle.compress_masked(ids, m, 10, dead)
    assert flags == 0 and out.tolist() == [5, oracle.DEAD, 9, oracle.DEAD, 2]


def test_dead_token_blocks_lookback_like_a_sequence_start():
    """A blocked lookback and the pad before position 0 agree (VeOmni PR page,
    pack_ngram_inputs commit): the tokens after a dead one hash exactly like a
    fresh sequence, the tokens before it are untouched, the dead token itself has
    only dead rows."""
    g = np.random.default_rng(21)
    e = g.integers(1, 100_000, size=(1, 14)).astype(np.int32)
    p = 5
    ed = e.copy()
    ed[0, p] = oracle.DEAD
    plain, _ = oracle.hash_ids(e, 3, BIG_ROWS)
    got, flags = oracle.hash_ids(ed, 3, BIG_ROWS)
    assert flags == 0
    assert (got[0, :p] == plain[0, :p]).all()
    assert (got[0, p] == oracle.DEAD).all()
    fresh, _ = oracle.hash_ids(e[:, p + 1:], 3, BIG_ROWS)
    assert (got[0, p + 1:] == fresh[0]).all()


def test_packed_samples_hash_like_separate_sequences():
    """Positions restarting at 0 per packed sample keep every n-gram inside its
    sample (VeOmni PR page, review of pack_ngram_inputs)."""
    g = np.random.default_rng(22)
    lens = [5, 1, 9, 2]
    samples = [g.integers(1, 100_000, size=n).astype(np.int32) for n in lens]
    packed = np.concatenate(samples)[None, :]
    positions = np.concatenate([np.arange(n) for n in lens]).astype(np.int32)[None, :]
    got, flags = oracle.hash_ids(packed, 2, BIG_ROWS, positions=positions)
    assert flags == 0
    parts = [oracle.hash_ids(smp[None, :], 2, BIG_ROWS)[0][0] for smp in samples]
    assert (got[0] == np.concatenate(parts)).all()
    # positions equal to the index reproduce the plain hash
    same, _ = oracle.hash_ids(packed, 2, BIG_ROWS, positions=np.arange(17, dtype=np.int32)[None, :])
    plain, _ = oracle.hash_ids(packed, 2, BIG_ROWS)
    assert (same == plain).all()


@pytest.mark.parametrize("pos", [0, 1, 2, 3, 50])
def test_decode_start_position_bounds_the_history(pos):
    """The history sets how far back the walk can read, the start position whether
    it reached the true start (VeOmni PR page, decode cache commit): a step at
    position p hashes like the last token of the p+1-token sequence whose first
    ids are the history tail."""
    hist = np.array([[11, 22, 33]], np.int32)
    tok = np.array([[44]], np.int32)
    got, _ = oracle.hash_ids(tok, 2, BIG_ROWS, history=hist, positions=np.array([[pos]], np.int32))
    seq = np.concatenate([hist[0, 3 - min(pos, 3):], tok[0]])[None, :]
    ref, _ = oracle.hash_ids(seq, 2, BIG_ROWS)
    assert (got[0, 0] == ref[0, -1]).all()


def test_dead_history_entry_blocks_and_is_carried():
    hist = np.array([[11, oracle.DEAD, 33]], np.int32)
    tok = np.array([[44, 55]], np.int32)
    got, hout, _ = oracle.hash_ids(tok, 2, BIG_ROWS, history=hist, want_history=True)
    ref, _ = oracle.hash_ids(np.array([[33, 44, 55]], np.int32), 2, BIG_ROWS)
    assert (got[0] == ref[0, 1:]).all()
    assert hout.tolist() == [[33, 44, 55]]
    _, hout2, _ = oracle.hash_ids(np.array([[oracle.DEAD]], np.int32), 2, BIG_ROWS, history=hist,
                                  want_history=True)
    assert hout2.tolist() == [[oracle.DEAD, 33, oracle.DEAD]]


def test_dead_tokens_pass_through_with_zero_gate():
    """A dead token's gate is zeroed (vLLM page, DeepseekV4Model.forward): its
    streams come out bit for bit, g = 0, m = 0; a token with some dead and some
    live row ids is a bad row."""
    tabs, scales, ids, x, alpha = _random_case(oracle.FP8, seed=11)
    ids = ids.copy()
    ids[3] = oracle.DEAD
    ids[6, 2] = oracle.DEAD
    y, gate, m, flags = oracle.lookup(ids, 3, oracle.FP8, tabs, scales, x, alpha, 1e-6, aux=True,
                                      fill=0x1234)
    assert flags == oracle.BAD_ROW
    assert (y[3] == x[3]).all() and gate[3] == 0 and (m[3] == 0).all()
    assert (y[6] == 0x1234).all()
    live = [t for t in range(ids.shape[0]) if t not in (3, 6)]
    y2, _ = oracle.lookup(ids[live], 3, oracle.FP8, tabs, scales, x[live], alpha, 1e-6)
    assert (y[live] == y2).all()


# ----------------------------------------------------------------- e8m0 block scales

def test_e8m0_all_bytes_match_torch_cast():
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e8m0fnu).double().numpy()
    for e in range(256):
        v = oracle.e8m0_decode(e)
        assert (math.isnan(v) and math.isnan(ref[e])) or v == ref[e], e


def test_e8m0_ocp_mx_values():
    with open(os.path.join(GOLDEN, "e8m0_ocp_mx.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            b, v = line.split()
            got = oracle.e8m0_decode(int(b, 16))
            assert math.isnan(got) if v == "nan" else got == float(v), b


def test_e8m0_blocks_gather_matches_torch_decode():
    """m = mean over r of decode(row) * 2^(e - 127), each column with its own
    32-column block's exponent, decoded by torch's casts."""
    g = np.random.default_rng(12)
    H, D, rows, T = 2, 96, (19, 23, 29), 11
    tabs = [W._to_e4m3_bytes(g.standard_normal((r, D)).astype(np.float32) * 4) for r in rows]
    scs = [g.integers(110, 140, size=(r, D // 32)).astype(np.uint8) for r in rows]
    ids = np.stack([g.integers(0, rows[r // H], size=T) for r in range(3 * H)], 1).astype(np.int32)
    x = W._to_bf16_bits(g.standard_normal((T, 4, D)).astype(np.float32))
    _, _, m, flags = oracle.lookup(ids, H, oracle.FP8_E8M0, tabs, scs, x, np.ones(4, np.float32),
                                   1e-6, aux=True)
    assert flags == 0
    acc = np.zeros((T, D))
    for r in range(3 * H):
        n = r // H
        dec = torch.from_numpy(tabs[n]).view(torch.float8_e4m3fn).double().numpy()[ids[:, r]]
        sc = torch.from_numpy(scs[n]).view(torch.float8_e8m0fnu).double().numpy()[ids[:, r]]
        acc += dec * np.repeat(sc, 32, axis=1)
    assert np.allclose(m, acc / (3 * H), rtol=1e-15, atol=0)


def test_e8m0_uniform_blocks_equal_row_scales():
    """Every block of a row sharing exponent e gives the per-row-scale result with
    scale 2^(e - 127), bit for bit."""
    tabs, _, ids, x, alpha = _random_case(oracle.FP8, seed=13, D=64)
    g = np.random.default_rng(13)
    e_rows = [g.integers(115, 125, size=t.shape[0]).astype(np.uint8) for t in tabs]
    blocks = [np.repeat(e[:, None], 2, axis=1) for e in e_rows]
    rows_scale = [np.ldexp(1.0, e.astype(np.int64) - 127).astype(np.float32) for e in e_rows]
    y1, g1, m1, _ = oracle.lookup(ids, 3, oracle.FP8_E8M0, tabs, blocks, x, alpha, 1e-6, aux=True)
    y2, g2, m2, _ = oracle.lookup(ids, 3, oracle.FP8, tabs, rows_scale, x, alpha, 1e-6, aux=True)
    assert (y1 == y2).all() and (g1 == g2).all() and (m1 == m2).all()


# ----------------------------------------------------------------- prime buckets

def _bucket_golden():
    out = []
    with open(os.path.join(GOLDEN, "bucket_layout_pages.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            left, right = line.split(":")
            out.append(([int(v) for v in left.split()], [int(v) for v in right.split()]))
    return out


def test_bucket_primes_reproduce_the_pages_row_counts():
    for (layers, max_n, heads, vocab), sums in _bucket_golden():
        primes = oracle.bucket_primes(layers, max_n, heads, vocab)
        assert primes.sum(axis=(1, 2)).tolist() == sums


def test_bucket_primes_are_distinct_primes_above_the_vocab():
    sympy = pytest.importorskip("sympy")
    primes = oracle.bucket_primes(2, 4, 8, 16_000_000)
    flat = primes.reshape(-1).tolist()
    assert len(set(flat)) == len(flat) and min(flat) >= 16_000_000
    assert all(sympy.isprime(int(p)) for p in flat)
    # each order starts again from the vocabulary: the first head of every order
    # of layer 0 takes the smallest prime not yet used
    assert flat[0] == sympy.nextprime(16_000_000 - 1)


def test_bucketed_rows_land_in_their_bucket_at_h_mod_p():
    """row = offset_r + (h mod p_r), offsets the running sum of the buckets in
    draw order; h from an independent Python-int restatement of the fold."""
    def sm(x):
        z = (x + 0x9E3779B97F4A7C15) & M64
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
        return z ^ (z >> 31)
    H = 3
    primes = oracle.bucket_primes(1, 4, H, 1000)[0]           # [3, H]
    offsets = np.concatenate([[0], np.cumsum(primes.reshape(-1))[:-1]]).reshape(3, H)
    g = np.random.default_rng(40)
    eids = g.integers(1, 5000, size=(2, 9)).astype(np.int32)
    got, flags = oracle.hash_bucketed(eids, H, primes)
    assert flags == 0
    for b in range(2):
        seq = [0, 0, 0] + [int(v) for v in eids[b]]
        for s in range(9):
            for n in (2, 3, 4):
                for j in range(H):
                    h = sm(n * 16 + j)
                    for e in seq[s + 4 - n: s + 4]:
                        h = ((h ^ e) * FOLD) & M64
                        h ^= h >> 29
                    assert got[b, s, n - 2, j] == offsets[n - 2, j] + h % int(primes[n - 2, j])


def test_bucketed_hash_keeps_dead_and_packed_rules():
    primes = oracle.bucket_primes(1, 4, 2, 10_000)[0]
    e = np.array([[5, 6, oracle.DEAD, 7, 8, 9]], np.int32)
    got, _ = oracle.hash_bucketed(e, 2, primes)
    assert (got[0, 2] == oracle.DEAD).all()
    fresh, _ = oracle.hash_bucketed(e[:, 3:], 2, primes)
    assert (got[0, 3:] == fresh[0]).all()


# ----------------------------------------------------------------- wkv connection

def _connection_case(seed, T=7, H=2, d=64, D=96, rows=(13, 17, 19), dtype=oracle.FP8_E8M0):
    g = np.random.default_rng(seed)
    if dtype == oracle.FP8_E8M0:
        tabs = [W._to_e4m3_bytes(g.standard_normal((r, d)).astype(np.float32) * 4) for r in rows]
        scs = [g.integers(118, 130, size=(r, d // 32)).astype(np.uint8) for r in rows]
    else:
        tabs = [W._to_bf16_bits(g.standard_normal((r, d)).astype(np.float32)) for r in rows]
        scs = None
    ids = np.stack([g.integers(0, rows[r // H], size=T) for r in range(3 * H)], 1).astype(np.int32)
    wkv = W._to_bf16_bits((g.standard_normal((D, 3 * H * d)) * 0.05).astype(np.float32))
    x = W._to_bf16_bits(g.standard_normal((T, 4, D)).astype(np.float32))
    alpha = g.standard_normal(4).astype(np.float32)
    return tabs, scs, ids, wkv, x, alpha


def _decoded_concat(tabs, scs, ids, H, dtype):
    parts = []
    for r in range(ids.shape[1]):
        n = r // H
        if dtype == oracle.FP8_E8M0:
            v = torch.from_numpy(tabs[n]).view(torch.float8_e4m3fn).double().numpy()[ids[:, r]]
            sc = torch.from_numpy(scs[n]).view(torch.float8_e8m0fnu).double().numpy()[ids[:, r]]
            parts.append(v * np.repeat(sc, 32, axis=1))
        else:
            parts.append(torch.from_numpy(tabs[n].view(np.int16)).view(torch.bfloat16).double()
                         .numpy()[ids[:, r]])
    return np.concatenate(parts, axis=1)


@pytest.mark.parametrize("dtype", [oracle.FP8_E8M0, oracle.BF16])
def test_connection_projection_matches_numpy_matmul(dtype):
    """k = wkv @ concat(rows), checked with torch's decodes and NumPy's matmul."""
    H = 2
    tabs, scs, ids, wkv, x, alpha = _connection_case(1, H=H, dtype=dtype)
    _, gate, k, flags = oracle.connection(ids, H, dtype, tabs, scs, wkv, x, alpha, 1e-6)
    assert flags == 0
    e = _decoded_concat(tabs, scs, ids, H, dtype)
    w = torch.from_numpy(wkv.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.allclose(k, e @ w.T, rtol=1e-12, atol=1e-12)
    a = oracle.bf16_bits_to_float(x[:, 0, :]).astype(np.float64)
    cos = np.einsum("td,td->t", a, k) / (np.linalg.norm(a, axis=1) * np.linalg.norm(k, axis=1))
    _, g0, _, _ = oracle.connection(ids, H, dtype, tabs, scs, wkv, x, alpha, 0.0)
    assert np.allclose(g0, 1 / (1 + np.exp(-cos * math.sqrt(a.shape[1]))), rtol=1e-12)


def test_connection_identity_weights_give_the_concatenated_rows():
    H, d = 1, 32
    tabs, scs, ids, _, _, alpha = _connection_case(2, H=H, d=d, D=3 * d)
    wkv = W._to_bf16_bits(np.eye(3 * d, dtype=np.float32))
    x = W._to_bf16_bits(np.random.default_rng(2).standard_normal((ids.shape[0], 4, 3 * d))
                        .astype(np.float32))
    _, _, k, _ = oracle.connection(ids, H, oracle.FP8_E8M0, tabs, scs, wkv, x, alpha, 1e-6)
    assert (k == _decoded_concat(tabs, scs, ids, H, oracle.FP8_E8M0)).all()


def test_connection_gate_half_and_dead_pass_through():
    H, d, D = 1, 32, 64
    tabs, scs, ids, wkv, x, alpha = _connection_case(3, H=H, d=d, D=D)
    # k constant over the columns (equal weight rows) and stream 0 summing to zero: g = 1/2
    wkv = np.tile(wkv[:1], (D, 1))
    xf = np.random.default_rng(3).standard_normal((ids.shape[0], 4, D)).astype(np.float32)
    xf[:, 0, :] = np.tile(np.array([0.75, -0.75], np.float32), D // 2)
    x = W._to_bf16_bits(xf)
    ids = ids.copy()
    ids[4] = oracle.DEAD
    y, gate, k, flags = oracle.connection(ids, H, oracle.FP8_E8M0, tabs, scs, wkv, x, alpha, 1e-6)
    assert flags == 0
    live = [t for t in range(ids.shape[0]) if t != 4]
    assert np.all(gate[live] == 0.5)
    assert (y[4] == x[4]).all() and gate[4] == 0
