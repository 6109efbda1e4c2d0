"""A worked example small enough to follow on paper: D = 16, H = 1, S = 3,
tables of 7 rows.  Every intermediate value of the path is written out below as
a literal, derived from the definitions (the splitmix64 seeds, the
xor-multiply-xorshift fold, h mod rows, the mean of the 3H dequantised rows,
the RMSNorm dot-product sigmoid gate, the once-rounded gated add), and the
oracle must reproduce each one.

Inputs (chosen so that the arithmetic stays exact where it can):
* vocabulary of 8 tokens, tid2eid = [5, 1, 4, 2, 7, 3, 2, 6] (eids 1..7; tokens
  3 and 6 both compress to eid 2), tokens [3, 1, 6];
* table n (n = 2, 3, 4), row r, column i holds the e4m3fn value
  ((r + i + n) mod 5 - 2) / 2, one of -1, -1/2, 0, 1/2, 1 (bytes 0xB8, 0xB0,
  0x00, 0x30, 0x38), with the fp32 row scale (r + 1) / 8;
* streams X[t, s, i] = (i - 8)/4 + s/2 - t/8 (exact in bf16);
* alpha = [1, -1/2, 2, 1/4], eps = 1e-6.
"""
from fractions import Fraction as F

import numpy as np
import pytest

import oracle

D, H, S, ROWS = 16, 1, 3, 7
TID2EID = np.array([5, 1, 4, 2, 7, 3, 2, 6], np.int32)
N_EIDS = 7
TOKENS = np.array([[3, 1, 6]], np.int32)
ALPHA = np.array([1.0, -0.5, 2.0, 0.25], np.float32)
EPS = 1e-6

# a1: compression
EIDS = [2, 1, 2]

# a3: seed(n, 0) = splitmix64(16 n), first output of the generator (state + the
# golden-ratio increment, then the two xor-shift-multiply rounds and a final
# xor-shift)
SEEDS = {2: 0xEAEB7F27B54E2401, 3: 0x040A2076F607FF23, 4: 0xD6967248FBE68CC3}

# a2 + a3: the window of each token and order (oldest first, pad 0 before the
# start), h after each fold h = (h ^ e) * 0x9E3779B97F4A7C15; h ^= h >> 29, and
# row = h mod 7
FOLDS = {
    (0, 2): ([0, 2], [0x1A08543F7061D1E8, 0xF6C2F320EB400908], 1),
    (0, 3): ([0, 0, 2], [0xA0E34A1E2C40B106, 0xF9EE57C3D3BBD35E, 0x721BA94285BDAC84], 1),
    (0, 4): ([0, 0, 0, 2], [0x51CBCE664D2B8CD9, 0x6236BF0FDB3051AB, 0xFD9D86813E1FB331,
                            0xF4D0EC9B2BA303CB], 4),
    (1, 2): ([2, 1], [0x567747B02D0255AB, 0xF276A44178667CC5], 3),
    (1, 3): ([0, 2, 1], [0xA0E34A1E2C40B106, 0xBD7F6454F5CF57DC, 0x506640412241433C], 0),
    (1, 4): ([0, 0, 2, 1], [0x51CBCE664D2B8CD9, 0x6236BF0FDB3051AB, 0xC12E9315DD2A1643,
                            0x0137BED2BDF23DFF], 1),
    (2, 2): ([1, 2], [0x7BD0DA85FE5E2031, 0xAA196D3841C431C7], 4),
    (2, 3): ([2, 1, 2], [0x647456AB0F675CF4, 0xACE1AC8CD95E2854, 0x9339B8335AD336B0], 0),
    (2, 4): ([0, 2, 1, 2], [0x51CBCE664D2B8CD9, 0x9EA5B27B3C373209, 0x4ACB0ED74D4A8C00,
                            0xFEE6F38B1EB5E84D], 3),
}

# a4 + a5: m_t = (v2 s2 + v3 s3 + v4 s4) / 3 over the three rows above; the
# columns repeat with period 5
M = {
    0: ["11/48", "5/24", "-1/3", "-7/48", "1/24"],
    1: ["-11/48", "-1/12", "-1/24", "5/48", "1/4"],
    2: ["-1/12", "1/8", "11/48", "1/48", "-7/24"],
}

# a6: the gate's three sums (exact), and g = sigmoid(sum(a m) /
# (sqrt(sum(a^2)/16 + eps) sqrt(sum(m^2)/16 + eps) sqrt(16))), a = X[t, 0]
GATE_SUMS = {0: ("43/2", "1711/2304", "-7/48"),
             1: ("89/4", "1051/2304", "187/384"),
             2: ("47/2", "563/1152", "-33/64")}
LOGIT = {0: -0.14598524281935943, 1: 0.61141694778392142, 2: -0.60858999903270727}
GATE = {0: 0.46356836796587114, 1: 0.64826395923030389, 2: 0.35238090525568616}

# a7: out[t, s, i] = bf16_rne(X[t, s, i] + g_t alpha_s m_t[i]), as bf16 bits
OUT = {
    0: [[0xbff2, 0xbfd4, 0xbfd4, 0xbfa9, 0xbf7b, 0xbf25, 0xbecf, 0xbecf,
         0xbd8a, 0x3e8a, 0x3f1b, 0x3f59, 0x3f58, 0x3f97, 0x3fc2, 0x3fee],
        [0xbfc7, 0xbfa6, 0xbf6c, 0xbf37, 0xbf02, 0xbe9b, 0xbd46, 0x3ea8,
         0x3f09, 0x3f3e, 0x3f72, 0x3f9a, 0x3fca, 0x3fe4, 0x3fff, 0x400d],
        [0xbf4a, 0xbf0f, 0xbf4f, 0xbec5, 0x3d1e, 0x3eed, 0x3f31, 0x3ee2,
         0x3f5d, 0x3fa5, 0x3fdb, 0x3ff9, 0x3fd8, 0x4007, 0x4022, 0x403e],
        [0xbef2, 0xbe67, 0xbd1e, 0x3e6f, 0x3f01, 0x3f47, 0x3f83, 0x3f9b,
         0x3fbe, 0x3fe1, 0x4002, 0x4012, 0x401e, 0x402f, 0x4040, 0x4052]],
    1: [[0xc012, 0xbff7, 0xbfd3, 0xbfa7, 0xbf77, 0xbf83, 0xbf2e, 0xbece,
         0xbd6b, 0x3e93, 0x3e68, 0x3f12, 0x3f59, 0x3f99, 0x3fc5, 0x3fbd],
        [0xbfc6, 0xbfad, 0xbf8e, 0xbf69, 0xbf35, 0xbe9a, 0xbdc9, 0x3e0e,
         0x3eaf, 0x3f0b, 0x3f73, 0x3f93, 0x3fb2, 0x3fcc, 0x3fe6, 0x400d],
        [0xbfb6, 0xbf7c, 0xbf2e, 0xbe76, 0x3e4c, 0xbe30, 0x3e89, 0x3f12,
         0x3f81, 0x3fb9, 0x3f8a, 0x3fc2, 0x3fe9, 0x4011, 0x402d, 0x4015],
        [0xbf2a, 0xbec7, 0xbe07, 0x3e11, 0x3ed5, 0x3f16, 0x3f5d, 0x3f8f,
         0x3fb2, 0x3fd5, 0x3feb, 0x4007, 0x4018, 0x4029, 0x403b, 0x4046]],
    2: [[0xc012, 0xbffa, 0xbfd6, 0xbfbf, 0xbfad, 0xbf84, 0xbf35, 0xbed7,
         0xbe78, 0xbdd2, 0x3e62, 0x3f0b, 0x3f55, 0x3f81, 0x3f93, 0x3fbc],
        [0xbfde, 0xbfc3, 0xbfa5, 0xbf80, 0xbf33, 0xbef8, 0xbe8b, 0xbd25,
         0x3e7c, 0x3f0d, 0x3f44, 0x3f7a, 0x3f9b, 0x3fc0, 0x3fe7, 0x4001],
        [0xbfa8, 0xbf69, 0xbf17, 0xbef8, 0xbee9, 0xbd71, 0x3ead, 0x3f29,
         0x3f44, 0x3f4b, 0x3f98, 0x3fcb, 0x3ff5, 0x4001, 0x4003, 0x401c],
        [0xbf42, 0xbefa, 0xbe6b, 0x3af1, 0x3e66, 0x3efc, 0x3f43, 0x3f83,
         0x3fa0, 0x3fbd, 0x3fdf, 0x4001, 0x4011, 0x4020, 0x402e, 0x4040]],
}

E4M3 = {-2: 0xB8, -1: 0xB0, 0: 0x00, 1: 0x30, 2: 0x38}   # value * 2 -> byte


def _tables():
    tabs, scales = [], []
    for n in (2, 3, 4):
        t = np.array([[E4M3[(r + i + n) % 5 - 2] for i in range(D)] for r in range(ROWS)], np.uint8)
        tabs.append(t)
        scales.append(np.array([(r + 1) / 8 for r in range(ROWS)], np.float32))
    return tabs, scales


def _streams():
    x = np.array([[[(i - 8) / 4 + s / 2 - t / 8 for i in range(D)] for s in range(4)]
                  for t in range(S)], np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)   # exact: every value fits bf16


def test_hand_worked_compression_seeds_folds_and_rows():
    eids, f = oracle.compress(TOKENS, TID2EID, N_EIDS)
    assert f == 0 and eids.tolist() == [EIDS]
    for n, s in SEEDS.items():
        assert oracle.seed(n, 0) == s
    for (t, n), (window, hs, row) in FOLDS.items():
        # the window is the token's last n eids, pad before the start
        assert window == [EIDS[p] if p >= 0 else 0 for p in range(t - n + 1, t + 1)]
        assert oracle.ngram_hash(window, n, 0) == hs[-1]
        assert hs[-1] % ROWS == row
    rows, flags = oracle.hash_ids(np.array([EIDS], np.int32), H, (ROWS,) * 3)
    assert flags == 0
    assert rows.reshape(S, 3).tolist() == [[FOLDS[(t, n)][2] for n in (2, 3, 4)] for t in range(S)]


def test_hand_worked_memory_gate_and_streams():
    rows = np.array([[FOLDS[(t, n)][2] for n in (2, 3, 4)] for t in range(S)], np.int32)
    tabs, scales = _tables()
    x = _streams()
    y, g, m, flags = oracle.lookup(rows, H, oracle.FP8, tabs, scales, x, ALPHA, EPS, aux=True)
    assert flags == 0
    for t in range(S):
        want_m = np.array([float(F(M[t][i % 5])) for i in range(D)])
        np.testing.assert_allclose(m[t], want_m, rtol=1e-15, atol=0)
        a = x[t, 0].astype(np.uint32) << 16
        a = a.view(np.float32).astype(np.float64)
        saa, smm, sam = (float(F(v)) for v in GATE_SUMS[t])
        assert np.sum(a * a) == saa                       # exact in fp64
        assert np.sum(m[t] * m[t]) == pytest.approx(smm, rel=1e-15)
        assert np.sum(a * m[t]) == pytest.approx(sam, rel=1e-14)
        logit = sam / (np.sqrt(saa / D + EPS) * np.sqrt(smm / D + EPS) * np.sqrt(D))
        assert logit == pytest.approx(LOGIT[t], rel=1e-14)
        assert g[t] == pytest.approx(GATE[t], rel=1e-14)
        assert y[t].tolist() == OUT[t], f"token {t}"
