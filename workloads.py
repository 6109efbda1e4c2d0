"""Seeded synthetic inputs for the Engram hashed n-gram memory lookup.

This module only draws random inputs: token ids, the tid2eid compression map, the
per-slot decode history, the n-gram tables (FP8 e4m3fn bytes + one fp32 scale per
row, or BF16), the four mHC residual streams and the per-stream alpha.  It holds
none of the method's arithmetic (no compression, hashing, dequantisation, gate or
add), so that the CPU oracle and the CUDA path can both be fed from it without
sharing any computation.

The five workloads restate the sizes and value distributions of the Engram
lookup described on the VeOmni PR page ("support DeepSeek-V4.1-Flash in
SeedOmni", PR description: three hashed 2/3/4-gram tables, 15.12M rows in total,
FP8 with row-wise dequantisation or BF16, tid2eid compression, 129,280-token
vocabulary) with the hash, gate and row width fixed by the workload spec
(splitmix64 seeds, 4096-wide rows, RMSNorm dot-product sigmoid gate).

Host generation uses NumPy PCG64 streams keyed by (seed, kind); the FP8 and BF16
casts are PyTorch CPU casts (round to nearest even; values are clipped to the
e4m3fn range first because torch's e4m3fn cast does not saturate).  Large tables
and streams are generated on the GPU with torch's seeded CUDA generator in
chunks; the oracle then reads the same bytes back.
"""
from __future__ import annotations

import dataclasses

import numpy as np

# Input kinds: one independent PCG64 stream per kind.
_K_IDS, _K_MAP, _K_TABLE, _K_SCALE, _K_STREAMS, _K_ALPHA, _K_HIST, _K_SPANS, _K_PACK, _K_WKV = \
    range(10)

FP8 = "fp8_e4m3fn"
BF16 = "bf16"
FP8_E8M0 = "fp8_e4m3fn_e8m0_1x32"   # one e8m0 exponent per row per 32 columns
# the same values, each row's exponents stored right after its bytes (rows padded
# to a multiple of 16 bytes)
FP8_E8M0_ROWS = "fp8_e4m3fn_e8m0_1x32_rows"
E4M3_MAX = 448.0


@dataclasses.dataclass(frozen=True)
class EngramConfig:
    """One synthetic Engram workload (sizes and distributions only)."""

    name: str
    seed: int
    B: int                 # batch (decode: slots)
    S: int                 # sequence length (decode: 1)
    vocab: int             # tokenizer vocabulary V
    n_eids: int            # compressed ids are 1..n_eids; 0 is the pad id
    H: int                 # hash heads per n-gram order
    D: int                 # row width = hidden size
    rows: tuple            # rows of the 2-, 3- and 4-gram tables
    dtype: str             # FP8 or BF16 tables
    ids: str = "uniform"   # "uniform" or "zipf"
    zipf_s: float = 1.1
    id_range: int = 0      # uniform ids in [0, id_range); 0 means [0, vocab)
    repeat_frac: float = 0.0   # fraction of positions that copy an earlier 4-token span
    decode: bool = False   # one new token per slot with a 3-id history
    packed: bool = False   # samples packed into each row; positions restart per sample
    mean_sample_len: int = 0
    image_span: int = 0    # length of one image span (dead positions)
    image_frac: float = 0.0  # target fraction of positions inside image spans
    bf16_std: float = 0.02
    scale_lo: float = 1e-3
    scale_hi: float = 1e-2
    e8m0_lo: int = 117     # block exponents uniform in [e8m0_lo, e8m0_hi]: 2^-10 .. 2^-7
    e8m0_hi: int = 120
    # The released layout: one table of rows[0] rows cut into prime buckets drawn
    # above hash_vocab (0: one table per n-gram order)
    hash_vocab: int = 0
    eps: float = 1e-6
    # The connection with a wkv projection: the 3H rows (width D) concatenated and
    # projected to `hidden` columns by wkv bf16 [hidden, 3H*D] from N(0, wkv_std^2);
    # the streams are then [B, S, 4, hidden].  0: no projection (the mean; streams
    # have the row width D)
    hidden: int = 0
    wkv_std: float = 1.0

    @property
    def T(self) -> int:
        return self.B * self.S

    @property
    def R(self) -> int:
        return 3 * self.H

    @property
    def width(self) -> int:
        """Width of the mHC streams: hidden with a projection, else the row width."""
        return self.hidden or self.D

    @property
    def K(self) -> int:
        """Width of a token's concatenated rows (the projection's inner dimension)."""
        return self.R * self.D

    def scaled(self, **kw) -> "EngramConfig":
        """Same distributions, other sizes (for parity cases the oracle finishes quickly)."""
        return dataclasses.replace(self, **kw)

    def row_bytes(self) -> int:
        """Bytes of one table row with its scales: FP8 D + 4 (fp32 row scale),
        FP8 with e8m0 blocks D + D/32 (apart or after the row), BF16 2D."""
        if self.dtype == FP8:
            return self.D + 4
        if self.dtype in (FP8_E8M0, FP8_E8M0_ROWS):
            return self.D + self.D // 32
        return 2 * self.D

    def stored_row_bytes(self) -> int:
        """Bytes a table row takes in memory (the rows-with-exponents layout pads
        each row to a multiple of 16 bytes)."""
        if self.dtype == FP8_E8M0_ROWS:
            return (self.D + self.D // 32 + 15) // 16 * 16
        return self.row_bytes()

    def table_bytes(self) -> int:
        if self.hash_vocab:
            return self.rows[0] * self.stored_row_bytes()
        return sum(r * self.stored_row_bytes() for r in self.rows)

    def algorithmic_bytes_per_token(self) -> int:
        """Bytes the fused lookup must move per token, with no cache credit:
        3H rows (+ their scales), the 3H int32 row ids, and the four bf16 streams
        read once and written once."""
        return self.R * self.row_bytes() + self.R * 4 + 2 * 4 * self.width * 2

    def connection_flops_per_token(self) -> int:
        """Multiply-adds of k = wkv e, counted as 2 flops each."""
        return 2 * self.hidden * self.K


CONFIGS = [
    # 0: tiny, CPU-checkable
    EngramConfig(name="tiny_fp8_d256", seed=0, B=1, S=256, vocab=1024, n_eids=800, H=2, D=256,
                 rows=(4096, 4096, 4096), dtype=FP8, ids="uniform"),
    # 1: mid prefill
    EngramConfig(name="mid_prefill_fp8", seed=1, B=4, S=4096, vocab=129_280, n_eids=100_000, H=4,
                 D=4096, rows=(1_000_000,) * 3, dtype=FP8, ids="zipf"),
    # 2: decode step, 512 slots x 1 token with a 3-id history per slot
    EngramConfig(name="decode_fp8", seed=2, B=512, S=1, vocab=129_280, n_eids=100_000, H=4,
                 D=4096, rows=(5_040_000,) * 3, dtype=FP8, ids="uniform", decode=True),
    # 3: full-size prefill with repeated n-grams
    EngramConfig(name="full_prefill_fp8", seed=3, B=8, S=8192, vocab=129_280, n_eids=100_000,
                 H=8, D=4096, rows=(5_040_000,) * 3, dtype=FP8, ids="zipf", repeat_frac=0.05),
    # 4: BF16 tables, uniform (cache-hostile) ids
    EngramConfig(name="bf16_tables", seed=4, B=4, S=8192, vocab=129_280, n_eids=100_000, H=4,
                 D=4096, rows=(5_040_000,) * 3, dtype=BF16, ids="uniform"),
    # 5: packed multimodal prefill: samples of ~1024 tokens packed into each row
    #    (positions restart per sample), a quarter of the positions in 256-token
    #    image spans (dead); otherwise the full-size prefill
    EngramConfig(name="packed_mm_fp8", seed=5, B=8, S=8192, vocab=129_280, n_eids=100_000,
                 H=8, D=4096, rows=(5_040_000,) * 3, dtype=FP8, ids="zipf", packed=True,
                 mean_sample_len=1024, image_span=256, image_frac=0.25),
    # 6: full-size prefill with e8m0 block-scaled FP8 tables (the release's dequantisation)
    EngramConfig(name="full_prefill_fp8_e8m0", seed=6, B=8, S=8192, vocab=129_280,
                 n_eids=100_000, H=8, D=4096, rows=(5_040_000,) * 3, dtype=FP8_E8M0, ids="zipf",
                 repeat_frac=0.05),
    # 6b: the same tables with each row's exponents stored after its bytes
    #     (4224-byte rows): the same seed, so the same values as 6
    EngramConfig(name="full_prefill_fp8_e8m0_rows", seed=6, B=8, S=8192, vocab=129_280,
                 n_eids=100_000, H=8, D=4096, rows=(5_040_000,) * 3, dtype=FP8_E8M0_ROWS,
                 ids="zipf", repeat_frac=0.05),
    # 7: the released table layout: one Engram layer's table of 384,006,168 rows
    #    of 256 FP8 values with (1, 32) e8m0 blocks (98 GB), cut into 24 prime
    #    buckets (orders 2..4 x 8 heads) drawn above a 16,000,000 hash vocabulary
    EngramConfig(name="release_layout_fp8", seed=7, B=8, S=8192, vocab=129_280, n_eids=100_000,
                 H=8, D=256, rows=(384_006_168,) * 3, dtype=FP8_E8M0, ids="zipf",
                 repeat_frac=0.05, hash_vocab=16_000_000),
    # 7b: the released table layout with each row's exponents stored after its
    #     bytes (272-byte rows, 104 GB): the same seed, so the same values as 7
    EngramConfig(name="release_layout_fp8_rows", seed=7, B=8, S=8192, vocab=129_280,
                 n_eids=100_000, H=8, D=256, rows=(384_006_168,) * 3, dtype=FP8_E8M0_ROWS,
                 ids="zipf", repeat_frac=0.05, hash_vocab=16_000_000),
    # 8: the connection with a wkv projection on the released table layout: a
    #    token's 24 rows of 256 (K = 6144) projected to the 4096-wide streams;
    #    wkv_std 2 gives k about the streams' unit scale (rows ~ 0.0045 rms)
    EngramConfig(name="release_connection_e8m0", seed=8, B=8, S=8192, vocab=129_280,
                 n_eids=100_000, H=8, D=256, rows=(384_006_168,) * 3, dtype=FP8_E8M0, ids="zipf",
                 repeat_frac=0.05, hash_vocab=16_000_000, hidden=4096, wkv_std=2.0),
]


def by_name(name: str) -> EngramConfig:
    """The workload of that name."""
    for c in CONFIGS:
        if c.name == name:
            return c
    raise KeyError(name)


def rng(cfg: EngramConfig, kind: int, sub: int = 0) -> np.random.Generator:
    return np.random.default_rng([cfg.seed, kind, sub])


# ---------------------------------------------------------------- small inputs

def _zipf_ranks(g: np.random.Generator, n: int, vocab: int, s: float) -> np.ndarray:
    """Finite Zipf over ranks 1..vocab, P(k) proportional to k^-s; returns rank-1."""
    k = np.arange(1, vocab + 1, dtype=np.float64)
    cdf = np.cumsum(k ** (-s))
    cdf /= cdf[-1]
    u = g.random(n)
    idx = np.searchsorted(cdf, u, side="right")
    return np.minimum(idx, vocab - 1).astype(np.int32)


def plant_repeats(ids: np.ndarray, frac: float, g: np.random.Generator) -> list:
    """Copy earlier 4-token spans into round(frac*S/4) non-overlapping 4-aligned
    destination spans of every sequence, destinations taken left to right, each
    source start drawn uniformly from the positions whose span ends at or before
    the destination.  Returns [(b, src, dst)] for tests."""
    B, S = ids.shape
    n_spans = int(round(frac * S / 4))
    planted = []
    if n_spans == 0 or S < 8:
        return planted
    for b in range(B):
        blocks = g.choice(np.arange(1, S // 4), size=min(n_spans, S // 4 - 1), replace=False)
        for dst in np.sort(blocks) * 4:
            src = int(g.integers(0, dst - 4 + 1))
            ids[b, dst:dst + 4] = ids[b, src:src + 4]
            planted.append((b, src, int(dst)))
    return planted


def token_ids(cfg: EngramConfig, rank: int = 0) -> np.ndarray:
    """[B, S] int32 token ids.  `rank` picks an independent batch per replica."""
    g = rng(cfg, _K_IDS, rank)
    n = cfg.T
    if cfg.ids == "zipf":
        ids = _zipf_ranks(g, n, cfg.vocab, cfg.zipf_s)
    else:
        hi = cfg.id_range or cfg.vocab
        ids = g.integers(0, hi, size=n, dtype=np.int64).astype(np.int32)
    ids = ids.reshape(cfg.B, cfg.S)
    if cfg.repeat_frac > 0:
        plant_repeats(ids, cfg.repeat_frac, rng(cfg, _K_SPANS, rank))
    return np.ascontiguousarray(ids)


def packed_layout(cfg: EngramConfig, rank: int = 0):
    """(positions [B, S] int32, dead [B, S] uint8) of a packed batch: every row is
    cut into samples of U[L/2, 3L/2] tokens (L = mean_sample_len, the last one cut
    at the row's end), positions count from 0 in each sample, and a sample holds
    one image span of image_span dead positions at a uniform offset with
    probability image_frac * len / image_span (capped at 1)."""
    B, S = cfg.B, cfg.S
    pos = np.zeros((B, S), np.int32)
    dead = np.zeros((B, S), np.uint8)
    if not cfg.packed:
        pos[:] = np.arange(S, dtype=np.int32)[None, :]
        return pos, dead
    g = rng(cfg, _K_PACK, rank)
    L = max(1, cfg.mean_sample_len)
    for b in range(B):
        s0 = 0
        while s0 < S:
            n = int(min(S - s0, g.integers(max(1, L // 2), L + L // 2 + 1)))
            pos[b, s0:s0 + n] = np.arange(n, dtype=np.int32)
            span = cfg.image_span
            if span and n > span and g.random() < min(1.0, cfg.image_frac * n / span):
                off = int(g.integers(0, n - span + 1))
                dead[b, s0 + off:s0 + off + span] = 1
            s0 += n
    return pos, dead


def tid2eid(cfg: EngramConfig) -> np.ndarray:
    """[vocab] int32 many-to-one map onto 1..n_eids (0 stays the pad id)."""
    return rng(cfg, _K_MAP).integers(1, cfg.n_eids + 1, size=cfg.vocab, dtype=np.int64).astype(np.int32)


def history(cfg: EngramConfig, rank: int = 0) -> np.ndarray | None:
    """[B, 3] int32 previous eids, oldest first, for decode workloads."""
    if not cfg.decode:
        return None
    g = rng(cfg, _K_HIST, rank)
    return g.integers(1, cfg.n_eids + 1, size=(cfg.B, 3), dtype=np.int64).astype(np.int32)


def alpha(cfg: EngramConfig) -> np.ndarray:
    """[4] fp32 per-stream scale, N(0,1)."""
    return rng(cfg, _K_ALPHA).standard_normal(4).astype(np.float32)


def _to_bf16_bits(x: np.ndarray) -> np.ndarray:
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


def _to_e4m3_bytes(x: np.ndarray) -> np.ndarray:
    import torch
    x = np.clip(x, -E4M3_MAX, E4M3_MAX).astype(np.float32)
    return torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def streams_host(cfg: EngramConfig, rank: int = 0) -> np.ndarray:
    """[B, S, 4, width] bf16 bit patterns (uint16), N(0,1)."""
    g = rng(cfg, _K_STREAMS, rank)
    x = g.standard_normal((cfg.B, cfg.S, 4, cfg.width), dtype=np.float32)
    return _to_bf16_bits(x)


def wkv_host(cfg: EngramConfig) -> np.ndarray:
    """[hidden, K] bf16 bit patterns (uint16), N(0, wkv_std^2)."""
    g = rng(cfg, _K_WKV)
    x = g.standard_normal((cfg.hidden, cfg.K), dtype=np.float32) * np.float32(cfg.wkv_std)
    return _to_bf16_bits(x)


def tables_host(cfg: EngramConfig):
    """Three tables on the host: (tables, scales).  FP8: uint8 [rows, D] from N(0,1)
    clipped to +-448 + fp32 scales U[scale_lo, scale_hi]; FP8_E8M0: the same bytes
    + uint8 e8m0 exponents [rows, D/32] uniform in [e8m0_lo, e8m0_hi]; BF16:
    uint16 bits from N(0, bf16_std), scales None."""
    tabs, scales = [], []
    for n in range(1 if cfg.hash_vocab else 3):
        g = rng(cfg, _K_TABLE, n)
        x = g.standard_normal((cfg.rows[n], cfg.D), dtype=np.float32)
        if cfg.dtype == FP8:
            tabs.append(_to_e4m3_bytes(x))
            gs = rng(cfg, _K_SCALE, n)
            scales.append(gs.uniform(cfg.scale_lo, cfg.scale_hi, size=cfg.rows[n]).astype(np.float32))
        elif cfg.dtype in (FP8_E8M0, FP8_E8M0_ROWS):
            t = _to_e4m3_bytes(x)
            gs = rng(cfg, _K_SCALE, n)
            e = gs.integers(cfg.e8m0_lo, cfg.e8m0_hi + 1, size=(cfg.rows[n], cfg.D // 32),
                            dtype=np.int64).astype(np.uint8)
            if cfg.dtype == FP8_E8M0:
                tabs.append(t)
                scales.append(e)
            else:   # each row, then its exponents, then zeros
                packed = np.zeros((cfg.rows[n], cfg.stored_row_bytes()), np.uint8)
                packed[:, :cfg.D] = t
                packed[:, cfg.D:cfg.D + cfg.D // 32] = e
                tabs.append(packed)
                scales.append(None)
        else:
            tabs.append(_to_bf16_bits(x * np.float32(cfg.bf16_std)))
            scales.append(None)
    if cfg.hash_vocab:   # one table, shared by the three orders
        tabs, scales = tabs * 3, scales * 3
    return tabs, scales


# ---------------------------------------------------------------- device inputs

def _dev_gen(device, seed: int):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def tables_device(cfg: EngramConfig, device, chunk_rows: int = 1 << 18):
    """Three tables generated on the GPU in chunks with torch's seeded CUDA
    generator (same distributions as tables_host, different bytes).  Returns
    (tables, scales): uint8 [rows, D] or bf16-as-int16 [rows, D] tensors and fp32
    [rows] scales (None for BF16)."""
    import torch
    tabs, scales = [], []
    for n in range(1 if cfg.hash_vocab else 3):
        rows = cfg.rows[n]
        g = _dev_gen(device, cfg.seed * 1_000_003 + 101 * n + 7)
        fp8 = cfg.dtype in (FP8, FP8_E8M0, FP8_E8M0_ROWS)
        packed = cfg.dtype == FP8_E8M0_ROWS
        if packed:   # rows with their exponents after them: [rows, stored_row_bytes]
            t = torch.zeros((rows, cfg.stored_row_bytes()), dtype=torch.uint8, device=device)
        elif fp8:
            t = torch.empty((rows, cfg.D), dtype=torch.uint8, device=device)
        else:
            t = torch.empty((rows, cfg.D), dtype=torch.int16, device=device)
        for r0 in range(0, rows, chunk_rows):
            r1 = min(rows, r0 + chunk_rows)
            x = torch.randn((r1 - r0, cfg.D), generator=g, device=device, dtype=torch.float32)
            if fp8:
                t[r0:r1, :cfg.D] = x.clamp_(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8)
            else:
                t[r0:r1] = x.mul_(cfg.bf16_std).to(torch.bfloat16).view(torch.int16)
            del x
        tabs.append(t)
        if cfg.dtype == FP8:
            gs = _dev_gen(device, cfg.seed * 1_000_003 + 101 * n + 11)
            s = torch.rand((rows,), generator=gs, device=device, dtype=torch.float32)
            scales.append(s.mul_(cfg.scale_hi - cfg.scale_lo).add_(cfg.scale_lo))
        elif cfg.dtype == FP8_E8M0:
            gs = _dev_gen(device, cfg.seed * 1_000_003 + 101 * n + 11)
            scales.append(torch.randint(cfg.e8m0_lo, cfg.e8m0_hi + 1, (rows, cfg.D // 32),
                                        generator=gs, device=device, dtype=torch.int32)
                          .to(torch.uint8))
        elif packed:   # the same draws as FP8_E8M0, written after each row, in chunks
            gs = _dev_gen(device, cfg.seed * 1_000_003 + 101 * n + 11)
            e = torch.randint(cfg.e8m0_lo, cfg.e8m0_hi + 1, (rows, cfg.D // 32),
                              generator=gs, device=device, dtype=torch.int32)
            for r0 in range(0, rows, 1 << 24):
                r1 = min(rows, r0 + (1 << 24))
                t[r0:r1, cfg.D:cfg.D + cfg.D // 32] = e[r0:r1].to(torch.uint8)
            del e
            scales.append(None)
        else:
            scales.append(None)
    if cfg.hash_vocab:   # one table, shared by the three orders
        tabs, scales = tabs * 3, scales * 3
    return tabs, scales


def streams_device(cfg: EngramConfig, device, rank: int = 0, chunk_tokens: int = 4096):
    """[B, S, 4, width] bf16 N(0,1) streams generated on the GPU (as int16 bits)."""
    import torch
    out = torch.empty((cfg.T, 4, cfg.width), dtype=torch.int16, device=device)
    g = _dev_gen(device, cfg.seed * 1_000_003 + 977 + 13 * rank)
    for t0 in range(0, cfg.T, chunk_tokens):
        t1 = min(cfg.T, t0 + chunk_tokens)
        x = torch.randn((t1 - t0, 4, cfg.width), generator=g, device=device, dtype=torch.float32)
        out[t0:t1] = x.to(torch.bfloat16).view(torch.int16)
        del x
    return out.view(cfg.B, cfg.S, 4, cfg.width)


def wkv_device(cfg: EngramConfig, device):
    """[hidden, K] bf16 N(0, wkv_std^2) projection generated on the GPU (as int16 bits)."""
    import torch
    g = _dev_gen(device, cfg.seed * 1_000_003 + 4099)
    x = torch.randn((cfg.hidden, cfg.K), generator=g, device=device, dtype=torch.float32)
    return x.mul_(cfg.wkv_std).to(torch.bfloat16).view(torch.int16)


def bytes_human(n: float) -> str:
    for unit in ("B", "KB", "MB", "GB", "TB"):
        if abs(n) < 1000 or unit == "TB":
            return f"{n:.3g} {unit}"
        n /= 1000.0
    return f"{n} B"

