"""Plain CPU oracle of the Engram hashed n-gram memory lookup (NumPy front end).

TEST INFRASTRUCTURE ONLY.  The oracle is the parity reference for the CUDA
library.  Only the test suite, the smoke check and the benchmark's CPU-baseline
leg may import it; the library never does, and this package never imports the
library.  The arithmetic lives in engram_oracle.c (fp64, one token at a time);
this module marshals NumPy arrays into it.
"""
from __future__ import annotations

import ctypes as C

import numpy as np

from . import build as _build

FP8 = 0
BF16 = 1
FP8_E8M0 = 2
DEAD = -1
BAD_TOKEN, BAD_EID, BAD_ROW, BAD_ARG = 1, 2, 4, 16

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        i32p = C.POINTER(C.c_int32)
        L.orc_splitmix64.restype = C.c_uint64
        L.orc_splitmix64.argtypes = [C.c_uint64]
        L.orc_seed.restype = C.c_uint64
        L.orc_seed.argtypes = [C.c_int, C.c_int]
        L.orc_ngram_hash.restype = C.c_uint64
        L.orc_ngram_hash.argtypes = [i32p, C.c_int, C.c_int]
        L.orc_e4m3fn_decode.restype = C.c_double
        L.orc_e4m3fn_decode.argtypes = [C.c_uint8]
        L.orc_bf16_decode.restype = C.c_double
        L.orc_bf16_decode.argtypes = [C.c_uint16]
        L.orc_e8m0_decode.restype = C.c_double
        L.orc_e8m0_decode.argtypes = [C.c_uint8]
        L.orc_bf16_round.restype = C.c_uint16
        L.orc_bf16_round.argtypes = [C.c_double]
        L.orc_compress.restype = C.c_int
        L.orc_compress.argtypes = [C.c_void_p, C.c_int64, C.c_void_p, C.c_int32, C.c_int32,
                                   C.c_void_p]
        L.orc_compress_masked.restype = C.c_int
        L.orc_compress_masked.argtypes = [C.c_void_p, C.c_int64, C.c_void_p, C.c_int32, C.c_int32,
                                          C.c_void_p, C.c_void_p]
        L.orc_hash_packed.restype = C.c_int
        L.orc_hash_packed.argtypes = [C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p,
                                      C.c_int32, C.POINTER(C.c_int64), C.c_void_p, C.c_void_p]
        L.orc_bucket_primes.restype = C.c_int
        L.orc_bucket_primes.argtypes = [C.c_int32, C.c_int32, C.c_int32, C.c_int64, C.c_void_p]
        L.orc_hash_bucketed.restype = C.c_int
        L.orc_hash_bucketed.argtypes = [C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p,
                                        C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p]
        L.orc_hash.restype = C.c_int
        L.orc_hash.argtypes = [C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_int32,
                               C.POINTER(C.c_int64), C.c_void_p, C.c_void_p]
        L.orc_lookup.restype = C.c_int
        L.orc_lookup.argtypes = [C.c_void_p, C.c_int64, C.c_int32, C.c_int32, C.c_int32,
                                 C.c_void_p * 3, C.c_void_p * 3, C.POINTER(C.c_int64),
                                 C.c_void_p, C.c_void_p, C.c_double, C.c_void_p, C.c_void_p,
                                 C.c_void_p]
        L.orc_connection.restype = C.c_int
        L.orc_connection.argtypes = [C.c_void_p, C.c_int64, C.c_int32, C.c_int32, C.c_int32,
                                     C.c_void_p * 3, C.c_void_p * 3, C.POINTER(C.c_int64),
                                     C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p, C.c_double,
                                     C.c_void_p, C.c_void_p, C.c_void_p]
        L.orc_num_threads.restype = C.c_int
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return int(lib().orc_num_threads())


def splitmix64(x: int) -> int:
    return int(lib().orc_splitmix64(x))


def seed(n: int, j: int) -> int:
    return int(lib().orc_seed(n, j))


def ngram_hash(window, n: int, j: int) -> int:
    w = _c(window, np.int32)
    assert w.size == n
    return int(lib().orc_ngram_hash(w.ctypes.data_as(C.POINTER(C.c_int32)), n, j))


def e4m3fn_decode(b: int) -> float:
    return float(lib().orc_e4m3fn_decode(b))


def bf16_decode(bits: int) -> float:
    return float(lib().orc_bf16_decode(bits))


def e8m0_decode(e: int) -> float:
    return float(lib().orc_e8m0_decode(e))


def bf16_round(y: float) -> int:
    return int(lib().orc_bf16_round(y))


def compress(token_ids, tid2eid, n_eids: int, fill: int = -7):
    """eids (same shape as token_ids) and the error flags; unwritten outputs keep `fill`."""
    tid = _c(token_ids, np.int32)
    m = _c(tid2eid, np.int32)
    out = np.full(tid.shape, fill, dtype=np.int32)
    flags = lib().orc_compress(_p(tid), tid.size, _p(m), m.size, n_eids, _p(out))
    return out, int(flags)


def compress_masked(token_ids, tid2eid, n_eids: int, dead, fill: int = -7):
    """As compress, with dead positions (mask != 0) set to DEAD."""
    tid = _c(token_ids, np.int32)
    m = _c(tid2eid, np.int32)
    d = _c(dead, np.uint8)
    assert d.shape == tid.shape
    out = np.full(tid.shape, fill, dtype=np.int32)
    flags = lib().orc_compress_masked(_p(tid), tid.size, _p(m), m.size, n_eids, _p(d), _p(out))
    return out, int(flags)


def hash_ids(eids, n_heads: int, rows, history=None, want_history: bool = False,
             fill: int = -7, positions=None):
    """Row ids [B, S, 3, H] (and the next history [B, 3]) and the error flags.
    positions [B, S] (optional): each token's index within its packed sample."""
    e = _c(eids, np.int32)
    assert e.ndim == 2
    B, S = e.shape
    hist = None if history is None else _c(history, np.int32).reshape(B, 3)
    pos = None if positions is None else _c(positions, np.int32).reshape(B, S)
    out = np.full((B, S, 3, n_heads), fill, dtype=np.int32)
    hout = np.full((B, 3), fill, dtype=np.int32) if want_history else None
    r = (C.c_int64 * 3)(*[int(x) for x in rows])
    flags = lib().orc_hash_packed(_p(e), B, S, _p(pos), _p(hist), n_heads, r, _p(out), _p(hout))
    if want_history:
        return out, hout, int(flags)
    return out, int(flags)


def bucket_primes(n_layers: int, max_ngram: int, n_heads: int, hash_vocab: int) -> np.ndarray:
    """[n_layers, max_ngram - 1, n_heads] int64 primes of the bucket layout."""
    out = np.zeros(n_layers * (max_ngram - 1) * n_heads, np.int64)
    flags = lib().orc_bucket_primes(n_layers, max_ngram, n_heads, hash_vocab, _p(out))
    assert flags == 0
    return out.reshape(n_layers, max_ngram - 1, n_heads)


def hash_bucketed(eids, n_heads: int, primes, history=None, positions=None,
                  want_history: bool = False, fill: int = -7):
    """Row ids [B, S, 3, H] into one prime-bucketed table (primes [3, H] of one layer)."""
    e = _c(eids, np.int32)
    B, S = e.shape
    hist = None if history is None else _c(history, np.int32).reshape(B, 3)
    pos = None if positions is None else _c(positions, np.int32).reshape(B, S)
    pr = _c(primes, np.int64).reshape(-1)
    assert pr.size == 3 * n_heads
    out = np.full((B, S, 3, n_heads), fill, dtype=np.int32)
    hout = np.full((B, 3), fill, dtype=np.int32) if want_history else None
    flags = lib().orc_hash_bucketed(_p(e), B, S, _p(pos), _p(hist), n_heads, _p(pr), _p(out),
                                    _p(hout))
    if want_history:
        return out, hout, int(flags)
    return out, int(flags)


def lookup(row_ids, n_heads: int, dtype: int, tables, scales, streams, alpha, eps: float,
           rows=None, aux: bool = False, fill: int = 0xDEAD):
    """The fused lookup on [T, 3H] row ids and [T, 4, D] bf16 streams (uint16 bits).

    Returns streams_out (uint16, same shape as streams), and with aux=True also the
    gate g [T] and memory m [T, D] in fp64, plus the error flags."""
    ids = _c(row_ids, np.int32)
    x = _c(streams, np.uint16)
    D = x.shape[-1]
    T = x.size // (4 * D)
    assert ids.size == T * 3 * n_heads
    tabs = [_c(t, np.uint16 if dtype == BF16 else np.uint8) for t in tables]
    sdt = np.uint8 if dtype == FP8_E8M0 else np.float32
    scs = [(_c(s, sdt) if s is not None else None) for s in scales] if scales else [None] * 3
    if rows is None:
        rows = [t.shape[0] for t in tabs]
    a = _c(alpha, np.float32)
    y = np.full(x.shape, fill, dtype=np.uint16)
    g = np.full(T, np.nan) if aux else None
    m = np.full((T, D), np.nan) if aux else None
    tp = (C.c_void_p * 3)(*[t.ctypes.data for t in tabs])
    sp = (C.c_void_p * 3)(*[(s.ctypes.data if s is not None else None) for s in scs])
    r = (C.c_int64 * 3)(*[int(v) for v in rows])
    flags = lib().orc_lookup(_p(ids), T, n_heads, dtype, D, tp, sp, r, _p(x), _p(a), float(eps),
                             _p(y), _p(g), _p(m))
    if aux:
        return y, g, m, int(flags)
    return y, int(flags)


def connection(row_ids, n_heads: int, dtype: int, tables, scales, wkv, streams, alpha, eps: float,
               rows=None, fill: int = 0xDEAD):
    """The wkv connection: rows concatenated per token, projected by wkv [D, K]
    (bf16 bits), gated and added into the streams [T, 4, D].  Returns
    (streams_out, gate [T], k [T, D], flags)."""
    ids = _c(row_ids, np.int32)
    x = _c(streams, np.uint16)
    D = x.shape[-1]
    T = x.size // (4 * D)
    tabs = [_c(t, np.uint16 if dtype == BF16 else np.uint8) for t in tables]
    d = tabs[0].shape[1]
    scs = [(_c(s, np.uint8) if s is not None else None) for s in scales] if scales else [None] * 3
    w = _c(wkv, np.uint16)
    assert w.shape == (D, 3 * n_heads * d)
    if rows is None:
        rows = [t.shape[0] for t in tabs]
    a = _c(alpha, np.float32)
    y = np.full(x.shape, fill, dtype=np.uint16)
    g = np.full(T, np.nan)
    k = np.full((T, D), np.nan)
    tp = (C.c_void_p * 3)(*[t.ctypes.data for t in tabs])
    sp = (C.c_void_p * 3)(*[(s.ctypes.data if s is not None else None) for s in scs])
    r = (C.c_int64 * 3)(*[int(v) for v in rows])
    flags = lib().orc_connection(_p(ids), T, n_heads, dtype, d, tp, sp, r, _p(w), D, _p(x), _p(a),
                                 float(eps), _p(y), _p(g), _p(k))
    return y, g, k, int(flags)


def bf16_bits_to_float(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (for comparisons)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)

