"""Engram hashed n-gram memory lookup for GB300 (sm_103a).

A thin Python binding over libengram.so, whose C ABI is include/engram.h.  The
functions carry the C names and only marshal arguments: torch tensors become
device pointers, the current torch CUDA stream becomes the cudaStream_t, and a
non-zero status becomes an EngramError.  Every step of the path runs in the
library's CUDA kernels; there is no CPU or PyTorch fallback, and importing this
package fails if the library has not been built.
"""
from __future__ import annotations

import ctypes as C
import dataclasses
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libengram.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_OUT_OF_RANGE, ERR_TIMEOUT = range(6)
FLAG_BAD_TOKEN, FLAG_BAD_EID, FLAG_BAD_ROW, FLAG_TIMEOUT = 1, 2, 4, 8
TABLE_FP8_E4M3FN, TABLE_BF16, TABLE_FP8_E8M0, TABLE_FP8_E8M0_ROWS = 0, 1, 2, 3
EID_DEAD = ROW_DEAD = -1
LOOKUP_AUTO, LOOKUP_GATHER, LOOKUP_BULK = 0, 1, 2
PROJECTION_AUTO, PROJECTION_SINGLE, PROJECTION_PAIR = 0, 1, 2
MAX_HEADS, MAX_D = 32, 4096


class EngramError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(message)
        self.code = code


class engram_tables(C.Structure):
    _fields_ = [("dtype", C.c_int32), ("D", C.c_int32), ("rows", C.c_int64 * 3),
                ("table", C.c_void_p * 3), ("scale", C.c_void_p * 3)]


class engram_layout(C.Structure):
    _fields_ = [("positions", C.c_void_p), ("dead", C.c_void_p),
                ("primes", C.POINTER(C.c_int64))]


def _layout(positions, dead, primes, host: bool):
    """The engram_layout struct for the whole-path calls (None when all three are
    None).  positions / dead are device tensors, or host tensors when `host`;
    primes is [3][n_heads] bucket sizes (host ints).  The struct keeps the
    primes array alive."""
    import torch
    if positions is None and dead is None and primes is None:
        return None
    for t, name, dts in ((positions, "positions", (torch.int32,)),
                         (dead, "dead", (torch.uint8, torch.bool))):
        if t is None:
            continue
        if t.is_cuda == host:
            where = "host" if host else "CUDA"
            raise EngramError(ERR_INVALID_ARG, f"{name} must be a {where} tensor here")
        if t.dtype not in dts or not t.is_contiguous():
            raise EngramError(ERR_INVALID_ARG, f"{name} must be contiguous {dts}")
    lay = engram_layout()
    lay.positions = None if positions is None else positions.data_ptr()
    lay.dead = None if dead is None else dead.data_ptr()
    if primes is not None:
        flat = [int(v) for order in primes for v in order]
        lay._primes = (C.c_int64 * len(flat))(*flat)
        lay.primes = C.cast(lay._primes, C.POINTER(C.c_int64))
    return lay


def _ref(lay):
    return None if lay is None else C.byref(lay)


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build the CUDA library first "
            "(python hashed_gram_memory_gb300/build.py, or __graft_entry__.build())")
    L = C.CDLL(LIB_PATH)
    vp, i32, i64 = C.c_void_p, C.c_int32, C.c_int64
    L.engram_compress.argtypes = [vp, i64, vp, i32, i32, vp, vp, vp]
    L.engram_compress_masked.argtypes = [vp, i64, vp, i32, i32, vp, vp, vp, vp]
    L.engram_hash.argtypes = [vp, i32, i32, vp, vp, i32, C.POINTER(C.c_int64), vp, vp, vp]
    L.engram_hash_packed.argtypes = [vp, i32, i32, vp, vp, vp, i32, C.POINTER(C.c_int64), vp, vp,
                                     vp]
    L.engram_hash_bucketed.argtypes = [vp, i32, i32, vp, vp, vp, i32, C.POINTER(C.c_int64), vp, vp,
                                       vp]
    L.engram_bucket_primes.argtypes = [i32, i32, i32, i64, C.POINTER(C.c_int64)]
    L.engram_compress_hash.argtypes = [vp, i32, i32, vp, i32, i32, vp, vp, i32,
                                       C.POINTER(C.c_int64), C.POINTER(engram_layout), vp, vp, vp,
                                       vp]
    L.engram_lookup_fused.argtypes = [vp, i64, i32, C.POINTER(engram_tables), vp, vp, vp,
                                      C.c_float, vp, vp, vp, vp]
    L.engram_read_status.argtypes = [vp, C.POINTER(C.c_int32), vp]
    for f in ("engram_compress", "engram_compress_masked", "engram_hash", "engram_hash_packed",
              "engram_hash_bucketed", "engram_bucket_primes", "engram_compress_hash",
              "engram_lookup_fused", "engram_read_status"):
        getattr(L, f).restype = C.c_int32
    L.engram_status_string.argtypes = [C.c_int32]
    L.engram_status_string.restype = C.c_char_p
    L.engram_last_error.argtypes = []
    L.engram_last_error.restype = C.c_char_p
    L.engram_abi_version.restype = C.c_int32
    L.engram_set_lookup_kernel.argtypes = [C.c_int32]
    L.engram_set_lookup_kernel.restype = C.c_int32
    L.engram_set_projection_kernel.argtypes = [C.c_int32]
    L.engram_set_projection_kernel.restype = C.c_int32
    L.engram_set_wait_limit_ns.argtypes = [C.c_int64]
    L.engram_set_wait_limit_ns.restype = C.c_int64
    L.engram_debug_withhold_copies.argtypes = [C.c_int32]
    L.engram_debug_withhold_copies.restype = None
    sz = C.c_size_t
    L.engram_forward_workspace_bytes.argtypes = [i32, i32, i32]
    L.engram_forward_workspace_bytes.restype = sz
    tabp, layp = C.POINTER(engram_tables), C.POINTER(engram_layout)
    L.engram_forward.argtypes = [vp, i32, i32, vp, i32, i32, vp, vp, i32, tabp, layp,
                                 vp, vp, vp, C.c_float, vp, sz, vp, vp]
    L.engram_forward.restype = i32
    L.engram_forward_host_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
    L.engram_forward_host_workspace_bytes.restype = sz
    L.engram_forward_host.argtypes = [vp, i32, i32, vp, i32, i32, vp, vp, i32, tabp, layp,
                                      vp, vp, vp, C.c_float, i32, vp, sz, vp, vp]
    L.engram_forward_host.restype = i32
    L.engram_forward_static.argtypes = [vp, i32, i32, vp, i32, i32, vp, vp, i32, tabp, layp,
                                        vp, vp, vp, C.c_float, vp, vp]
    L.engram_forward_static.restype = i32
    L.engram_connection_host_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
    L.engram_connection_host_workspace_bytes.restype = sz
    L.engram_connection_host.argtypes = [vp, i32, i32, vp, i32, i32, vp, vp, i32, tabp, layp,
                                         vp, i32, vp, vp, vp, C.c_float, i32, vp, sz, vp, vp]
    L.engram_connection_host.restype = i32
    L.engram_connection_workspace_bytes.argtypes = [i64, i32, i32, i32]
    L.engram_connection_workspace_bytes.restype = sz
    L.engram_connection.argtypes = [vp, i64, i32, C.POINTER(engram_tables), vp, i32, vp, vp, vp,
                                    C.c_float, vp, sz, vp, vp, vp, vp]
    L.engram_connection.restype = i32
    L.engram_concat_rows.argtypes = [vp, i64, i32, C.POINTER(engram_tables), vp, vp, vp, vp]
    L.engram_concat_rows.restype = i32
    L.engram_wkv_project.argtypes = [vp, i64, i32, vp, i32, vp, vp, vp]
    L.engram_wkv_project.restype = i32
    L.engram_gate_add.argtypes = [vp, vp, i64, i32, vp, vp, vp, C.c_float, vp, vp]
    L.engram_gate_add.restype = i32
    L.engram_pack_e8m0_rows.argtypes = [vp, vp, i64, i32, vp, vp]
    L.engram_pack_e8m0_rows.restype = i32
    return L


lib = _load()


def _check(code: int, what: str):
    if code != OK:
        msg = lib.engram_last_error().decode() or lib.engram_status_string(code).decode()
        raise EngramError(code, f"{what}: {lib.engram_status_string(code).decode()}: {msg}")


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        return C.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return C.c_void_p(stream)
    return C.c_void_p(stream.cuda_stream)


def _need(t, dtypes, name, contiguous=True):
    if t is None:
        return
    if not t.is_cuda:
        raise EngramError(ERR_INVALID_ARG, f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise EngramError(ERR_INVALID_ARG, f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if contiguous and not t.is_contiguous():
        raise EngramError(ERR_INVALID_ARG, f"{name} must be contiguous")


def e8m0_row_bytes(D: int) -> int:
    """Bytes of one row of a TABLE_FP8_E8M0_ROWS table of width D (the row, its
    D/32 exponents, zeros up to a multiple of 16)."""
    return (D + D // 32 + 15) // 16 * 16


@dataclasses.dataclass
class Tables:
    """The three device tables (orders 2, 3, 4) and their scales: fp32 [rows] for
    TABLE_FP8_E4M3FN, uint8 e8m0 exponents [rows, D/32] for TABLE_FP8_E8M0, none
    for TABLE_BF16.  TABLE_FP8_E8M0_ROWS tables are uint8 [rows,
    e8m0_row_bytes(D)] (engram_pack_e8m0_rows) with no scales; their D is the
    widest multiple of 32 whose packed row fills the table's row."""

    dtype: int
    tables: list
    scales: list | None = None

    @property
    def D(self) -> int:
        width = int(self.tables[0].shape[1])
        if self.dtype != TABLE_FP8_E8M0_ROWS:
            return width
        D = width * 32 // 33 // 32 * 32
        while D > 0 and e8m0_row_bytes(D) > width:
            D -= 32
        if D <= 0 or e8m0_row_bytes(D) != width:
            raise EngramError(ERR_INVALID_ARG, f"{width} bytes is no packed e8m0 row width")
        return D

    @property
    def rows(self):
        return [int(t.shape[0]) for t in self.tables]

    def struct(self) -> engram_tables:
        s = engram_tables()
        s.dtype = self.dtype
        s.D = self.D
        for n in range(3):
            s.rows[n] = int(self.tables[n].shape[0])
            s.table[n] = self.tables[n].data_ptr()
            sc = self.scales[n] if self.scales else None
            s.scale[n] = sc.data_ptr() if sc is not None else None
        return s


def engram_pack_e8m0_rows(table, exps, packed=None, stream=None):
    """A TABLE_FP8_E8M0_ROWS table from a TABLE_FP8_E8M0 one: table uint8 [rows, D],
    exps uint8 [rows, D/32] -> uint8 [rows, e8m0_row_bytes(D)] (each row, then its
    exponents, then zeros)."""
    import torch
    _need(table, (torch.uint8,), "table")
    _need(exps, (torch.uint8,), "exps")
    rows, D = table.shape
    if tuple(exps.shape) != (rows, D // 32):
        raise EngramError(ERR_INVALID_ARG, "exps must be [rows, D/32]")
    if packed is None:
        packed = torch.empty((rows, e8m0_row_bytes(D)), dtype=torch.uint8, device=table.device)
    _need(packed, (torch.uint8,), "packed")
    _check(lib.engram_pack_e8m0_rows(_ptr(table), _ptr(exps), rows, D, _ptr(packed),
                                     _stream(stream)), "engram_pack_e8m0_rows")
    return packed


def engram_compress(token_ids, tid2eid, n_eids: int, eids_out=None, status=None, stream=None,
                    dead=None):
    """eids_out[i] = tid2eid[token_ids[i]] (int32, same shape as token_ids); with a
    dead mask (uint8/bool, same shape) dead positions become EID_DEAD."""
    import torch
    _need(token_ids, (torch.int32,), "token_ids")
    _need(tid2eid, (torch.int32,), "tid2eid")
    _need(dead, (torch.uint8, torch.bool), "dead")
    if eids_out is None:
        eids_out = torch.empty_like(token_ids)
    _need(eids_out, (torch.int32,), "eids_out")
    _check(lib.engram_compress_masked(_ptr(token_ids), token_ids.numel(), _ptr(tid2eid),
                                      tid2eid.numel(), n_eids, _ptr(dead), _ptr(eids_out),
                                      _ptr(status), _stream(stream)),
           "engram_compress")
    return eids_out


def engram_bucket_primes(n_layers: int, max_ngram: int, n_heads: int, hash_vocab: int):
    """The released layout's bucket sizes, [n_layers][max_ngram - 1][n_heads] (host ints)."""
    n = n_layers * (max_ngram - 1) * n_heads
    out = (C.c_int64 * n)()
    _check(lib.engram_bucket_primes(n_layers, max_ngram, n_heads, hash_vocab, out),
           "engram_bucket_primes")
    flat = list(out)
    k = max_ngram - 1
    return [[flat[(l * k + i) * n_heads:(l * k + i + 1) * n_heads] for i in range(k)]
            for l in range(n_layers)]


def engram_hash(eids, n_heads: int, rows, history=None, history_out=None, row_ids_out=None,
                status=None, stream=None, positions=None, primes=None):
    """Row ids [B, S, 3, n_heads] int32 for eids [B, S]; history/history_out [B, 3];
    positions [B, S] (optional): each token's index within its packed sample.
    With primes ([3][n_heads] bucket sizes of one layer) the ids index one table
    cut into prime buckets (engram_hash_bucketed) and rows is not used."""
    import torch
    _need(eids, (torch.int32,), "eids")
    if eids.dim() != 2:
        raise EngramError(ERR_INVALID_ARG, "eids must be [batch, seq]")
    B, S = eids.shape
    if row_ids_out is None:
        row_ids_out = torch.empty((B, S, 3, n_heads), dtype=torch.int32, device=eids.device)
    _need(row_ids_out, (torch.int32,), "row_ids_out")
    _need(history, (torch.int32,), "history")
    _need(history_out, (torch.int32,), "history_out")
    _need(positions, (torch.int32,), "positions")
    if primes is not None:
        flat = [int(v) for order in primes for v in order]
        pr = (C.c_int64 * len(flat))(*flat)
        _check(lib.engram_hash_bucketed(_ptr(eids), B, S, _ptr(positions), _ptr(history),
                                        _ptr(history_out), n_heads, pr, _ptr(row_ids_out),
                                        _ptr(status), _stream(stream)), "engram_hash_bucketed")
        return row_ids_out
    r = (C.c_int64 * 3)(*[int(x) for x in rows])
    _check(lib.engram_hash_packed(_ptr(eids), B, S, _ptr(positions), _ptr(history),
                                  _ptr(history_out), n_heads, r, _ptr(row_ids_out), _ptr(status),
                                  _stream(stream)), "engram_hash")
    return row_ids_out


def engram_compress_hash(token_ids, tid2eid, n_eids: int, n_heads: int, rows, history=None,
                         history_out=None, row_ids_out=None, eids_out=None, status=None,
                         stream=None, positions=None, dead=None, primes=None):
    """Compression and hash in one launch: row ids [B, S, 3, n_heads] int32 for token
    ids [B, S]; positions / dead (device) and primes as for engram_forward;
    eids_out (optional, int32 [B, S]) receives the compressed ids."""
    import torch
    _need(token_ids, (torch.int32,), "token_ids")
    _need(tid2eid, (torch.int32,), "tid2eid")
    if token_ids.dim() != 2:
        raise EngramError(ERR_INVALID_ARG, "token_ids must be [batch, seq]")
    B, S = token_ids.shape
    if row_ids_out is None:
        row_ids_out = torch.empty((B, S, 3, n_heads), dtype=torch.int32, device=token_ids.device)
    _need(row_ids_out, (torch.int32,), "row_ids_out")
    _need(eids_out, (torch.int32,), "eids_out")
    _need(history, (torch.int32,), "history")
    _need(history_out, (torch.int32,), "history_out")
    r = None if rows is None else (C.c_int64 * 3)(*[int(x) for x in rows])  # unused with primes
    lay = _layout(positions, dead, primes, host=False)
    _check(lib.engram_compress_hash(_ptr(token_ids), B, S, _ptr(tid2eid), tid2eid.numel(), n_eids,
                                    _ptr(history), _ptr(history_out), n_heads, r, _ref(lay),
                                    _ptr(eids_out), _ptr(row_ids_out), _ptr(status),
                                    _stream(stream)), "engram_compress_hash")
    return row_ids_out


def engram_lookup_fused(row_ids, n_heads: int, tables: Tables, streams_in, alpha,
                        eps: float = 1e-6, streams_out=None, gate_out=None, mem_out=None,
                        status=None, stream=None):
    """The fused gather / mean / gate / add.  streams_in: bf16 [..., 4, D]; returns streams_out."""
    import torch
    _need(row_ids, (torch.int32,), "row_ids")
    bf = (torch.bfloat16, torch.int16)
    _need(streams_in, bf, "streams_in")
    _need(alpha, (torch.float32,), "alpha")
    D = tables.D
    if streams_in.shape[-2:] != (4, D):
        raise EngramError(ERR_INVALID_ARG, f"streams_in must be [..., 4, {D}]")
    T = streams_in.numel() // (4 * D)
    if row_ids.numel() != T * 3 * n_heads:
        raise EngramError(ERR_INVALID_ARG, "row_ids and streams disagree on the token count")
    if streams_out is None:
        streams_out = torch.empty_like(streams_in)
    _need(streams_out, bf, "streams_out")
    _need(gate_out, (torch.float32,), "gate_out")
    _need(mem_out, (torch.float32,), "mem_out")
    s = tables.struct()
    _check(lib.engram_lookup_fused(_ptr(row_ids), T, n_heads, C.byref(s), _ptr(streams_in),
                                   _ptr(streams_out), _ptr(alpha), float(eps), _ptr(gate_out),
                                   _ptr(mem_out), _ptr(status), _stream(stream)),
           "engram_lookup_fused")
    return streams_out


def engram_connection_workspace_bytes(n_tokens: int, n_heads: int, d: int, D: int) -> int:
    return int(lib.engram_connection_workspace_bytes(n_tokens, n_heads, d, D))


def engram_connection(row_ids, n_heads: int, tables: Tables, wkv, streams_in, alpha,
                      eps: float = 1e-6, streams_out=None, workspace=None, gate_out=None,
                      k_out=None, status=None, stream=None):
    """The connection with a wkv projection: rows concatenated, k = wkv e, gate, add.
    wkv: bf16 [D, 3*n_heads*d]; streams_in: bf16 [..., 4, D]; returns streams_out."""
    import torch
    _need(row_ids, (torch.int32,), "row_ids")
    bf = (torch.bfloat16, torch.int16)
    _need(streams_in, bf, "streams_in")
    _need(wkv, bf, "wkv")
    _need(alpha, (torch.float32,), "alpha")
    D = streams_in.shape[-1]
    if streams_in.shape[-2] != 4:
        raise EngramError(ERR_INVALID_ARG, "streams_in must be [..., 4, D]")
    T = streams_in.numel() // (4 * D)
    if row_ids.numel() != T * 3 * n_heads:
        raise EngramError(ERR_INVALID_ARG, "row_ids and streams disagree on the token count")
    if tuple(wkv.shape) != (D, 3 * n_heads * tables.D):
        raise EngramError(ERR_INVALID_ARG, f"wkv must be [{D}, {3 * n_heads * tables.D}]")
    if streams_out is None:
        streams_out = torch.empty_like(streams_in)
    _need(streams_out, bf, "streams_out")
    _need(gate_out, (torch.float32,), "gate_out")
    _need(k_out, (torch.float32,), "k_out")
    need = engram_connection_workspace_bytes(T, n_heads, tables.D, D)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=streams_in.device)
    s = tables.struct()
    _check(lib.engram_connection(_ptr(row_ids), T, n_heads, C.byref(s), _ptr(wkv), D,
                                 _ptr(streams_in), _ptr(streams_out), _ptr(alpha), float(eps),
                                 _ptr(workspace), workspace.numel(), _ptr(gate_out), _ptr(k_out),
                                 _ptr(status), _stream(stream)),
           "engram_connection")
    return streams_out


def engram_concat_rows(row_ids, n_heads: int, tables: Tables, e_out=None, state_out=None,
                       status=None, stream=None):
    """E = the tokens' concatenated rows (bf16 [T, 3*n_heads*d]) and their state
    (uint8 [T]: 0 live, 1 dead, 2 bad).  Returns (E, state)."""
    import torch
    _need(row_ids, (torch.int32,), "row_ids")
    T = row_ids.numel() // (3 * n_heads)
    K = 3 * n_heads * tables.D
    dev = row_ids.device
    if e_out is None:
        e_out = torch.empty((T, K), dtype=torch.bfloat16, device=dev)
    if state_out is None:
        state_out = torch.empty((T,), dtype=torch.uint8, device=dev)
    _need(e_out, (torch.bfloat16, torch.int16), "e_out")
    _need(state_out, (torch.uint8,), "state_out")
    if e_out.numel() != T * K or state_out.numel() != T:
        raise EngramError(ERR_INVALID_ARG, "e_out / state_out sizes")
    s = tables.struct()
    _check(lib.engram_concat_rows(_ptr(row_ids), T, n_heads, C.byref(s), _ptr(e_out),
                                  _ptr(state_out), _ptr(status), _stream(stream)),
           "engram_concat_rows")
    return e_out, state_out


def engram_wkv_project(e, wkv, k_out=None, status=None, stream=None):
    """k = E wkv^T on the tensor cores: e bf16 [T, K], wkv bf16 [D, K] -> k fp32 [T, D]."""
    import torch
    bf = (torch.bfloat16, torch.int16)
    _need(e, bf, "e")
    _need(wkv, bf, "wkv")
    T, K = e.shape
    D = wkv.shape[0]
    if wkv.shape[1] != K:
        raise EngramError(ERR_INVALID_ARG, "e and wkv disagree on K")
    if k_out is None:
        k_out = torch.empty((T, D), dtype=torch.float32, device=e.device)
    _need(k_out, (torch.float32,), "k_out")
    if k_out.numel() != T * D:
        raise EngramError(ERR_INVALID_ARG, "k_out must be [T, D]")
    _check(lib.engram_wkv_project(_ptr(e), T, K, _ptr(wkv), D, _ptr(k_out), _ptr(status),
                                  _stream(stream)), "engram_wkv_project")
    return k_out


def engram_gate_add(k, state, streams_in, alpha, eps: float = 1e-6, streams_out=None,
                    gate_out=None, stream=None):
    """The gate of k against stream 0 and the gated add into the four streams."""
    import torch
    _need(k, (torch.float32,), "k")
    _need(state, (torch.uint8,), "state")
    bf = (torch.bfloat16, torch.int16)
    _need(streams_in, bf, "streams_in")
    _need(alpha, (torch.float32,), "alpha")
    D = streams_in.shape[-1]
    T = streams_in.numel() // (4 * D)
    if k.numel() != T * D or state.numel() != T:
        raise EngramError(ERR_INVALID_ARG, "k / state sizes disagree with the streams")
    if streams_out is None:
        streams_out = torch.empty_like(streams_in)
    _need(streams_out, bf, "streams_out")
    _need(gate_out, (torch.float32,), "gate_out")
    _check(lib.engram_gate_add(_ptr(k), _ptr(state), T, D, _ptr(streams_in), _ptr(streams_out),
                               _ptr(alpha), float(eps), _ptr(gate_out), _stream(stream)),
           "engram_gate_add")
    return streams_out


def engram_read_status(status, stream=None):
    """(code, flags): waits for the stream and reads the device status word."""
    v = C.c_int32(0)
    code = lib.engram_read_status(_ptr(status), C.byref(v), _stream(stream))
    if code not in (OK, ERR_OUT_OF_RANGE, ERR_TIMEOUT):
        _check(code, "engram_read_status")
    return code, int(v.value)


def engram_status_string(code: int) -> str:
    return lib.engram_status_string(code).decode()


def engram_abi_version() -> int:
    return int(lib.engram_abi_version())


def engram_set_projection_kernel(which: int) -> int:
    """PROJECTION_AUTO / PROJECTION_SINGLE / PROJECTION_PAIR for this process; returns the
    previous one."""
    prev = int(lib.engram_set_projection_kernel(which))
    if prev < 0:
        raise EngramError(ERR_INVALID_ARG, f"unknown projection kernel {which}")
    return prev


def engram_set_lookup_kernel(which: int) -> int:
    """LOOKUP_AUTO / LOOKUP_GATHER / LOOKUP_BULK for this process; returns the previous one."""
    prev = int(lib.engram_set_lookup_kernel(which))
    if prev < 0:
        raise EngramError(ERR_INVALID_ARG, f"unknown lookup kernel {which}")
    return prev


def engram_set_wait_limit_ns(ns: int) -> int:
    return int(lib.engram_set_wait_limit_ns(int(ns)))


def engram_debug_withhold_copies(launches: int) -> None:
    lib.engram_debug_withhold_copies(int(launches))


def engram_forward_workspace_bytes(batch: int, seq: int, n_heads: int) -> int:
    return int(lib.engram_forward_workspace_bytes(batch, seq, n_heads))


def engram_forward(token_ids, tid2eid, n_eids: int, n_heads: int, tables: Tables, streams_in,
                   alpha, eps: float = 1e-6, history=None, history_out=None, streams_out=None,
                   workspace=None, status=None, stream=None, positions=None, dead=None,
                   primes=None):
    """compress -> hash -> fused lookup in one call on device tensors; token_ids [B, S].
    positions [B, S] int32 and dead [B, S] uint8 (device) describe a packed batch;
    primes ([3][n_heads] bucket sizes) selects the prime-bucket table layout."""
    import torch
    _need(token_ids, (torch.int32,), "token_ids")
    B, S = token_ids.shape
    if streams_out is None:
        streams_out = torch.empty_like(streams_in)
    need = engram_forward_workspace_bytes(B, S, n_heads)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=token_ids.device)
    s = tables.struct()
    lay = _layout(positions, dead, primes, host=False)
    _check(lib.engram_forward(_ptr(token_ids), B, S, _ptr(tid2eid), tid2eid.numel(), n_eids,
                              _ptr(history), _ptr(history_out), n_heads, C.byref(s), _ref(lay),
                              _ptr(streams_in), _ptr(streams_out), _ptr(alpha), float(eps),
                              _ptr(workspace), workspace.numel(), _ptr(status), _stream(stream)),
           "engram_forward")
    return streams_out


def engram_forward_host_workspace_bytes(batch: int, seq: int, n_heads: int, D: int,
                                        chunk_tokens: int = 0) -> int:
    return int(lib.engram_forward_host_workspace_bytes(batch, seq, n_heads, D, chunk_tokens))


def engram_forward_host(token_ids_host, tid2eid, n_eids: int, n_heads: int, tables: Tables,
                        streams_in_host, streams_out_host, alpha, workspace, eps: float = 1e-6,
                        history=None, history_out=None, chunk_tokens: int = 0, status=None,
                        stream=None, positions=None, dead=None, primes=None):
    """The whole path with host (CPU, ideally pinned) token ids [B, S] and streams
    [B*S, 4, D]; positions / dead, when given, are host tensors too.  workspace is
    a device uint8 tensor of engram_forward_host_workspace_bytes(...) bytes.
    Asynchronous on `stream`."""
    B, S = token_ids_host.shape
    s = tables.struct()
    lay = _layout(positions, dead, primes, host=True)
    _check(lib.engram_forward_host(_ptr(token_ids_host), B, S, _ptr(tid2eid), tid2eid.numel(),
                                   n_eids, _ptr(history), _ptr(history_out), n_heads, C.byref(s),
                                   _ref(lay), _ptr(streams_in_host), _ptr(streams_out_host), _ptr(alpha),
                                   float(eps), chunk_tokens, _ptr(workspace), workspace.numel(),
                                   _ptr(status), _stream(stream)),
           "engram_forward_host")
    return streams_out_host


def engram_connection_host_workspace_bytes(batch: int, seq: int, n_heads: int, d: int, D: int,
                                           chunk_tokens: int = 0) -> int:
    return int(lib.engram_connection_host_workspace_bytes(batch, seq, n_heads, d, D, chunk_tokens))


def engram_connection_host(token_ids_host, tid2eid, n_eids: int, n_heads: int, tables: Tables,
                           wkv, streams_in_host, streams_out_host, alpha, workspace,
                           eps: float = 1e-6, history=None, history_out=None,
                           chunk_tokens: int = 0, status=None, stream=None, positions=None,
                           dead=None, primes=None):
    """The connection's whole path with host (ideally pinned) token ids [B, S] and
    streams [B*S, 4, D] (positions / dead host tensors too); wkv bf16 [D,
    3*n_heads*d] on the device; workspace a device uint8 tensor of
    engram_connection_host_workspace_bytes(...) bytes.  Asynchronous on `stream`."""
    B, S = token_ids_host.shape
    D = int(wkv.shape[0])
    s = tables.struct()
    lay = _layout(positions, dead, primes, host=True)
    _check(lib.engram_connection_host(_ptr(token_ids_host), B, S, _ptr(tid2eid), tid2eid.numel(),
                                      n_eids, _ptr(history), _ptr(history_out), n_heads,
                                      C.byref(s), _ref(lay), _ptr(wkv), D, _ptr(streams_in_host),
                                      _ptr(streams_out_host), _ptr(alpha), float(eps),
                                      chunk_tokens, _ptr(workspace), workspace.numel(),
                                      _ptr(status), _stream(stream)),
           "engram_connection_host")
    return streams_out_host


STATIC_WORKSPACE_BYTES = 16 << 20


def engram_forward_static(token_ids, tid2eid, n_eids: int, n_heads: int, tables: Tables,
                          streams_in, alpha, eps: float = 1e-6, history=None, history_out=None,
                          streams_out=None, status=None, stream=None, positions=None, dead=None,
                          primes=None):
    """engram_forward without a workspace: the library's fixed device array holds
    the ids (for callers that must not allocate device memory; see engram.h)."""
    import torch
    _need(token_ids, (torch.int32,), "token_ids")
    B, S = token_ids.shape
    if streams_out is None:
        streams_out = torch.empty_like(streams_in)
    s = tables.struct()
    lay = _layout(positions, dead, primes, host=False)
    _check(lib.engram_forward_static(_ptr(token_ids), B, S, _ptr(tid2eid), tid2eid.numel(), n_eids,
                                     _ptr(history), _ptr(history_out), n_heads, C.byref(s),
                                     _ref(lay), _ptr(streams_in), _ptr(streams_out), _ptr(alpha), float(eps),
                                     _ptr(status), _stream(stream)),
           "engram_forward_static")
    return streams_out
