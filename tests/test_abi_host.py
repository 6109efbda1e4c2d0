"""The C ABI on the host, without a GPU: the library loads, exports every entry
point include/engram.h declares (and no other engram_ symbol), and argument
errors come back synchronously as ENGRAM_ERR_INVALID_ARG / UNSUPPORTED before
anything touches a device."""
import ctypes as C
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "engram.h")


@pytest.fixture(scope="module")
def eg():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_engram_build", os.path.join(ROOT, "hashed_gram_memory_gb300", "build.py"))
    build = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(build)
    build.build()
    import hashed_gram_memory_gb300 as eg
    return eg


def declared():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"ENGRAM_API\s+[\w\s\*]+?\b(engram_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared()
    for n in ("engram_compress", "engram_compress_masked", "engram_hash", "engram_hash_packed",
              "engram_lookup_fused", "engram_read_status",
              "engram_status_string", "engram_last_error", "engram_abi_version"):
        assert n in names


def test_header_is_plain_c():
    src = open(HEADER).read()
    assert "torch" not in src and "cuda_runtime" not in src and "<c10" not in src
    r = subprocess.run(["gcc", "-std=c99", "-fsyntax-only", "-x", "c", HEADER], capture_output=True,
                       text=True)
    assert r.returncode == 0, r.stderr


def test_library_exports_every_declared_symbol(eg):
    for n in declared():
        assert hasattr(eg.lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", eg.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = sorted({ln.split()[-1] for ln in out.splitlines() if " T engram_" in ln})
    assert exported == declared()


def test_abi_version_and_strings(eg):
    assert eg.engram_abi_version() == 4
    for code in range(6):
        assert eg.engram_status_string(code).startswith("ENGRAM")
    assert "unknown" in eg.engram_status_string(99)


def _tables(dtype=0, D=64, rows=(10, 10, 10), ptr=0x10000, scale=0x20000):
    import hashed_gram_memory_gb300 as eg
    s = eg.engram_tables()
    s.dtype, s.D = dtype, D
    for n in range(3):
        s.rows[n] = rows[n]
        s.table[n] = ptr + n * 0x100000
        s.scale[n] = scale + n * 0x1000 if scale else None
    return s


def test_host_argument_errors(eg):
    L = eg.lib
    INV, UNS = eg.ERR_INVALID_ARG, eg.ERR_UNSUPPORTED
    rows = (C.c_int64 * 3)(5, 5, 5)
    bad_rows = (C.c_int64 * 3)(5, 0, 5)
    p = C.c_void_p(0x1000)
    assert L.engram_compress(p, -1, p, 10, 5, p, None, None) == INV
    assert L.engram_compress(p, 4, None, 10, 5, p, None, None) == INV
    assert L.engram_compress(p, 4, p, 0, 5, p, None, None) == INV
    assert L.engram_compress(C.c_void_p(0x1002), 4, p, 10, 5, C.c_void_p(0x2000), None, None) == INV
    assert L.engram_compress(C.c_void_p(0x1000), 4, p, 10, 5, C.c_void_p(0x1004), None, None) == INV
    assert b"partially" in L.engram_last_error()
    assert L.engram_hash(p, 2, 3, None, None, 0, rows, C.c_void_p(0x9000), None, None) == INV
    assert L.engram_hash(p, 2, 3, None, None, 33, rows, C.c_void_p(0x9000), None, None) == INV
    assert L.engram_hash(p, 2, 3, None, None, 2, bad_rows, C.c_void_p(0x9000), None, None) == INV
    assert L.engram_hash(p, -1, 3, None, None, 2, rows, C.c_void_p(0x9000), None, None) == INV
    assert L.engram_hash(p, 2, 3, None, None, 2, rows, C.c_void_p(0x1008), None, None) == INV
    # history and history_out may be the same buffer, but not partially overlap
    assert L.engram_hash(p, 2, 3, C.c_void_p(0x5000), C.c_void_p(0x5004), 2, rows,
                         C.c_void_p(0x9000), None, None) == INV
    # empty work returns OK without a launch or a device query
    assert L.engram_hash(None, 0, 3, None, None, 2, rows, None, None, None) == eg.OK
    assert L.engram_compress(None, 0, p, 10, 5, None, None, None) == eg.OK

    x, y, a, ids = C.c_void_p(0x100000000), C.c_void_p(0x200000000), C.c_void_p(0x3000), C.c_void_p(0x4000)
    t = _tables()
    assert L.engram_lookup_fused(ids, 8, 0, C.byref(t), x, y, a, 1e-6, None, None, None, None) == INV
    assert L.engram_lookup_fused(ids, 8, 2, None, x, y, a, 1e-6, None, None, None, None) == INV
    for bad in (_tables(D=40), _tables(D=0), _tables(dtype=7), _tables(rows=(10, 0, 10)),
                _tables(ptr=0x10008), _tables(scale=0)):
        assert L.engram_lookup_fused(ids, 8, 2, C.byref(bad), x, y, a, 1e-6, None, None, None,
                                     None) == INV
    assert L.engram_lookup_fused(ids, 8, 2, C.byref(_tables(D=8192)), x, y, a, 1e-6, None, None,
                                 None, None) == UNS
    assert L.engram_lookup_fused(ids, 8, 2, C.byref(t), x, y, a, -1.0, None, None, None, None) == INV
    assert L.engram_lookup_fused(ids, 8, 2, C.byref(t), x, y, a, float("nan"), None, None, None,
                                 None) == INV
    assert L.engram_lookup_fused(ids, 8, 2, C.byref(t), x, y, None, 1e-6, None, None, None,
                                 None) == INV
    assert L.engram_lookup_fused(ids, 8, 2, C.byref(t), C.c_void_p(0x100000008), y, a, 1e-6, None,
                                 None, None, None) == INV
    # streams_out overlapping streams_in without being equal
    assert L.engram_lookup_fused(ids, 8, 2, C.byref(t), x, C.c_void_p(0x100000010), a, 1e-6, None,
                                 None, None, None) == INV
    # BF16 tables do not need scales
    tb = _tables(dtype=1, scale=0)
    assert L.engram_lookup_fused(ids, 0, 2, C.byref(tb), None, None, a, 1e-6, None, None, None,
                                 None) == eg.OK


def test_connection_host_argument_errors(eg):
    """engram_connection and its three stages check their arguments on the host,
    before any device query or launch."""
    L = eg.lib
    INV, UNS, OK = eg.ERR_INVALID_ARG, eg.ERR_UNSUPPORTED, eg.OK
    ids, w, x, y, a = (C.c_void_p(v) for v in (0x4000, 0x8000000, 0x100000000, 0x200000000, 0x3000))
    ws = C.c_void_p(0x300000000)
    e8 = _tables(dtype=2, D=256)
    need = eg.engram_connection_workspace_bytes(100, 8, 256, 4096)
    assert need == 100 * 6144 * 2 + 100 * 4096 * 4 + 256   # E, k, state (256-byte rounded)

    def conn(tb, D=4096, H=8, n=100, wkv=w, xin=x, out=y, alpha=a, eps=1e-6, work=ws, wb=need):
        return L.engram_connection(ids, n, H, C.byref(tb) if tb is not None else None, wkv, D,
                                   xin, out, alpha, eps, work, wb, None, None, None, None)

    assert conn(_tables(dtype=0, D=256)) == UNS            # per-row fp32 scales: not exact in bf16
    assert conn(e8, D=4000) == UNS                         # D not a multiple of 256
    assert conn(e8, D=8448) == UNS                         # D above 8192
    assert conn(_tables(dtype=2, D=48)) == INV             # row width not a multiple of 32
    assert conn(_tables(dtype=1, D=32, scale=0), H=1, n=5) == UNS  # K = 96 not a multiple of 64
    assert conn(None) == INV
    assert conn(e8, H=0) == INV
    assert conn(_tables(dtype=2, D=256, scale=0)) == INV   # e8m0 tables need their exponents
    assert conn(e8, wkv=C.c_void_p(0x8000008)) == INV      # wkv not 16-byte aligned
    assert conn(e8, alpha=None) == INV
    assert conn(e8, eps=float("nan")) == INV
    assert conn(e8, wb=need - 1) == INV                    # short workspace
    assert conn(e8, work=C.c_void_p(0x300000080)) == INV   # workspace not 256-byte aligned
    assert conn(e8, out=C.c_void_p(0x100000010)) == INV    # partial overlap of the streams
    assert conn(e8, n=0, work=None, wb=0) == OK            # nothing to do

    e, k, st = C.c_void_p(0x500000000), C.c_void_p(0x600000000), C.c_void_p(0x7000)
    assert L.engram_concat_rows(ids, 10, 8, C.byref(_tables(dtype=0, D=256)), e, st, None,
                                None) == UNS
    assert L.engram_concat_rows(ids, 10, 8, C.byref(e8), C.c_void_p(0x500000008), st, None,
                                None) == INV
    assert L.engram_concat_rows(ids, 0, 8, C.byref(e8), None, None, None, None) == OK
    assert L.engram_wkv_project(e, 10, 6144, w, 300, k, None, None) == UNS
    assert L.engram_wkv_project(e, 10, 6100, w, 4096, k, None, None) == UNS
    assert L.engram_wkv_project(e, 10, 6144, w, 4096, C.c_void_p(0x600000004), None, None) == INV
    assert L.engram_wkv_project(None, 0, 6144, w, 4096, None, None, None) == OK
    assert L.engram_gate_add(k, st, 10, 4095, x, y, a, 1e-6, None, None) == INV
    assert L.engram_gate_add(k, st, 10, 8208, x, y, a, 1e-6, None, None) == INV
    assert L.engram_gate_add(k, None, 10, 4096, x, y, a, 1e-6, None, None) == INV
    assert L.engram_gate_add(None, None, 0, 4096, None, None, a, 1e-6, None, None) == OK


def test_kernel_selectors(eg):
    """The lookup and projection selectors take their documented values, return
    the previous one, and refuse anything else without changing the setting."""
    for setter, raw, values in ((eg.engram_set_lookup_kernel, eg.lib.engram_set_lookup_kernel,
                                 (eg.LOOKUP_GATHER, eg.LOOKUP_BULK, eg.LOOKUP_AUTO)),
                                (eg.engram_set_projection_kernel,
                                 eg.lib.engram_set_projection_kernel,
                                 (eg.PROJECTION_SINGLE, eg.PROJECTION_PAIR, eg.PROJECTION_AUTO))):
        prev = setter(values[0])
        try:
            assert setter(values[1]) == values[0]
            assert raw(7) == -1 and raw(-3) == -1
            with pytest.raises(eg.EngramError):
                setter(9)
            assert setter(values[2]) == values[1]   # unchanged by the refused values
        finally:
            setter(prev)


def test_forward_decode_host_argument_errors(eg):
    """engram_forward with one token a slot (the fused decode launch) checks its
    arguments on the host like the three calls it replaces."""
    L = eg.lib
    INV, OK = eg.ERR_INVALID_ARG, eg.OK
    tok, m, x, y, a = (C.c_void_p(v) for v in (0x4000, 0x8000, 0x100000000, 0x200000000, 0x3000))
    h = C.c_void_p(0x9000)
    ws = C.c_void_p(0x300000000)
    t = _tables(D=4096)
    need = eg.engram_forward_workspace_bytes(64, 1, 4)

    def fwd(tok=tok, m=m, vocab=100, n_eids=50, hist=h, hist_out=h, x=x, y=y, a=a, eps=1e-6,
            tb=t, batch=64, lay=None):
        return L.engram_forward(tok, batch, 1, m, vocab, n_eids, hist, hist_out, 4,
                                C.byref(tb) if tb is not None else None,
                                C.byref(lay) if lay is not None else None, x, y, a, eps, ws, need,
                                None, None)

    def layout(pos=None, dead=None, primes=None):
        lay = eg.engram_layout()
        lay.positions, lay.dead = pos, dead
        if primes is not None:
            lay._keep = (C.c_int64 * len(primes))(*primes)
            lay.primes = C.cast(lay._keep, C.POINTER(C.c_int64))
        return lay

    assert fwd(tok=None) == INV
    assert fwd(m=C.c_void_p(0x8002)) == INV              # map not 4-byte aligned
    assert fwd(vocab=0) == INV
    assert fwd(n_eids=-1) == INV
    assert fwd(hist_out=C.c_void_p(0x9004)) == INV       # partial overlap with history
    assert fwd(hist_out=C.c_void_p(0x200000010)) == INV  # history_out inside streams_out
    assert fwd(eps=float("nan")) == INV
    assert fwd(a=None) == INV
    assert fwd(y=C.c_void_p(0x100000010)) == INV         # streams overlap partially
    assert fwd(tb=_tables(D=4096, rows=(10, 0, 10))) == INV
    assert fwd(tb=None) == INV
    assert fwd(lay=layout(pos=0xA002)) == INV            # positions not 4-byte aligned
    assert fwd(hist=None, hist_out=C.c_void_p(0xA000), lay=layout(pos=0xA000)) == INV
    assert fwd(lay=layout(primes=[7] * 11 + [0])) == INV  # a bucket of no rows
    assert fwd(lay=layout(primes=[11] * 12)) == INV      # 132 bucket rows > the 10-row tables
    assert fwd(batch=0) == OK                            # nothing to do
    assert fwd(batch=0, tb=_tables(D=4096, rows=(100, 100, 100)),
               lay=layout(pos=0xA000, dead=0xB000, primes=[7] * 12)) == OK


def test_host_buffer_calls_argument_errors(eg):
    """engram_forward_host and engram_connection_host check their arguments,
    workspace and layout before creating copy streams or touching a device."""
    L = eg.lib
    INV, OK = eg.ERR_INVALID_ARG, eg.OK
    tok, m, x, y, a = (C.c_void_p(v) for v in (0x4000, 0x8000, 0x100000000, 0x200000000, 0x3000))
    w = C.c_void_p(0x8000000)
    t = _tables(D=4096)
    e8 = _tables(dtype=2, D=256, rows=(100000, 100000, 100000))
    need_f = eg.engram_forward_host_workspace_bytes(8, 128, 4, 4096, 0)
    need_c = eg.engram_connection_host_workspace_bytes(8, 128, 8, 256, 4096, 0)
    # ids, positions, eids, dead, rows, then three chunk buffers each way (+ the connection's)
    assert need_f == 3 * 4096 + 1024 + 1024 * 12 * 4 + 6 * 2048 * 4 * 4096 * 2
    assert need_c == (3 * 4096 + 1024 + 1024 * 24 * 4 + 6 * 8192 * 4 * 4096 * 2 +
                      eg.engram_connection_workspace_bytes(8192, 8, 256, 4096))
    ws = C.c_void_p(0x300000000)

    def fh(tok=tok, tb=t, work=ws, wb=need_f, chunk=0, xin=x, lay=None):
        return L.engram_forward_host(tok, 8, 128, m, 100, 50, None, None, 4,
                                     C.byref(tb) if tb is not None else None,
                                     C.byref(lay) if lay is not None else None, xin, y, a, 1e-6,
                                     chunk, work, wb, None, None)

    def ch(tok=tok, tb=e8, work=ws, wb=need_c, chunk=0, xin=x, lay=None, D=4096):
        return L.engram_connection_host(tok, 8, 128, m, 100, 50, None, None, 8,
                                        C.byref(tb) if tb is not None else None,
                                        C.byref(lay) if lay is not None else None, w, D, xin, y,
                                        a, 1e-6, chunk, work, wb, None, None)

    for call, need in ((fh, need_f), (ch, need_c)):
        assert call(tok=None) == INV                      # NULL host ids
        assert call(xin=None) == INV                      # NULL host streams
        assert call(tb=None) == INV
        assert call(work=None) == INV
        assert call(wb=need - 1) == INV                   # short workspace
        assert call(chunk=-1) == INV
        bad = eg.engram_layout()
        bad._keep = (C.c_int64 * 24)(*([0] * 24))
        bad.primes = C.cast(bad._keep, C.POINTER(C.c_int64))
        assert call(lay=bad) == INV                       # buckets of no rows
    assert ch(work=C.c_void_p(0x300000080)) == INV        # not 256-byte aligned
    assert fh(tb=_tables(D=4100)) == INV                  # row width not a multiple of 16
    assert ch(D=0) == INV
    # the lookup's and the connection's own checks run before anything is enqueued
    assert fh(tb=_tables(dtype=7, D=4096)) == INV         # unknown table type
    assert ch(tb=_tables(dtype=0, D=256, rows=(100000,) * 3)) == eg.ERR_UNSUPPORTED
    assert ch(D=4000) == eg.ERR_UNSUPPORTED               # stream width not a multiple of 256


def test_python_binding_rejects_cpu_tensors(eg):
    import torch
    with pytest.raises(eg.EngramError):
        eg.engram_compress(torch.zeros(4, dtype=torch.int32), torch.zeros(4, dtype=torch.int32), 3)


def test_library_bucket_primes_match_oracle_and_pages(eg):
    """engram_bucket_primes is host code: its draw must equal the oracle's and give
    the pages' row counts (384006168 / 384016682; 462)."""
    import oracle
    lib_p = eg.engram_bucket_primes(2, 4, 8, 16_000_000)
    assert [sum(sum(o) for o in layer) for layer in lib_p] == [384006168, 384016682]
    assert sum(sum(o) for o in eg.engram_bucket_primes(1, 4, 2, 64)[0]) == 462
    for args in [(2, 4, 8, 16_000_000), (1, 4, 3, 1000), (3, 5, 2, 97)]:
        assert (oracle.bucket_primes(*args).tolist() == eg.engram_bucket_primes(*args))


def test_ctypes_structs_match_the_header(eg, tmp_path):
    """The binding's engram_tables and engram_layout have the C structs' size and
    field offsets, as gcc lays them out from include/engram.h."""
    import ctypes
    src = tmp_path / "layout.c"
    src.write_text(
        '#include <stddef.h>\n#include <stdio.h>\n#include "engram.h"\n'
        "int main(void) {\n"
        '  printf("%zu %zu %zu %zu %zu %zu\\n", sizeof(engram_tables),\n'
        "         offsetof(engram_tables, D), offsetof(engram_tables, rows),\n"
        "         offsetof(engram_tables, table), offsetof(engram_tables, scale), 0ul);\n"
        '  printf("%zu %zu %zu %zu\\n", sizeof(engram_layout), offsetof(engram_layout, positions),\n'
        "         offsetof(engram_layout, dead), offsetof(engram_layout, primes));\n"
        "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o",
                    str(exe)], check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    t = [int(v) for v in out[0].split()]
    lay = [int(v) for v in out[1].split()]
    T, L = eg.engram_tables, eg.engram_layout
    assert t[:5] == [ctypes.sizeof(T), T.D.offset, T.rows.offset, T.table.offset, T.scale.offset]
    assert lay == [ctypes.sizeof(L), L.positions.offset, L.dead.offset, L.primes.offset]


def test_compress_hash_argument_errors(eg):
    """engram_compress_hash checks the compression's and the hash's arguments on
    the host, before any device query."""
    L = eg.lib
    INV, OK = eg.ERR_INVALID_ARG, eg.OK
    tok, m, rows_out, e_out = (C.c_void_p(v) for v in (0x10000, 0x80000, 0x200000, 0x400000))
    rows = (C.c_int64 * 3)(11, 13, 17)

    def ch(tok=tok, batch=2, seq=8, m=m, vocab=100, n_eids=50, H=2, rows=rows, lay=None,
           e=None, out=rows_out, hist=None, hout=None):
        return L.engram_compress_hash(tok, batch, seq, m, vocab, n_eids, hist, hout, H, rows,
                                      C.byref(lay) if lay is not None else None, e, out, None,
                                      None)

    assert ch(tok=None) == INV
    assert ch(m=None) == INV
    assert ch(vocab=0) == INV
    assert ch(n_eids=-1) == INV
    assert ch(H=0) == INV
    assert ch(rows=(C.c_int64 * 3)(11, 0, 17)) == INV
    assert ch(tok=C.c_void_p(0x10002)) == INV              # misaligned
    assert ch(e=C.c_void_p(0x10008)) == INV                # eids_out over the token ids
    assert ch(e=C.c_void_p(0x200010)) == INV               # eids_out over the row ids
    assert ch(out=C.c_void_p(0x10000)) == INV              # row ids over the token ids
    assert ch(out=C.c_void_p(0x80040)) == INV              # row ids over the map
    assert ch(out=None) == INV
    bad = eg.engram_layout()
    bad._keep = (C.c_int64 * 6)(7, 11, 0, 13, 17, 19)
    bad.primes = C.cast(bad._keep, C.POINTER(C.c_int64))
    assert ch(lay=bad) == INV                             # a bucket of no rows
    assert ch(batch=0) == OK                              # nothing to do
    assert ch(seq=0, tok=None, out=None) == OK


def test_plain_c_program_links_and_runs(eg, tmp_path):
    """tests/c/engram_host_check.c, plain C99 against include/engram.h, links
    against libengram.so and passes its host-only checks (version, strings, the
    bucket draw's 462, argument errors, workspace sizes)."""
    exe = tmp_path / "engram_host_check"
    pkg = os.path.dirname(eg.LIB_PATH)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c", "engram_host_check.c"), "-o", str(exe),
                    "-L", pkg, "-lengram", "-Wl,-rpath," + pkg],
                   check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "FAIL" not in r.stdout and r.stdout.count("ok") >= 9



def test_rows_layout_and_packing_argument_errors(eg):
    """Tables whose rows carry their e8m0 exponents, and engram_pack_e8m0_rows:
    every argument error returns before a launch."""
    L = eg.lib
    INV = eg.ERR_INVALID_ARG
    x, y, a, ids = C.c_void_p(0x100000000), C.c_void_p(0x200000000), C.c_void_p(0x3000), C.c_void_p(0x4000)
    # D % 32 != 0 is refused; a rows-layout table needs no scales (an empty call is OK)
    bad = _tables(dtype=eg.TABLE_FP8_E8M0_ROWS, D=48, scale=0)
    assert L.engram_lookup_fused(ids, 8, 2, C.byref(bad), x, y, a, 1e-6, None, None, None, None) == INV
    assert b"32" in L.engram_last_error()
    ok = _tables(dtype=eg.TABLE_FP8_E8M0_ROWS, D=256, scale=0)
    assert L.engram_lookup_fused(ids, 0, 2, C.byref(ok), None, None, a, 1e-6, None, None, None,
                                 None) == eg.OK
    # the rows-layout macro and the binding agree
    assert [eg.e8m0_row_bytes(D) for D in (32, 256, 4096)] == [48, 272, 4224]
    p, e, q = C.c_void_p(0x10000), C.c_void_p(0x80000), C.c_void_p(0x100000)
    assert L.engram_pack_e8m0_rows(p, e, 10, 48, q, None) == INV          # D % 32
    assert L.engram_pack_e8m0_rows(p, e, 10, 8192, q, None) == INV        # D > ENGRAM_MAX_D
    assert L.engram_pack_e8m0_rows(p, e, -1, 256, q, None) == INV         # rows < 0
    assert L.engram_pack_e8m0_rows(None, e, 10, 256, q, None) == INV      # NULL table
    assert L.engram_pack_e8m0_rows(p, e, 10, 256, C.c_void_p(0x100008), None) == INV  # misaligned
    assert L.engram_pack_e8m0_rows(p, e, 10, 256, C.c_void_p(0x10100), None) == INV   # overlaps table
    assert b"overlaps" in L.engram_last_error()
    assert L.engram_pack_e8m0_rows(None, None, 0, 256, None, None) == eg.OK  # nothing to do
