"""engram_forward_static: engram_forward for callers that cannot allocate device
memory (a plugin handed only its input and output buffers, a runtime whose pool
forbids outside allocations, code that must not allocate after start-up).  It
keeps its ids in the library's fixed device array instead of a caller
workspace.  Checked here through the C ABI with ctypes: a zero-token warm-up
call does the per-device set-up; then two calls in a row (and a third of
another kind) give the same streams and history as engram_forward and as the
oracle, and neither torch's allocator nor the device's free memory moves while
they run.  This file is collected last on purpose."""
import ctypes as C

import numpy as np
import pytest

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


def _p(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _static_call(eg, cfg, dev, out, status, stream, history_out=None):
    B, S = dev["ids"].shape
    tb = dev["tables"].struct()
    lay = eg._layout(dev.get("positions"), dev.get("dead"), None, host=False)
    return eg.lib.engram_forward_static(
        _p(dev["ids"]), B, S, _p(dev["tid2eid"]), dev["tid2eid"].numel(), cfg.n_eids,
        _p(dev["history"]), _p(history_out), cfg.H, C.byref(tb),
        None if lay is None else C.byref(lay), _p(dev["streams"]), _p(out), _p(dev["alpha"]),
        float(cfg.eps), _p(status), C.c_void_p(stream.cuda_stream))


def _warm_up(eg, stream):
    """A call of no tokens: looks up the array's device address on this device
    (the set-up a caller makes once at start-up, outside any stream capture)
    and launches nothing."""
    import torch
    cfg = W.by_name("tiny_fp8_d256")
    dev = dict(ids=torch.zeros((0, 1), dtype=torch.int32, device="cuda"),
               tid2eid=torch.ones(cfg.vocab, dtype=torch.int32, device="cuda"), history=None,
               streams=torch.zeros((0, 1, 4, cfg.D), dtype=torch.int16, device="cuda"),
               alpha=torch.zeros(4, dtype=torch.float32, device="cuda"),
               tables=eg.Tables(eg.TABLE_FP8_E4M3FN,
                                [torch.zeros((r, cfg.D), dtype=torch.uint8, device="cuda")
                                 for r in (5, 5, 5)],
                                [torch.ones(5, dtype=torch.float32, device="cuda")] * 3))
    code = _static_call(eg, cfg, dev, dev["streams"], None, stream)
    assert code == eg.OK, eg.lib.engram_last_error()
    stream.synchronize()


CASES = [W.by_name("full_prefill_fp8").scaled(B=2, S=517, rows=(6007, 6011, 6029)),   # prefill, 8 heads
         W.by_name("decode_fp8").scaled(B=300, rows=(7001, 7013, 7019)),             # decode + history
         W.by_name("packed_mm_fp8").scaled(B=2, S=300, rows=(6007, 6011, 6029),      # packed, dead spans
                                           mean_sample_len=40, image_span=8, image_frac=0.3)]


def test_static_entry_point_matches_forward_and_oracle_without_allocating(eg):
    import torch
    stream = torch.cuda.Stream()
    _warm_up(eg, stream)
    # Inputs, outputs and engram_forward's reference results are made first:
    # the static calls below must then leave device memory as they found it.
    runs = []
    for i, cfg in enumerate(CASES):
        inp = P.host_inputs(cfg, rank=i)
        dev = P.to_device(inp)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = [torch.full_like(dev["streams"], 0x7777) for _ in range(2)]
        hist = ([torch.full_like(dev["history"], -7) for _ in range(2)]
                if dev["history"] is not None else [None, None])
        ref_hist = torch.full_like(dev["history"], -7) if dev["history"] is not None else None
        with torch.cuda.stream(stream):
            ref = eg.engram_forward(dev["ids"], dev["tid2eid"], cfg.n_eids, cfg.H, dev["tables"],
                                    dev["streams"], dev["alpha"], cfg.eps, history=dev["history"],
                                    history_out=ref_hist, positions=dev["positions"],
                                    dead=dev["dead"])
        runs.append((cfg, inp, dev, status, out, hist, ref, ref_hist))
    # one static call of each kind first: its kernels are then loaded on the device
    for cfg, inp, dev, status, out, hist, *_ in runs:
        assert _static_call(eg, cfg, dev, out[0], status, stream, hist[0]) == eg.OK, \
            eg.lib.engram_last_error()
    stream.synchronize()
    torch.cuda.synchronize()
    alloc0 = torch.cuda.memory_allocated()
    free0 = torch.cuda.mem_get_info()[0]
    # two calls in a row of each kind, into fresh outputs
    for cfg, inp, dev, status, out, hist, *_ in runs:
        for k in range(2):
            out[k].fill_(0x7777)
            if hist[k] is not None:
                hist[k].fill_(-7)
        stream.synchronize()
        for k in range(2):
            code = _static_call(eg, cfg, dev, out[k], status, stream, hist[k])
            assert code == eg.OK, eg.lib.engram_last_error()
    stream.synchronize()
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.cuda.mem_get_info()[0] == free0, "device free memory moved during static calls"
    for i, (cfg, inp, dev, status, out, hist, ref, ref_hist) in enumerate(runs):
        assert eg.engram_read_status(status)[1] == 0
        want = ref.cpu().numpy().view(np.uint16)
        orc = P.oracle_path(inp)
        assert orc["flags"] == 0
        for k in range(2):
            got = out[k].cpu().numpy().view(np.uint16)
            assert np.array_equal(got, want), f"static call {i}.{k} differs from engram_forward"
            P.compare_streams(got, orc["streams"], inp.streams, what=f"static call {i}.{k} vs oracle")
            if hist[k] is not None:
                assert np.array_equal(hist[k].cpu().numpy(), ref_hist.cpu().numpy())
                assert np.array_equal(hist[k].cpu().numpy(), orc["history"])


def test_static_entry_point_rejects_oversized_requests(eg):
    import torch
    cfg = W.by_name("full_prefill_fp8").scaled(B=64, S=8192, rows=(11, 13, 17))   # 524,288 tokens at 8 heads
    need = eg.engram_forward_workspace_bytes(cfg.B, cfg.S, cfg.H)
    assert need > eg.STATIC_WORKSPACE_BYTES
    dev = dict(ids=torch.zeros((cfg.B, cfg.S), dtype=torch.int32, device="cuda"),
               tid2eid=torch.zeros(cfg.vocab, dtype=torch.int32, device="cuda"), history=None,
               streams=torch.zeros((1, 4, cfg.D), dtype=torch.int16, device="cuda"),
               alpha=torch.zeros(4, dtype=torch.float32, device="cuda"),
               tables=eg.Tables(eg.TABLE_FP8_E4M3FN,
                                [torch.zeros((r, cfg.D), dtype=torch.uint8, device="cuda")
                                 for r in cfg.rows],
                                [torch.ones(r, dtype=torch.float32, device="cuda") for r in cfg.rows]))
    code = _static_call(eg, cfg, dev, dev["streams"], None, torch.cuda.current_stream())
    assert code == eg.ERR_UNSUPPORTED
    assert b"static workspace" in eg.lib.engram_last_error()
