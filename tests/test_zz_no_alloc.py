"""engram_forward_static, the entry point for callers that cannot allocate device
memory (it keeps its ids in the library's fixed device array instead of a
caller workspace), against engram_forward on the same inputs, on two calls in a
row with different shapes.  It goes through the C ABI directly with ctypes.
This file is collected last on purpose."""
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


def _static_call(eg, cfg, dev, out, status, stream):
    B, S = dev["ids"].shape
    tb = dev["tables"].struct()
    lay = eg._layout(dev.get("positions"), dev.get("dead"), None, host=False)
    return eg.lib.engram_forward_static(
        _p(dev["ids"]), B, S, _p(dev["tid2eid"]), dev["tid2eid"].numel(), cfg.n_eids,
        _p(dev["history"]), None, cfg.H, C.byref(tb), None if lay is None else C.byref(lay),
        _p(dev["streams"]), _p(out), _p(dev["alpha"]), float(cfg.eps), _p(status),
        C.c_void_p(stream.cuda_stream))


def test_static_entry_point_matches_forward_on_two_calls(eg):
    import torch
    cases = [W.by_name("full_prefill_fp8").scaled(B=2, S=517, rows=(6007, 6011, 6029)),       # prefill, 8 heads
             W.by_name("decode_fp8").scaled(B=300, rows=(7001, 7013, 7019)),           # decode with history
             W.by_name("packed_mm_fp8").scaled(B=2, S=300, rows=(6007, 6011, 6029),    # packed, dead spans
                                               mean_sample_len=40, image_span=8, image_frac=0.3)]
    stream = torch.cuda.Stream()
    for i, cfg in enumerate(cases):
        inp = P.host_inputs(cfg, rank=i)
        dev = P.to_device(inp)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = torch.full_like(dev["streams"], 0x7777)
        with torch.cuda.stream(stream):
            code = _static_call(eg, cfg, dev, out, status, stream)
            assert code == eg.OK, eg.lib.engram_last_error()
            ref = eg.engram_forward(dev["ids"], dev["tid2eid"], cfg.n_eids, cfg.H, dev["tables"],
                                    dev["streams"], dev["alpha"], cfg.eps, history=dev["history"],
                                    positions=dev["positions"], dead=dev["dead"])
        stream.synchronize()
        assert eg.engram_read_status(status)[1] == 0
        got = out.cpu().numpy().view(np.uint16)
        want = ref.cpu().numpy().view(np.uint16)
        P.compare_streams(got, want, inp.streams, what=f"static call {i}")
        assert np.array_equal(got, want)


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
