"""Benchmark of the Engram hashed n-gram memory lookup on GB300.

One step = the whole hot path over one batch through the C ABI:
engram_compress_hash (compression and hash in one launch) -> engram_lookup_fused.
The default workload is the full-size prefill (batch 8 x seq 8192 = 65,536
tokens, Zipf token ids with 5 % of positions copying an earlier 4-token span, 8
hash heads, three 5,040,000-row FP8 e4m3fn tables of 4096-wide rows with fp32 row
scales = 57.7 GiB, bf16 streams [8, 8192, 4, 4096]), the largest configuration
that fits one GPU; --workload picks another (workloads.py: the mid-size prefill,
a 512-slot decode step, BF16 tables, packed batches, e8m0 block scales, the
released bucket layout, the wkv connection).  Inputs are resident in HBM when
the timed region starts, larger than the 129 MB L2, or rotated among buffers
when a step's streams fit in it.  The K timed steps are captured once into a
CUDA graph (--eager launches them one by one from Python); the timed region
replays that graph back to back until it has lasted at least a second (so the
clock samples taken every 100 ms cover it), each replay of exactly K steps
between CUDA events, and reports the median replay.  CUDA events recorded
inside a second graph time the dominant kernel.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle, timed on host cores

For N > 1 (torchrun, one rank per GPU) every rank holds a replica of the tables
and processes its own batch (weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

DEFAULT_WORKLOAD = "full_prefill_fp8"
METRIC = "Engram fused lookup tokens/s and achieved HBM GB/s (% of GB300 peak), 1 GPU"
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "lookup_fused_traffic.json")
# The timed region replays the K steps until it has lasted this long, so that the
# clock sampler (one sample every 100 ms) sees it.
MIN_TIMED_S = 1.0
REPLAYS_PER_ROUND = 8


def parse():
    ap = argparse.ArgumentParser(description="One JSON line: the Engram step's tokens/s, the "
                                 "dominant kernel against its roofline, end to end through "
                                 "host buffers, and the CPU oracle's throughput.")
    ap.add_argument("--gpus", type=int, default=1,
                    help="ranks (one GPU each, launched by torchrun; replicas, weak scaling)")
    ap.add_argument("--steps", type=int, default=1000, help="K: steps in each timed replay")
    ap.add_argument("--warmup", type=int, default=20, help="untimed steps first (at least 3)")
    ap.add_argument("--impl", default="native", choices=["native", "reference"],
                    help="reference: the CPU oracle alone, on the host cores")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=[c.name for c in W.CONFIGS])
    ap.add_argument("--e2e-steps", type=int, default=10,
                    help="steps of each end-to-end round through host buffers")
    ap.add_argument("--cpu-sample-tokens", type=int, default=32768,
                    help="tokens (whole sequences) the oracle is timed on")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end measurement")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle's timing")
    ap.add_argument("--eager", action="store_true",
                    help="launch every timed step from Python instead of replaying the K steps "
                         "captured in one CUDA graph")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the batch (small cases for ncu captures)")
    ap.add_argument("--rows", type=int, default=0,
                    help="override the rows of each table (small cases for ncu captures)")
    ap.add_argument("--hash-vocab", type=int, default=0,
                    help="override the bucketed layout's hash vocabulary (the table shrinks to "
                         "the sum of its buckets; small cases for ncu captures)")
    ap.add_argument("--lookup-kernel", default="auto", choices=["auto", "gather", "bulk"],
                    help="engram_set_lookup_kernel's choice for the lookup")
    ap.add_argument("--min-timed-s", type=float, default=MIN_TIMED_S,
                    help="replay the K timed steps until the timed region lasts this long")
    return ap.parse_args()


def config_of(name: str, args=None) -> W.EngramConfig:
    cfg = next(c for c in W.CONFIGS if c.name == name)
    if args is not None and args.batch:
        cfg = cfg.scaled(B=args.batch)
    if args is not None and args.rows:
        cfg = cfg.scaled(rows=(args.rows,) * 3)
    if args is not None and args.hash_vocab and cfg.hash_vocab:
        import hashed_gram_memory_gb300 as eg
        total = sum(sum(o) for o in eg.engram_bucket_primes(1, 4, cfg.H, args.hash_vocab)[0])
        cfg = cfg.scaled(hash_vocab=args.hash_vocab, rows=(total,) * 3)
    return cfg


L2_BYTES = 126 * 2**20   # GB300 L2


def step_footprint(cfg: W.EngramConfig) -> int:
    """Bytes a step reads or writes that could stay in L2 from one step to the next:
    the streams in and out, and the table rows (with their scales) its tokens
    select, counted as if every row were distinct."""
    return cfg.T * 4 * cfg.width * 2 * 2 + cfg.T * cfg.R * cfg.row_bytes()


def stream_rotation(cfg: W.EngramConfig, l2_bytes: int = L2_BYTES) -> int:
    """How many separate input sets (token ids, history, streams in and out) the
    timed steps cycle through, so that a step finds neither its streams nor its
    table rows in L2: one when a step's footprint already exceeds twice the L2,
    else enough sets to exceed it.  Each set has its own token ids, so its rows
    are other rows of the tables."""
    per_step = step_footprint(cfg)
    if per_step >= 2 * l2_bytes:
        return 1
    return min(256, -(-2 * l2_bytes // per_step))


def l2_note(cfg: W.EngramConfig, l2_bytes: int = L2_BYTES) -> str:
    per_step = cfg.T * 4 * cfg.width * 2
    rows = cfg.T * cfg.R * cfg.row_bytes()
    n = stream_rotation(cfg, l2_bytes)
    if n == 1:
        return (f"no flush: every input is larger than the {l2_bytes / 2**20:.0f} MiB L2 (tables "
                f"{cfg.table_bytes() / 2**30:.1f} GiB, of which a step gathers "
                f"{rows / 1e9:.3f} GB of rows; streams {per_step / 1e9:.3f} GB read and "
                f"{per_step / 1e9:.3f} GB written per step)")
    return (f"inputs larger than L2 by rotation: a step's streams ({per_step / 1e6:.1f} MB read, as "
            f"many written) and the rows its tokens gather ({rows / 1e6:.1f} MB) fit in the "
            f"{l2_bytes / 2**20:.0f} MiB L2, so the timed steps cycle through {n} separate sets of "
            f"token ids, history, input and output streams ({n * step_footprint(cfg) / 1e6:.0f} MB "
            f"with their rows); tables {cfg.table_bytes() / 2**30:.1f} GiB")


def workload_desc(cfg: W.EngramConfig) -> dict:
    d = {
        "workload": cfg.name,
        "batch": cfg.B, "seq": cfg.S, "tokens_per_step": cfg.T, "hash_heads": cfg.H, "D": cfg.D,
        "table_rows": list(cfg.rows), "table_dtype": cfg.dtype,
        "table_bytes": cfg.table_bytes(), "token_ids": cfg.ids,
        "repeated_4gram_frac": cfg.repeat_frac, "decode_history": cfg.decode,
        "l2": l2_note(cfg),
        "parallelism": "replicas (weak scaling, no data-path collective)",
    }
    if cfg.hidden:
        d.update({"path": "connection: rows concatenated (K = 3H*D), k = wkv e on the tensor "
                          "cores, gate and add into the streams",
                  "hidden": cfg.hidden, "K": cfg.K, "wkv": f"bf16 [{cfg.hidden}, {cfg.K}]"})
    return d


FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def measured_tensor_burst():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if "bf16_tflops" in d:
            return float(d["bf16_tflops"])
    return None


def measured_tensor_peak():
    """Dense bf16 TFLOP/s sustained under the power cap (the projection runs inside
    a seconds-long loop of steps)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if "bf16_tflops_sustained" in d:
            return float(d["bf16_tflops_sustained"]), "measured"
    return FALLBACK_BF16_TFLOPS_SUSTAINED, "fallback"


def recorded_traffic(cfg, kernel: str):
    """Per-launch DRAM bytes of the lookup kernel from the committed ncu summary,
    scaled by tokens, or None when the kernel timed is not the one captured or its
    sources changed since the capture."""
    if kernel not in ("auto", "bulk", "gemm") or not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        d = json.load(f)
    rec = d.get(cfg.name)
    if not rec:
        return None
    h = hashlib.sha256()
    for src in rec["kernel_sources"]:
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    if h.hexdigest() != rec.get("kernel_sources_sha256"):
        return None
    return float(rec["dram_bytes_per_token"]) * cfg.T


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (every 100 ms) of the GPU's clocks and throttle reasons."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device_index: int):
        self.samples = []
        self.proc = None
        sel = []
        try:
            import torch
            props = torch.cuda.get_device_properties(device_index)
            uuid = str(getattr(props, "uuid", ""))
            if uuid:
                sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            sel = []
        cmd = ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits",
               "-lms", "100"] + sel
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [s.split(", ") for (t, s) in self.samples if t0 <= t <= t1]
        rows = [r for r in rows if len(r) == len(self.FIELDS)]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[3 + i].strip() == "Active"})
        pw = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(pw) if pw else None}


# ----------------------------------------------------------------- native arm

def device_inputs(eg, cfg, rank, device):
    import torch
    tabs, scales = W.tables_device(cfg, device)
    dt = {W.FP8: eg.TABLE_FP8_E4M3FN, W.FP8_E8M0: eg.TABLE_FP8_E8M0, W.BF16: eg.TABLE_BF16,
          W.FP8_E8M0_ROWS: eg.TABLE_FP8_E8M0_ROWS}[cfg.dtype]
    hist = W.history(cfg, rank)
    pos, dead = W.packed_layout(cfg, rank) if cfg.packed else (None, None)
    return dict(
        positions=None if pos is None else torch.from_numpy(pos).to(device),
        dead=None if dead is None else torch.from_numpy(dead).to(device),
        ids=torch.from_numpy(W.token_ids(cfg, rank)).to(device),
        tid2eid=torch.from_numpy(W.tid2eid(cfg)).to(device),
        history=None if hist is None else torch.from_numpy(hist).to(device),
        streams=W.streams_device(cfg, device, rank),
        alpha=torch.from_numpy(W.alpha(cfg)).to(device),
        tables=eg.Tables(dt, tabs, scales),
        wkv=W.wkv_device(cfg, device) if cfg.hidden else None,
    )


class Step:
    """Pre-allocated buffers and the C-ABI calls of one step: the compression and
    hash in one launch (engram_compress_hash), then the fused lookup (or the
    connection's three stages); a decode step is the one fused launch of
    engram_forward."""

    def __init__(self, eg, cfg, d, stream):
        import torch
        self.eg, self.cfg, self.d, self.stream = eg, cfg, d, stream
        dev = d["streams"].device
        self.rows = torch.empty((cfg.B, cfg.S, 3, cfg.H), dtype=torch.int32, device=dev)
        self.hist_out = torch.empty_like(d["history"]) if d["history"] is not None else None
        self.out = torch.empty_like(d["streams"])
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.primes = (eg.engram_bucket_primes(1, 4, cfg.H, cfg.hash_vocab)[0]
                       if cfg.hash_vocab else None)
        self.launches = 2
        # One new token a slot: the one-call engram_forward, which runs the decode
        # step as one fused launch (compress, window, hash and lookup).
        self.fused_decode = (cfg.S == 1 and not cfg.hidden and cfg.D % 512 == 0 and
                             args_lookup_kernel() != "gather")
        if self.fused_decode:
            self.ws = torch.empty(max(16, eg.engram_forward_workspace_bytes(cfg.B, cfg.S, cfg.H)),
                                  dtype=torch.uint8, device=dev)
            self.launches = 1
        if cfg.hidden:   # the connection: concat rows, project, gate + add
            self.e = torch.empty((cfg.T, cfg.K), dtype=torch.bfloat16, device=dev)
            self.state = torch.empty((cfg.T,), dtype=torch.uint8, device=dev)
            self.k = torch.empty((cfg.T, cfg.hidden), dtype=torch.float32, device=dev)
            self.launches = 4

    def __call__(self, ev_start=None, ev_end=None, ids=None, x=None, out=None, hist=None):
        eg, cfg, d = self.eg, self.cfg, self.d
        ids = d["ids"] if ids is None else ids
        hist = d["history"] if hist is None else hist
        x = d["streams"] if x is None else x
        out = self.out if out is None else out
        if self.fused_decode:
            if ev_start is not None:
                ev_start.record(self.stream)
            eg.engram_forward(ids, d["tid2eid"], cfg.n_eids, cfg.H, d["tables"], x, d["alpha"],
                              cfg.eps, history=hist, history_out=self.hist_out,
                              streams_out=out, workspace=self.ws, status=self.status,
                              stream=self.stream, positions=d["positions"], dead=d["dead"],
                              primes=self.primes)
            if ev_end is not None:
                ev_end.record(self.stream)
            return
        eg.engram_compress_hash(ids, d["tid2eid"], cfg.n_eids, cfg.H, cfg.rows,
                                history=hist, history_out=self.hist_out,
                                row_ids_out=self.rows, status=self.status, stream=self.stream,
                                positions=d["positions"], dead=d["dead"], primes=self.primes)
        if cfg.hidden:
            eg.engram_concat_rows(self.rows, cfg.H, d["tables"], e_out=self.e,
                                  state_out=self.state, status=self.status, stream=self.stream)
            if ev_start is not None:
                ev_start.record(self.stream)
            eg.engram_wkv_project(self.e, d["wkv"], k_out=self.k, status=self.status,
                                  stream=self.stream)
            if ev_end is not None:
                ev_end.record(self.stream)
            eg.engram_gate_add(self.k, self.state, x, d["alpha"], cfg.eps, streams_out=out,
                               stream=self.stream)
            return
        if ev_start is not None:
            ev_start.record(self.stream)
        eg.engram_lookup_fused(self.rows, cfg.H, d["tables"], x, d["alpha"], cfg.eps,
                               streams_out=out, status=self.status, stream=self.stream)
        if ev_end is not None:
            ev_end.record(self.stream)


def graph_timing_supported() -> bool:
    """Timing events inside a captured graph need torch's external events."""
    import inspect
    import torch
    try:
        return "external" in inspect.signature(torch.cuda.Event.__new__).parameters
    except (TypeError, ValueError):
        return False


_LOOKUP_KERNEL = ["auto"]


def args_lookup_kernel() -> str:
    return _LOOKUP_KERNEL[0]


def run_native(args):
    import torch
    import torch.distributed as dist
    import hashed_gram_memory_gb300 as eg
    from hashed_gram_memory_gb300.replicas import max_over_ranks, whole_job_throughput

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)

    cfg = config_of(args.workload, args)
    _LOOKUP_KERNEL[0] = args.lookup_kernel
    eg.engram_set_lookup_kernel({"auto": eg.LOOKUP_AUTO, "gather": eg.LOOKUP_GATHER,
                                 "bulk": eg.LOOKUP_BULK}[args.lookup_kernel])
    d = device_inputs(eg, cfg, rank, device)
    stream = torch.cuda.Stream(device)
    step = Step(eg, cfg, d, stream)
    torch.cuda.synchronize()

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            step()
    torch.cuda.synchronize()
    code, flags = eg.engram_read_status(step.status, stream)
    if flags:
        raise SystemExit(f"device status flags 0x{flags:x} during warm-up")

    K = args.steps
    # A step whose streams and rows fit in L2 rotates among separate input sets
    # (see stream_rotation): set 0 is the workload's own; set k > 0 has token ids
    # and history drawn as replica rank * 1000 + k draws them, so its rows are
    # others.
    n_rot = stream_rotation(cfg)
    xs_rot = [d["streams"]] + [d["streams"].clone() for _ in range(n_rot - 1)]
    ys_rot = [step.out] + [torch.empty_like(step.out) for _ in range(n_rot - 1)]
    ids_rot = [d["ids"]] + [torch.from_numpy(W.token_ids(cfg, rank * 1000 + k)).to(device)
                            for k in range(1, n_rot)]
    hist_rot = [d["history"]] + [None if d["history"] is None else
                                 torch.from_numpy(W.history(cfg, rank * 1000 + k)).to(device)
                                 for k in range(1, n_rot)]

    def rot(i):
        k = i % n_rot
        return dict(x=xs_rot[k], out=ys_rot[k], ids=ids_rot[k], hist=hist_rot[k])

    # The K timed steps are captured once into a CUDA graph and replayed, so the
    # GPU runs them back to back without waiting on Python between launches.
    # The step throughput comes from a graph of the K steps alone; the dominant
    # kernel's durations from a second replay of the same K steps, captured with
    # CUDA events around each of its launches (external event nodes, which add
    # their own few microseconds to a step and so stay out of the first graph).
    graphed = not args.eager and graph_timing_supported()
    ev_kw = {"enable_timing": True, "external": True} if graphed else {"enable_timing": True}
    ev = [(torch.cuda.Event(**ev_kw), torch.cuda.Event(**ev_kw)) for _ in range(K)]
    graph = graph_ev = None
    if graphed:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(K):
                step(**rot(i))
        graph_ev = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_ev, stream=stream):
            for i in range(K):
                step(ev[i][0], ev[i][1], **rot(i))
        with torch.cuda.stream(stream):
            graph.replay()       # untimed: a graph's first launch uploads it
            graph_ev.replay()
        torch.cuda.synchronize()

    def run_k():
        """Exactly K steps: one replay of the step graph, or K eager steps."""
        if graphed:
            with torch.cuda.stream(stream):
                graph.replay()
        else:
            for i in range(K):
                step(ev[i][0], ev[i][1], **rot(i))

    # The timed region: replays of the K steps back to back, each between CUDA
    # events, in rounds of REPLAYS_PER_ROUND; a round ends with a synchronize
    # (between two replays' events, so no replay's time holds the gap), and
    # rounds go on until the region has lasted --min-timed-s on the wall clock
    # (every rank as long as the slowest).
    clocks = ClockSampler(local) if rank == 0 else None
    time.sleep(0.5 if clocks else 0)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.time()
    rep_ms = []
    while True:
        marks = [torch.cuda.Event(enable_timing=True) for _ in range(REPLAYS_PER_ROUND + 1)]
        marks[0].record(stream)
        for r in range(REPLAYS_PER_ROUND):
            run_k()
            marks[r + 1].record(stream)
        torch.cuda.synchronize()
        rep_ms += [marks[r].elapsed_time(marks[r + 1]) for r in range(REPLAYS_PER_ROUND)]
        more = 1.0 if time.time() - wall0 < args.min_timed_s else 0.0
        if world > 1:
            more = max_over_ranks(more, device)
        if not more:
            break
    wall1 = time.time()
    n_rep = len(rep_ms)
    if graphed:   # the dominant kernel's durations: the same K steps with events
        with torch.cuda.stream(stream):
            graph_ev.replay()
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    ms_total = statistics.median(rep_ms)
    lookup_ms = [a.elapsed_time(b) for a, b in ev]
    ms_total = max_over_ranks(ms_total, device)
    code, flags = eg.engram_read_status(step.status, stream)
    clk = clocks.summary(wall0, wall1) if clocks else None
    if clocks:
        clocks.stop()

    if args.no_e2e:
        e2e = None
    elif cfg.hidden:
        e2e = run_e2e_connection(eg, cfg, step, stream, args.e2e_steps, world, device)
    else:
        e2e = run_e2e(eg, cfg, step, stream, args.e2e_steps, world, device)
    cpu = None if (args.no_cpu_baseline or rank != 0) else cpu_baseline(cfg, d, args.cpu_sample_tokens)

    if rank == 0:
        peak, peak_kind = measured_peaks()
        n_dead = int(d["dead"].sum().item()) if d["dead"] is not None else 0
        # a dead token moves its row ids and a copy of its streams, no table rows
        bytes_dead = cfg.R * 4 + 2 * 4 * cfg.width * 2
        bytes_tok = (cfg.algorithmic_bytes_per_token() * (cfg.T - n_dead) + bytes_dead * n_dead) / cfg.T
        if step.fused_decode:
            # the fused step keeps the row ids on chip and moves a token id, its map
            # entry and the slot's history in and out instead
            bytes_tok += 4 + 4 + 12 + 12 - cfg.R * 4
        lk = statistics.mean(lookup_ms)
        # The dominant kernel's mean duration.  When a step is that one launch
        # (the fused decode step), the timed region's own events hold exactly K
        # back-to-back launches of it: their mean (gaps between launches
        # included) is its duration, without the few microseconds an event node
        # around each launch adds.  Otherwise, the events around its launches.
        if step.launches == 1:
            kernel_ms = ms_total / K
            duration_source = ("timed region's CUDA events / K (each step is this one launch; "
                               "gaps between the K launches included)")
        else:
            kernel_ms = lk
            duration_source = ("CUDA events around each launch (event nodes in a second graph "
                               "replay of the K steps; they add a few microseconds a launch)")
        achieved = bytes_tok * cfg.T / (kernel_ms * 1e-3) / 1e9
        traffic = recorded_traffic(cfg, args.lookup_kernel)
        value = whole_job_throughput(world * cfg.T * K, ms_total * 1e-3)
        if cfg.hidden:
            tpeak, tpeak_kind = measured_tensor_peak()
            flops = cfg.connection_flops_per_token() * (cfg.T - n_dead)
            t_ach = flops / (lk * 1e-3) / 1e12
            roof = {
                "kernel": "engram_wkv_project (wkv_gemm_kernel)",
                "bound": "tensor",
                "achieved": t_ach,
                "peak": tpeak,
                "peak_source": f"{tpeak_kind} (MEASURED_PEAKS.json bf16_tflops_sustained: "
                               "cuBLAS bf16 back to back under the power cap)",
                "unit": "TFLOP/s",
                "frac": t_ach / tpeak,
                "frac_of_burst_peak": (t_ach / measured_tensor_burst()
                                       if measured_tensor_burst() else None),
                "traffic": recorded_traffic(cfg, "gemm"),
                "algorithmic_flops_per_token": cfg.connection_flops_per_token(),
                "flops_per_launch": flops,
                "gemm_shape": [cfg.T, cfg.hidden, cfg.K],
                "projection_ms_mean": lk,
                "projection_ms_median": statistics.median(lookup_ms),
            }
        line = {
            "metric": METRIC,
            "value": value,
            "unit": "tokens/s",
            "n_gpus": world,
            "steps": K,
            "warmup": max(args.warmup, 3),
            "ms_per_step": ms_total / K,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16 x bf16 -> f32 (tensor cores)" if cfg.hidden else "f32",
            "data": "synthetic (seeded; tables and streams generated on the GPU)",
            "config": workload_desc(cfg),
            "hbm_gbs_effective_step": bytes_tok * cfg.T * K / (ms_total * 1e-3) / 1e9,
            "roofline": roof if cfg.hidden else {
                "kernel": ("engram_forward (decode_step_kernel: compress, hash and lookup fused)"
                           if step.fused_decode else "engram_lookup_fused"),
                "lookup_kernel": args.lookup_kernel,
                "bound": "hbm",
                "achieved": achieved,
                "peak": peak,
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, copy bandwidth)",
                "unit": "GB/s",
                "frac": achieved / peak,
                "traffic": traffic,
                "algorithmic_bytes_per_token": bytes_tok,
                "dead_tokens_per_step": n_dead,
                "kernel_ms": kernel_ms,
                "duration_source": duration_source,
                "lookup_ms_mean": lk,
                "lookup_ms_median": statistics.median(lookup_ms),
            },
            "gpu_launches": step.launches * K * n_rep,
            "gpu_launches_per_step": step.launches,
            "replays": n_rep,
            "timed_region_s": sum(rep_ms) * 1e-3,
            "replay_ms": {"min": min(rep_ms), "median": statistics.median(rep_ms),
                          "max": max(rep_ms)},
            "launch_mode": ("one CUDA graph of the K steps (captured, then replayed twice "
                            "untimed); the timed region replays it back to back, each replay of "
                            f"exactly K steps between CUDA events, in rounds of {REPLAYS_PER_ROUND} "
                            "replays with a synchronize between rounds, until the region has "
                            f"lasted {args.min_timed_s:g} s ({n_rep} replays; ms_per_step and value "
                            "from the median replay); the dominant kernel timed in a further "
                            "replay of the same K steps with CUDA events around its launches")
                           if graphed else
                           f"eager, {n_rep} timed runs of K steps (median run; events around "
                           "the dominant kernel)",
            "status_flags": flags,
            "clocks": clk,
        }
        if e2e:
            line["e2e"] = e2e
        if cpu:
            line["cpu_baseline"] = cpu
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


E2E_ROUNDS = 9


def timed_rounds(one, stream, steps, device):
    """Times E2E_ROUNDS rounds of `steps` calls of one() (host timer, a stream
    sync at the end of each round, max over ranks) and returns the median round
    and all rounds: up to four rounds caught by a transient on the host (other
    jobs share the machine's host memory and link; such rounds run at about half
    the speed) do not decide the figure."""
    from hashed_gram_memory_gb300.replicas import max_over_ranks
    rounds = []
    for _ in range(E2E_ROUNDS):
        t0 = time.perf_counter()
        for _ in range(steps):
            one()
        stream.synchronize()
        rounds.append(max_over_ranks(time.perf_counter() - t0, device))
    return statistics.median(rounds), rounds


def host_inputs_pinned(step):
    """Pinned host copies of a step's per-token inputs: token ids, streams, and
    the packed layout's positions and dead mask when the workload has them;
    plus a pinned output buffer and the input bytes they hold."""
    import torch
    d = step.d

    def pin(t):
        return None if t is None else t.cpu().pin_memory()

    h = dict(ids=pin(d["ids"]), positions=pin(d["positions"]), dead=pin(d["dead"]))
    h["x"] = torch.empty(d["streams"].shape, dtype=d["streams"].dtype, pin_memory=True)
    h["x"].copy_(d["streams"])
    h["y"] = torch.empty(d["streams"].shape, dtype=d["streams"].dtype, pin_memory=True)
    h["h2d"] = sum(t.numel() * t.element_size() for k, t in h.items()
                   if k in ("ids", "positions", "dead", "x") and t is not None)
    h["d2h"] = h["y"].numel() * h["y"].element_size()
    return h


def run_e2e(eg, cfg, step, stream, steps, world, device):
    """Same metric through the C ABI with HOST buffers: every step is one
    engram_forward_host call that copies the token ids (with the packed layout's
    positions and dead mask) and the four input streams from pinned host memory,
    runs compress + hash + the fused lookup, and copies the updated streams back
    (chunked, copies overlapped with the lookup), all inside the timed region."""
    import torch
    from hashed_gram_memory_gb300.replicas import whole_job_throughput
    d = step.d
    h = host_inputs_pinned(step)
    ws = torch.empty(eg.engram_forward_host_workspace_bytes(cfg.B, cfg.S, cfg.H, cfg.D, 0),
                     dtype=torch.uint8, device=device)

    def one():
        eg.engram_forward_host(h["ids"], d["tid2eid"], cfg.n_eids, cfg.H, d["tables"], h["x"],
                               h["y"], d["alpha"], ws, cfg.eps, history=d["history"],
                               history_out=step.hist_out, status=step.status, stream=stream,
                               positions=h["positions"], dead=h["dead"], primes=step.primes)

    for _ in range(2):
        one()
    stream.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    dt, rounds = timed_rounds(one, stream, steps, device)
    ok = torch.equal(h["y"].to(device), step.out)   # same result as the device-resident step
    return {"value": whole_job_throughput(world * cfg.T * steps, dt), "unit": "tokens/s",
            "h2d_bytes_per_step": h["h2d"], "d2h_bytes_per_step": h["d2h"], "steps": steps,
            "rounds_tokens_per_s": [whole_job_throughput(world * cfg.T * steps, r) for r in rounds],
            "matches_device_step": bool(ok),
            "how": "engram_forward_host: pinned host ids (+ positions, dead mask) + streams in, "
                   "compress/hash/lookup, streams out; 2048-token chunks, copies overlapped with "
                   "the lookup on two copy streams; host timer around the steps + a final stream "
                   "sync; the median of nine rounds"}


def run_e2e_connection(eg, cfg, step, stream, steps, world, device):
    """The connection through the public API with HOST buffers: every step is one
    engram_connection_host call that copies the token ids and the four input
    streams from pinned host memory, runs compress and hash, then the
    connection (concat, projection, gate + add) chunk by chunk between the
    copies of its streams in and out, all inside the timed region."""
    import torch
    from hashed_gram_memory_gb300.replicas import whole_job_throughput
    d = step.d
    h = host_inputs_pinned(step)
    ws = torch.empty(eg.engram_connection_host_workspace_bytes(cfg.B, cfg.S, cfg.H, cfg.D,
                                                               cfg.hidden, 0),
                     dtype=torch.uint8, device=device)

    def one():
        eg.engram_connection_host(h["ids"], d["tid2eid"], cfg.n_eids, cfg.H, d["tables"],
                                  d["wkv"], h["x"], h["y"], d["alpha"], ws, cfg.eps,
                                  history=d["history"], history_out=step.hist_out,
                                  status=step.status, stream=stream, positions=h["positions"],
                                  dead=h["dead"], primes=step.primes)

    for _ in range(2):
        one()
    stream.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    dt, rounds = timed_rounds(one, stream, steps, device)
    ok = torch.equal(h["y"].to(device), step.out)
    return {"value": whole_job_throughput(world * cfg.T * steps, dt), "unit": "tokens/s",
            "h2d_bytes_per_step": h["h2d"], "d2h_bytes_per_step": h["d2h"], "steps": steps,
            "rounds_tokens_per_s": [whole_job_throughput(world * cfg.T * steps, r) for r in rounds],
            "matches_device_step": bool(ok),
            "how": "engram_connection_host: pinned host ids + streams in, compress / hash, then "
                   "concat / projection / gate + add in 8192-token chunks between the copies of "
                   "their streams in and out (two copy streams, overlapped); host timer around "
                   "the steps + a final stream sync; the median of nine rounds"}


# ----------------------------------------------------------------- CPU oracle

def oracle_sample(cfg, d, n_tokens):
    """Host inputs for the first n_tokens tokens of sequence 0 (self-contained
    windows), with exactly the table rows they need copied back from the device."""
    import torch
    import oracle
    if cfg.decode:
        n = min(n_tokens, cfg.B)
        ids = d["ids"][:n].cpu().numpy()
        hist = d["history"][:n].cpu().numpy()
        x = d["streams"][:n].cpu().numpy().view(np.uint16).reshape(n, 4, cfg.D)
    elif cfg.hidden:   # the first n tokens of sequence 0 (their windows start at position 0)
        n = min(n_tokens, cfg.S)
        ids = d["ids"][:1, :n].cpu().numpy()
        hist = None
        x = d["streams"][0, :n].cpu().numpy().view(np.uint16).reshape(n, 4, cfg.width)
    else:
        nseq = max(1, min(cfg.B, -(-n_tokens // cfg.S)))   # whole sequences: windows self-contained
        n = nseq * cfg.S
        ids = d["ids"][:nseq].cpu().numpy()
        hist = None
        x = d["streams"][:nseq].cpu().numpy().view(np.uint16).reshape(n, 4, cfg.D)
    tid2eid = d["tid2eid"].cpu().numpy()
    dead = None if d["dead"] is None else d["dead"][:ids.shape[0]].cpu().numpy()
    pos = None if d["positions"] is None else d["positions"][:ids.shape[0]].cpu().numpy()
    if dead is not None:
        e, _ = oracle.compress_masked(ids, tid2eid, cfg.n_eids, dead)
    else:
        e, _ = oracle.compress(ids, tid2eid, cfg.n_eids)
    if cfg.hash_vocab:
        r, _ = oracle.hash_bucketed(e, cfg.H, oracle.bucket_primes(1, 4, cfg.H, cfg.hash_vocab)[0],
                                    history=hist, positions=pos)
    else:
        r, _ = oracle.hash_ids(e, cfg.H, cfg.rows, history=hist, positions=pos)
    r = r.reshape(n, -1)
    # full-size host copies are too large: the oracle gets tables holding only the
    # rows the sample needs, with the row ids remapped onto them
    host_tabs, host_scales, remap = [], [], np.empty_like(r)
    for k in range(3):
        cols = slice(k * cfg.H, (k + 1) * cfg.H)
        live = r[:, cols] != oracle.DEAD
        uniq, inv = np.unique(np.where(live, r[:, cols], 0), return_inverse=True)
        remap[:, cols] = np.where(live, inv.reshape(r[:, cols].shape), oracle.DEAD)
        idx = torch.from_numpy(uniq.astype(np.int64)).to(d["tables"].tables[k].device)
        t = d["tables"].tables[k].index_select(0, idx).cpu().numpy()
        t = t.view(np.uint16) if cfg.dtype == W.BF16 else t.view(np.uint8)
        if cfg.dtype == W.FP8_E8M0_ROWS:   # the oracle takes the bytes and the exponents apart
            host_tabs.append(np.ascontiguousarray(t[:, :cfg.D]))
            host_scales.append(np.ascontiguousarray(t[:, cfg.D:cfg.D + cfg.D // 32]))
            continue
        host_tabs.append(t)
        host_scales.append(d["tables"].scales[k].index_select(0, idx).cpu().numpy()
                           if cfg.dtype != W.BF16 else None)
    wkv = d["wkv"].cpu().numpy().view(np.uint16) if cfg.hidden else None
    return dict(ids=ids, hist=hist, tid2eid=tid2eid, x=x, tables=host_tabs, scales=host_scales,
                remap=remap, rows=r, alpha=d["alpha"].cpu().numpy(), n=n, dead=dead, positions=pos,
                wkv=wkv)


def oracle_dtype(cfg):
    import oracle
    return {W.FP8: oracle.FP8, W.FP8_E8M0: oracle.FP8_E8M0, W.FP8_E8M0_ROWS: oracle.FP8_E8M0,
            W.BF16: oracle.BF16}[cfg.dtype]


def time_oracle(cfg, s, repeats=1):
    """Oracle compress + hash + lookup on the sample; returns seconds per pass."""
    import oracle
    t0 = time.perf_counter()
    for _ in range(repeats):
        if s.get("dead") is not None:
            e, _ = oracle.compress_masked(s["ids"], s["tid2eid"], cfg.n_eids, s["dead"])
        else:
            e, _ = oracle.compress(s["ids"], s["tid2eid"], cfg.n_eids)
        if cfg.hash_vocab:
            oracle.hash_bucketed(e, cfg.H, oracle.bucket_primes(1, 4, cfg.H, cfg.hash_vocab)[0],
                                 history=s["hist"], positions=s.get("positions"))
        else:
            oracle.hash_ids(e, cfg.H, cfg.rows, history=s["hist"], positions=s.get("positions"))
        if cfg.hidden:
            oracle.connection(s["remap"], cfg.H, oracle_dtype(cfg), s["tables"], s["scales"],
                              s["wkv"], s["x"], s["alpha"], cfg.eps)
        else:
            oracle.lookup(s["remap"], cfg.H, oracle_dtype(cfg), s["tables"], s["scales"], s["x"],
                          s["alpha"], cfg.eps)
    return (time.perf_counter() - t0) / repeats


CONNECTION_CPU_SAMPLE = 4096
CPU_BASELINE_SECONDS = 10.0   # about this much oracle work is timed (bounded)


def cpu_baseline(cfg, d, n_tokens):
    """The oracle's throughput on a bounded sample of the workload: one untimed
    pass over the sample (warm-up, and its duration), then as many timed passes
    as make about CPU_BASELINE_SECONDS of work (at most 100)."""
    import oracle
    if cfg.hidden:
        n_tokens = min(n_tokens, CONNECTION_CPU_SAMPLE)
    s = oracle_sample(cfg, d, n_tokens)
    first = time_oracle(cfg, s)
    passes = max(1, min(100, int(round(CPU_BASELINE_SECONDS / max(first, 1e-3)))))
    dt = time_oracle(cfg, s, passes)
    what = ("compress + hash + connection (concatenated rows, wkv projection, gate, add)"
            if cfg.hidden else "compress + hash + fused lookup")
    where = "of sequence 0" if cfg.hidden else "(whole sequences)"
    return {"value": s["n"] / dt, "unit": "tokens/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"first {s['n']} tokens {where} of the {cfg.name} batch (same seeded "
                      f"inputs, the rows they need copied from the device): {what} in the fp64 "
                      f"C oracle; {passes} timed passes after one untimed, "
                      f"{dt * passes:.1f} s wall"}


def reference_sample(cfg, n):
    """Host inputs for n tokens of the workload (same distributions, seeded): ids,
    map, streams, and tables holding just the rows those tokens hash to."""
    import oracle
    sub = cfg.scaled(B=1, S=n) if not cfg.decode else cfg.scaled(B=n)
    ids = W.token_ids(sub)
    tid2eid = W.tid2eid(cfg)
    hist = W.history(sub)
    pos, dead = W.packed_layout(sub) if sub.packed else (None, None)
    if dead is not None:
        e, _ = oracle.compress_masked(ids, tid2eid, cfg.n_eids, dead)
    else:
        e, _ = oracle.compress(ids, tid2eid, cfg.n_eids)
    if cfg.hash_vocab:
        r, _ = oracle.hash_bucketed(e, cfg.H, oracle.bucket_primes(1, 4, cfg.H, cfg.hash_vocab)[0],
                                    history=hist, positions=pos)
    else:
        r, _ = oracle.hash_ids(e, cfg.H, cfg.rows, history=hist, positions=pos)
    r = r.reshape(n, -1)
    g = np.random.default_rng([cfg.seed, 99])
    tabs, scs, remap = [], [], np.empty_like(r)
    for k in range(3):
        cols = slice(k * cfg.H, (k + 1) * cfg.H)
        live = r[:, cols] != oracle.DEAD
        uniq, inv = np.unique(np.where(live, r[:, cols], 0), return_inverse=True)
        remap[:, cols] = np.where(live, inv.reshape(r[:, cols].shape), oracle.DEAD)
        x = g.standard_normal((len(uniq), cfg.D), dtype=np.float32)
        if cfg.dtype == W.FP8:
            tabs.append(W._to_e4m3_bytes(x))
            scs.append(g.uniform(cfg.scale_lo, cfg.scale_hi, len(uniq)).astype(np.float32))
        elif cfg.dtype in (W.FP8_E8M0, W.FP8_E8M0_ROWS):   # the oracle reads both alike
            tabs.append(W._to_e4m3_bytes(x))
            scs.append(g.integers(cfg.e8m0_lo, cfg.e8m0_hi + 1, size=(len(uniq), cfg.D // 32))
                       .astype(np.uint8))
        else:
            tabs.append(W._to_bf16_bits(x * np.float32(cfg.bf16_std)))
            scs.append(None)
    return dict(ids=ids, hist=hist, tid2eid=tid2eid, x=W.streams_host(sub).reshape(n, 4, cfg.width),
                tables=tabs, scales=scs, remap=remap, alpha=W.alpha(cfg), n=n, dead=dead,
                positions=pos, wkv=W.wkv_host(cfg) if cfg.hidden else None)


def run_reference(args, budget_s: float = 60.0):
    """The oracle as it stands on the host cores (rank 0 only), same metric.  Each
    of the K timed steps runs a bounded sample of the workload, sized from a
    warm-up pass so that the K steps take about budget_s seconds."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    cfg = config_of(args.workload, args)
    K = max(1, args.steps)
    probe = reference_sample(cfg, min(256, cfg.T))
    rate = probe["n"] / time_oracle(cfg, probe)
    n = int(max(16, min(cfg.T, 32768, budget_s * rate / K)))
    s = reference_sample(cfg, n)
    for _ in range(max(args.warmup, 3)):
        time_oracle(cfg, s)
    t0 = time.perf_counter()
    for _ in range(K):
        time_oracle(cfg, s)
    dt = (time.perf_counter() - t0) / K
    value = n / dt
    line = {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": K,
        "warmup": max(args.warmup, 3), "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": workload_desc(cfg),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": f"each step: {n} of the {cfg.T} tokens of {cfg.name} through the "
                                   "fp64 C oracle (compress + hash + "
                                   + ("connection with the wkv projection" if cfg.hidden
                                      else "fused lookup")
                                   + "), with tables holding the rows those tokens need"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
