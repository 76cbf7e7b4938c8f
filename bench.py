#!/usr/bin/env python3
"""Benchmark of the KDA mixer core on GB300.

Prints one JSON line.  The headline is chunked-prefill throughput in tokens
per second per KDA layer on the long K3-shaped workload (B=1, T=32768, H=96,
d=128, bf16 I/O, fp32 state): one step is one kda_prefill call (pre-stage,
recurrence, RMSNormGated epilogue, ring update) over the whole sequence, with
inputs resident in HBM.  Alongside it:
  decode     batched decode of 256 sessions x 32 heads (state GB/s, session*tokens/s)
  e2e        the same prefill from pinned HOST buffers (kda_prefill_host: token
             segments whose host->device copies and device->host read of o overlap
             the kernels), all copies inside the timed region
  roofline   the dominant kernel against the method's own bytes (fused single pass)
  step       the whole step's HBM fraction and tensor-core fraction
  kernels    each kernel's own bytes over its time
  other_prefill  the same for the single-sequence T=4096 H=32 and the varlen H=64 workloads,
                 the long workload with the softplus gate, and the long workload with 8 heads
                 (one sequence whose recurrence runs as segments)
  cpu_baseline  the fp64 oracle on a bounded sample of the same workload

--impl reference times the oracle (the only other implementation) as the
reference arm.  Multi-GPU (torchrun) runs independent replicas: every rank
processes its own copy of the workload (weak scaling, no data-path collective).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import kda_synth  # noqa: E402

D = 128
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ----------------------------------------------------------------- helpers
def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def peaks():
    try:
        with open(PEAKS_FILE) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def source_sha(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def ncu_traffic(kernel: str, src: str, units: float):
    """DRAM bytes of one launch processing `units` (token-heads or session-heads),
    from the committed ncu summary scaled by the units it was captured on, or
    None when the kernel source changed since the counters were taken."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)[kernel]
        if d.get("source_sha") != source_sha(src):
            return None
        return float(d["dram_bytes_per_launch"]) * units / float(d["units"])
    except Exception:
        return None


class Clocks:
    """nvidia-smi sampler for the timed region: started (and its first sample
    awaited) before the region opens; the samples taken while it is open, or
    the one nearest to it when the region is shorter than the period, are
    summarised."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 10   # nvidia-smi kept up with 5 ms on GB300 (590 samples in 3 s)

    def __init__(self, device_index):
        self.proc = None
        self.dev = device_index
        self.lines = []  # (arrival time, line)
        self.t_open = self.t_close = None

    def _reader(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line))

    def __enter__(self):
        import threading
        try:
            try:
                uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
                if not uuid.startswith("GPU-"):
                    uuid = "GPU-" + uuid
            except Exception:
                uuid = None
            sel = uuid or os.environ.get("CUDA_VISIBLE_DEVICES", str(self.dev)).split(",")[self.dev]
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.PERIOD_MS), "-i", sel],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._reader, daemon=True).start()
            deadline = time.monotonic() + 5.0
            while not self.lines and time.monotonic() < deadline and self.proc.poll() is None:
                time.sleep(0.01)
        except Exception:
            self.proc = None
        self.t_open = time.monotonic()
        return self

    def __exit__(self, *exc):
        self.t_close = time.monotonic()
        if self.proc is not None:
            time.sleep(self.PERIOD_MS / 1000 * 1.5)  # the sample that covers the region's end
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    @staticmethod
    def _parse(line):
        parts = [x.strip() for x in line.split(",")]
        if len(parts) < 7:
            return None
        try:
            return float(parts[0]), float(parts[1]), parts[3:7]
        except ValueError:
            return None

    def summary(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        parsed = [(t, self._parse(l)) for t, l in self.lines]
        parsed = [(t, p) for t, p in parsed if p is not None]
        if not parsed or self.t_open is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        # a sample arriving up to one period after the region closed still covers it
        inside = [p for t, p in parsed if self.t_open <= t <= self.t_close + self.PERIOD_MS / 1000]
        if not inside:
            inside = [min(parsed, key=lambda tp: abs(tp[0] - self.t_open))[1]]
        reasons = set()
        for _, _, flags in inside:
            for nm, val in zip(names, flags):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(p[0] for p in inside), "sm_max_mhz": inside[-1][1],
                "reasons": sorted(reasons), "samples": len(inside), "period_ms": self.PERIOD_MS}


def allreduce_max(x: float, world: int) -> float:
    """Maximum of `x` over the ranks (the slowest replica sets the step time)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(units_per_rank: float, ms_max: float, world: int) -> float:
    """Throughput of the whole job: every rank processes its own copy of the
    workload (replicas), timed by the slowest rank."""
    return units_per_rank * world / (ms_max / 1e3)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------- algorithmic bytes
def prestage_bytes_per_token_head(io_bytes, out_bytes):
    # reads q,k,v,z (d each) + b; writes q^,k^,v^ + gate (fp32) + beta
    return 4 * D * io_bytes + io_bytes + 3 * D * out_bytes + 4 * D + 4


def scan_bytes_per_token_head():
    # reads q^,k^,v^, gate (fp32) + beta; writes o_core (fp32)
    return 3 * D * 4 + 4 * D + 4 + 4 * D


REC_BYTES = 70656  # one chunk-head record of operand tiles (kda_chunk_layout.cuh)

# The method's own per-token-head figures for prefill at bf16 I/O, independent of
# how the work is split into kernels:
#  - bytes: a single fused pass must read the raw q, k, v, z, gout rows (d each) and
#    the beta logit and write o (d): 5*256 + 2 + 256 = 1538 B;
#  - flops (64-token chunks): 6 d^2 for Q+S, WS and Kt^T U, plus 5 d C for the five
#    triangular C x C x d products (the useful half): 98304 + 40960 = 139264.
METHOD_BYTES_PER_TOKEN_HEAD = 5 * D * 2 + 2 + D * 2
METHOD_FLOP_PER_TOKEN_HEAD = 6 * D * D + 5 * D * 64


def prep_bytes_per_token_head(io_bytes):
    # reads raw q,k,v (+ the three rows before each 64-token chunk), z and b; writes the record
    return 3 * D * io_bytes * (64 + 3) / 64 + D * io_bytes + io_bytes + REC_BYTES / 64


def chunk_recurrence_bytes_per_token_head(io_bytes):
    # reads the record + gout; writes o
    return REC_BYTES / 64 + 2 * D * io_bytes


def epilogue_bytes_per_token_head(io_bytes):
    # reads o_core (fp32) + gout; writes o
    return 4 * D + 2 * D * io_bytes


def decode_bytes_per_session_head(io_bytes):
    # S read + write (fp32), q,k,v,z,gout + b in, o out, ring read + write
    return 2 * D * D * 4 + 5 * D * io_bytes + io_bytes + D * io_bytes + 2 * 3 * 3 * D * io_bytes


VERIFY_TOKENS = 4  # tokens per session in the verify-round measurement (K = 3 drafted + 1)


def verify_bytes_per_session_head(io_bytes, n_tok):
    # S read + written once; per token q,k,v,z,gout + b in, o out; ring read + written once
    return 2 * D * D * 4 + n_tok * (6 * D * io_bytes + io_bytes) + 2 * 3 * 3 * D * io_bytes


# ------------------------------------------------------------------- arms
PREFILL_WORKLOADS = {"long": 3, "prefill": 2, "varlen": 4}


def prefill_arm(args, dev, world, rank, idx=None, heads=None, steps=None, gate="bounded"):
    import gated_delta_rule_04_gb300 as kda
    idx = PREFILL_WORKLOADS[args.workload] if idx is None else idx
    steps = steps or args.steps
    w = kda_synth.workload(idx, device=dev, H=heads if heads is not None else args.heads)
    H, T, W = w.H, w.total_tokens, w.H * D
    kp = kda.make_params(w.params.conv_w, w.params.A_log, w.params.dt_bias, w.params.norm_w,
                         io_dtype=w.io, algo=args.algo, gate=gate)
    toks = list(w.tokens.fields())
    n = w.n_seqs
    cu = w.cu_seqlens
    S_in = ring_in = None
    if w.warmup_tokens is not None:
        # continuing sessions: state and ring after the warm-up tokens (timing input)
        _, S_in, ring_in = kda.kda_prefill(kp, *w.warmup_tokens.fields(), w.warmup_cu)
    o = torch.empty(T, W, dtype=torch.bfloat16, device=dev)
    S_out = torch.empty(n, H, D, D, device=dev)
    ring_out = torch.empty(n, 3, 3, W, dtype=torch.bfloat16, device=dev)
    ws_bytes = kda.kda_prefill_workspace_bytes(kp, n, T)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(evs=None):
        kda.kda_prefill(kp, *toks, cu, S_in=S_in, S_out=S_out, ring_in=ring_in, ring_out=ring_out, o=o,
                        workspace=ws, stream=stream, stage_events=evs)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    evsets = [[torch.cuda.Event(enable_timing=True) for _ in range(kda.KDA_PREFILL_EVENTS)]
              for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for evs in evsets:  # create the handles outside the timed region
        for e in evs:
            e.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    # the step as a user runs it (kda_prefill picks its schedule: the single
    # pass, or overlapped windows for one long sequence)
    with Clocks(dev.index or 0) as clk:
        start.record(stream)
        for _ in range(steps):
            step()
        end.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    ms = start.elapsed_time(end) / steps
    # each kernel alone: the single pass with events at the stage boundaries
    for _ in range(2):
        step(evsets[0])
    torch.cuda.synchronize()
    for evs in evsets:
        step(evs)
    torch.cuda.synchronize()
    stage_ms = [statistics.mean(evs[i].elapsed_time(evs[i + 1]) for evs in evsets)
                for i in range(kda.KDA_PREFILL_EVENTS - 1)]
    single_ms = statistics.mean(evs[0].elapsed_time(evs[-1]) for evs in evsets)
    ms_max = allreduce_max(ms, world)
    ws_status = kda.kda_workspace_status(ws, stream)
    algo = kda.kda_prefill_algo(kp)
    windows = kda.kda_prefill_windows(kp, n, T, ws_bytes)
    segments = kda.kda_prefill_segments(kp, n, T, ws_bytes)
    # chunked single pass: metadata, prep, recurrence, ring; windows: the windows' metadata, a prep
    # part per window (two from the second on), a recurrence per window and the ring; segments:
    # metadata, prep, two recurrence passes, the scan of the segment maps, ring; scan: metadata,
    # pre-stage, scan, epilogue, ring
    if algo != "chunked":
        per_step = 5
    elif segments:
        per_step = 6
    else:
        per_step = 4 if windows == 1 else 3 * windows + 1
    return dict(w=w, ms=ms, ms_max=ms_max, stage_ms=stage_ms, single_ms=single_ms, windows=windows,
                segments=segments, clocks=clk.summary(), kp=kp, launches=per_step * steps, ws_status=ws_status,
                algo_resolved=algo, gate=gate)


def e2e_arm(args, dev, w, kp):
    """The same prefill from pinned HOST buffers through kda_prefill_host: the
    library copies token segments in, runs them and copies o back, with the
    copies of one segment overlapping the kernels of its neighbours."""
    import gated_delta_rule_04_gb300 as kda
    H, T, W = w.H, w.total_tokens, w.H * D
    host = [t.cpu().pin_memory() for t in w.tokens.fields()]
    o_host = torch.empty(T, W, dtype=torch.bfloat16).pin_memory()
    S_out = torch.empty(w.n_seqs, H, D, D, device=dev)
    ring_out = torch.empty(w.n_seqs, 3, 3, W, dtype=torch.bfloat16, device=dev)
    seg = args.segment
    scratch = torch.empty(kda.kda_prefill_host_scratch_bytes(kp, w.cu_seqlens, seg), dtype=torch.uint8,
                          device=dev)
    stream = torch.cuda.current_stream()
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()

    def step():
        kda.kda_prefill_host(kp, *host, w.cu_seqlens, S_out=S_out, ring_out=ring_out, o=o_host,
                             segment_tokens=seg, scratch=scratch, stream=stream, h2d_stream=h2d, d2h_stream=d2h)

    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(args.steps):
        step()
    end.record(stream)
    torch.cuda.synchronize()
    ms = start.elapsed_time(end) / args.steps
    h2d_bytes = sum(t.numel() * t.element_size() for t in host)
    d2h_bytes = o_host.numel() * o_host.element_size()
    return ms, h2d_bytes, d2h_bytes, kda.kda_workspace_status(scratch, stream)


def decode_arm(args, dev):
    import gated_delta_rule_04_gb300 as kda
    w = kda_synth.workload(1, device=dev)
    kp = kda.make_params(w.params.conv_w, w.params.A_log, w.params.dt_bias, w.params.norm_w,
                         io_dtype=w.io, algo=args.algo)
    # state and ring from 512 warm-up tokens per session (input for timing)
    _, S, ring = kda.kda_prefill(kp, *w.warmup_tokens.fields(), w.warmup_cu)
    toks = list(w.tokens.fields())
    o = torch.empty_like(toks[0])
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        kda.kda_decode(kp, *toks, S, ring, o=o, stream=stream)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    steps = max(args.steps, 20)
    start.record(stream)
    for _ in range(steps):
        kda.kda_decode(kp, *toks, S, ring, o=o, stream=stream)
    end.record(stream)
    torch.cuda.synchronize()
    ms = start.elapsed_time(end) / steps
    n_units = w.n_seqs * w.H
    # a speculative verify round: VERIFY_TOKENS tokens per session in one call, in place
    n = w.n_seqs
    vt = kda_synth.draw_tokens(n * VERIFY_TOKENS, w.H, 1000 + 1 + 300_000, kda_synth.io_dtype(w.io), dev)
    vrounds = [t.reshape(n, VERIFY_TOKENS, *t.shape[1:]).contiguous() for t in vt.fields()]
    vo = torch.empty_like(vrounds[0])
    for _ in range(args.warmup):
        kda.kda_decode_multi(kp, *vrounds, S, ring, o=vo, stream=stream)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        kda.kda_decode_multi(kp, *vrounds, S, ring, o=vo, stream=stream)
    end.record(stream)
    torch.cuda.synchronize()
    vms = start.elapsed_time(end) / steps
    return dict(ms=ms, sessions=w.n_seqs, H=w.H, bytes=n_units * decode_bytes_per_session_head(2), steps=steps,
                verify_ms=vms, verify_bytes=n_units * verify_bytes_per_session_head(2, VERIFY_TOKENS))


def cpu_baseline(args, sample_heads=None, sample_tokens=32768):
    """The fp64 oracle, as it stands, on the long workload or a bounded part
    of it: `sample_heads` heads (default all) x the first `sample_tokens`
    tokens.  The whole workload is about 10 s on 16 host cores."""
    import oracle
    w = kda_synth.workload(3, device="cuda" if torch.cuda.is_available() else "cpu")
    sample_heads = sample_heads or w.H
    heads = list(range(sample_heads))
    sub = kda_synth.Tokens(*[t[:sample_tokens] for t in w.tokens.fields()])
    t0 = time.perf_counter()
    oracle.run_synth(w.params.to("cpu"), sub, [0, sample_tokens], heads=heads)
    dt = time.perf_counter() - t0
    token_heads = sample_heads * sample_tokens
    value = token_heads / w.H / dt  # full-layer tokens/s
    return {"value": value, "unit": "tokens/s/layer", "cores": oracle.default_threads(), "kind": "oracle",
            "sample": (f"{sample_heads} of {w.H} heads x first {sample_tokens} of {w.total_tokens} tokens "
                       f"(fp64, token by token), {dt:.2f} s wall incl. marshalling")}


# -------------------------------------------------------------- reference
REFERENCE_STEP = dict(tokens=2048, heads=16)  # one oracle step: the first heads x tokens of the long workload


def reference_main(args, world, rank):
    if rank != 0:
        return
    import oracle
    n_tok, n_heads = REFERENCE_STEP["tokens"], REFERENCE_STEP["heads"]
    w = kda_synth.workload(3, device="cpu", lens=[n_tok])
    heads = list(range(n_heads))
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.run_synth(w.params, w.tokens, w.cu_seqlens, heads=heads)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    dt = statistics.mean(times)
    value = len(heads) * w.total_tokens / w.H / dt
    sample = f"{n_heads} of {w.H} heads x {n_tok} tokens per step"
    line = {
        "impl": "reference", "metric": "KDA tokens/s/layer (chunked prefill)", "value": value,
        "unit": "tokens/s/layer", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"long prefill B=1 T=32768 H=96 d=128 bf16 inputs (oracle step: {sample})",
                   "global_batch": 1, "seq_len": 32768, "parallelism": "replicas"},
        "cpu_baseline": {"value": value, "unit": "tokens/s/layer", "cores": oracle.default_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s/layer", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def prefill_report(r, hbm, tc, tc_sus, peak_kind):
    """Roofline figures of one prefill measurement.

    roofline: the dominant kernel (largest share of the single pass) against the
      method's own bytes per token-head (a fused single pass: raw q, k, v, z, gout,
      beta in and o out) -- the bytes any implementation must move, whatever its
      kernels -- divided by that kernel's CUDA-event time.
    step: the same bytes and the method's algorithmic flops over the whole step as
      a user runs it: the HBM fraction and the tensor-core fraction (of the
      sustained bf16 peak: the step runs back to back).
    kernels: each kernel's own bytes (what it reads and writes, its intermediates
      included) over its time, as a fraction of the copy bandwidth.
    """
    w = r["w"]
    H, T = w.H, w.total_tokens
    chunked = r["algo_resolved"] == "chunked"
    stage_names = ["prestage", "chunk_prep", "recurrence", "epilogue", "ring"]
    kernels = ["prestage_kernel", "chunk_prep_kernel", "chunk_recurrence_kernel" if chunked else "scan_kernel",
               "epilogue_kernel", "ring_update_kernel"]
    srcs = ["kda_prestage.cu", "kda_chunk_prep.cu", "kda_chunk.cu" if chunked else "kda_scan.cu",
            "kda_epilogue.cu", "kda_prestage.cu"]
    state_bytes = 2 * D * D * 4 * w.n_seqs * H  # S read + written once per (sequence, head)
    own = [0 if chunked else prestage_bytes_per_token_head(2, 4) * T * H,
           prep_bytes_per_token_head(2) * T * H if chunked else 0,
           (chunk_recurrence_bytes_per_token_head(2) if chunked else scan_bytes_per_token_head()) * T * H
           + state_bytes,
           0 if chunked else epilogue_bytes_per_token_head(2) * T * H, 0]
    stage_ms = r["stage_ms"]
    dom = max(range(4), key=lambda i: stage_ms[i])
    method_bytes = METHOD_BYTES_PER_TOKEN_HEAD * T * H + (state_bytes if w.warmup_tokens is not None else 0)
    method_flop = METHOD_FLOP_PER_TOKEN_HEAD * T * H
    achieved = method_bytes / (stage_ms[dom] / 1e3) / 1e9
    src_path = os.path.join(ROOT, "gated_delta_rule_04_gb300", "csrc", srcs[dom])
    roofline = {"bound": "hbm", "kernel": kernels[dom], "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "peak_kind": f"{peak_kind} copy bandwidth",
                "traffic": ncu_traffic(kernels[dom], src_path, T * H),
                "bytes_basis": "method bytes: raw q,k,v,z,gout + beta in, o out (bf16)"
                               + (", S in and out (fp32)" if w.warmup_tokens is not None else ""),
                "algorithmic_bytes_per_launch": method_bytes,
                "bytes_per_token_head": method_bytes / (T * H), "ms_per_launch": stage_ms[dom],
                "timing": "each kernel alone: a second timed pass of the single-pass schedule with CUDA "
                          "events at the stage boundaries on the launching stream",
                "single_pass_ms_per_step": r["single_ms"]}
    step_s = r["ms_max"] / 1e3
    step = {"ms": r["ms_max"],
            "hbm_achieved_gbs": method_bytes / step_s / 1e9, "hbm_frac": method_bytes / step_s / 1e9 / hbm,
            "tflops_algorithmic": method_flop / step_s / 1e12,
            "tensor_frac": method_flop / step_s / 1e12 / tc_sus,
            "tensor_peak_tflops": tc_sus, "tensor_peak_kind": f"{peak_kind} bf16 dense, sustained",
            "flop_per_token_head": METHOD_FLOP_PER_TOKEN_HEAD,
            "bytes_per_token_head": method_bytes / (T * H),
            "tensor_cap_at_hbm_peak": (METHOD_FLOP_PER_TOKEN_HEAD / (method_bytes / (T * H))) * hbm / 1e3 / tc_sus}
    kern = {}
    for i, nm in enumerate(stage_names):
        if stage_ms[i] <= 0 or (i < 4 and own[i] == 0 and i != dom):
            continue
        k = {"ms": stage_ms[i], "share": stage_ms[i] / max(r["single_ms"], 1e-9)}
        if own[i]:
            k.update({"own_bytes_per_token_head": own[i] / (T * H),
                      "own_bytes_frac_of_hbm": own[i] / (stage_ms[i] / 1e3) / 1e9 / hbm})
        kern[kernels[i]] = k
    return {"roofline": roofline, "step": step, "kernels": kern}


def other_workload(args, dev, world, rank, idx, hbm, tc, tc_sus, peak_kind, heads=None, gate="bounded"):
    """A sub-line for another prefill workload: its own value, step and roofline."""
    r = prefill_arm(args, dev, world, rank, idx=idx, heads=heads or kda_synth.WORKLOADS[idx]["H"],
                    steps=max(args.steps, 20), gate=gate)
    w = r["w"]
    rep = prefill_report(r, hbm, tc, tc_sus, peak_kind)
    if r["segments"]:
        schedule = f"{r['segments']} segments (affine maps composed by a scan)"
    else:
        schedule = "single pass" if r["windows"] == 1 else f"{r['windows']} overlapped windows"
    gate_txt = ", softplus gate" if gate == "softplus" else ""
    if gate == "softplus" or r["segments"]:
        # the stored counters are the bounded-gate kernels' in the single pass
        rep["roofline"]["traffic"] = None
    return {"workload": kda_synth.describe(w.idx, w.H) + gate_txt + ", fp32 state", "metric": "KDA tokens/s/layer",
            "value": whole_job_value(w.total_tokens, r["ms_max"], world), "unit": "tokens/s/layer",
            "ms_per_step": r["ms_max"], "steps": max(args.steps, 20), "algo": r["algo_resolved"],
            "schedule": schedule,
            "step": rep["step"], "roofline": rep["roofline"], "kernels": rep["kernels"],
            "clocks": r["clocks"], "workspace_status": r["ws_status"]}, r["launches"]


# ------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--algo", default="auto", choices=["auto", "scan", "chunked"])
    ap.add_argument("--workload", default="long", choices=sorted(PREFILL_WORKLOADS),
                    help="prefill workload of the headline line: long (T=32768, H=96; the default), "
                         "prefill (T=4096, H=32) or varlen (8 sequences, H=64); the others are for profiling")
    ap.add_argument("--gate", default="bounded", choices=["bounded", "softplus"],
                    help="decay gate of the headline prefill (softplus: the unbounded gate, for profiling)")
    ap.add_argument("--heads", type=int, default=None,
                    help="override the head count of the prefill workload (smaller cases for profiling)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--segment", type=int, default=2048,
                    help="tokens per segment of the host-buffer (e2e) prefill")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-other", action="store_true",
                    help="skip the sub-lines of the other prefill workloads (T=4096 H=32; varlen H=64)")
    ap.add_argument("--no-cpu", action="store_true")
    args = ap.parse_args()
    world, rank, local = dist_info()
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        reference_main(args, world, rank)
        return

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    from gated_delta_rule_04_gb300 import build as kbuild
    kbuild.build()

    hbm, tc, tc_sus, peak_kind = peaks()
    r = prefill_arm(args, dev, world, rank, gate=args.gate)
    w = r["w"]
    H, T = w.H, w.total_tokens
    value = whole_job_value(T, r["ms_max"], world)
    rep = prefill_report(r, hbm, tc, tc_sus, peak_kind)
    roofline = rep["roofline"]

    line = {
        "metric": "KDA tokens/s/layer (chunked prefill)", "value": value, "unit": "tokens/s/layer",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms_max"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": kda_synth.describe(w.idx, w.H) + (", softplus gate" if args.gate == "softplus" else "")
                               + ", fp32 state",
                   "global_batch": world * w.n_seqs, "seq_len": T, "heads": H, "algo": r["algo_resolved"],
                   "schedule": (f"{r['segments']} segments (kda_prefill_segments)" if r["segments"] else
                                "single pass" if r["windows"] == 1 else
                                f"{r['windows']} overlapped windows (kda_prefill_windows)"),
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": f"inputs ({sum(t.numel() * t.element_size() for t in w.tokens.fields()) / 1e9:.2f} GB) larger than L2 (129 MB); no flush"},
        "roofline": roofline,
        "step": rep["step"],
        "kernels": rep["kernels"],
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
        "workspace_status": r["ws_status"],
    }
    if not args.no_other and args.heads is None and args.workload == "long":
        # the other prefill workloads, each with its own value and fractions
        line["other_prefill"] = {}
        for name, idx, heads, gate in (("prefill", 2, None, "bounded"), ("varlen", 4, None, "bounded"),
                                       ("long_softplus_gate", 3, None, "softplus"),
                                       ("long_8_heads", 3, 8, "bounded")):
            sub, launches = other_workload(args, dev, world, rank, idx, hbm, tc, tc_sus, peak_kind,
                                           heads=heads, gate=gate)
            line["other_prefill"][name] = sub
    if not args.no_decode:
        dr = decode_arm(args, dev)
        gbs = dr["bytes"] / (dr["ms"] / 1e3) / 1e9
        line["decode"] = {
            "workload": "batched decode: 256 sessions x H=32, d=128, one token each, bf16 I/O, fp32 state from 512 warm-up tokens",
            "value": whole_job_value(dr["sessions"], allreduce_max(dr["ms"], world), world), "unit": "session*tokens/s",
            "ms_per_step": dr["ms"], "steps": dr["steps"],
            "roofline": {"bound": "hbm", "kernel": "decode_kernel", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                         "frac": gbs / hbm, "peak_kind": f"{peak_kind} copy bandwidth",
                         "traffic": ncu_traffic("decode_kernel", os.path.join(ROOT, "gated_delta_rule_04_gb300", "csrc", "kda_decode.cu"),
                                                dr["sessions"] * dr["H"]),
                         "algorithmic_bytes_per_launch": dr["bytes"]},
            "verify": {
                "workload": f"verify round: {VERIFY_TOKENS} tokens per session in one call (kda_decode_multi), "
                            "same sessions and state",
                "value": dr["sessions"] * VERIFY_TOKENS * world / (allreduce_max(dr["verify_ms"], world) / 1e3),
                "unit": "session*tokens/s", "ms_per_step": dr["verify_ms"], "kernel": "decode_round_kernel",
                "hbm_frac": dr["verify_bytes"] / (dr["verify_ms"] / 1e3) / 1e9 / hbm,
                "traffic": ncu_traffic("decode_round_kernel",
                                       os.path.join(ROOT, "gated_delta_rule_04_gb300", "csrc", "kda_decode.cu"),
                                       dr["sessions"] * dr["H"]),
                "algorithmic_bytes_per_launch": dr["verify_bytes"]},
        }
    if not args.no_e2e:
        ms, h2d, d2h, e2e_status = e2e_arm(args, dev, w, r["kp"])
        ms = allreduce_max(ms, world)
        line["e2e"] = {"value": whole_job_value(T, ms, world), "unit": "tokens/s/layer", "ms_per_step": ms,
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "api": f"kda_prefill_host, {args.segment}-token segments", "workspace_status": e2e_status}
    if rank == 0 and world == 1 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(args)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
