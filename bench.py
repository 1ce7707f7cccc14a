"""Benchmark of the routed-expert GEMV path on GB300.

One step = one token through the 8-expert Q4 decode (d_model 4096, d_ff 1536,
group 64): the fused gate/up of all 8 experts in one grouped C-ABI call, then
their down projections in a second (smoe_experts_gate_up_q4 /
smoe_experts_down_q4), captured into a CUDA graph and replayed.  The same
step as 16 single-expert calls is timed alongside (`per_expert_calls`).
The metric is effective HBM bandwidth, (packed codes + scales + x + out
bytes) / device time, and the time per 8-expert FFN.  Weights rotate over
several copies whose total is far larger than L2, so every step reads its
weights from HBM.

Printed: one JSON line (rank 0).  Besides the contract keys it carries the
roofline of the dominant kernel, the end-to-end figure through host buffers,
the oracle timed on the host cores, sampled clocks, and `rows`: the other
rows of the hot path (Q2 decode, bf16 matvec shapes, token batch, the small
256/256 expert) each timed the same way.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--no-rows] [--no-cpu] [--rows PATTERN] [--rows-only]
"""
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import smoe_inputs as inp  # noqa: E402

METRIC = "effective HBM GB/s (and % of GB300 peak) per GEMV; µs per 8-expert Q4 FFN"
D_MODEL, D_FF, GROUP, N_EXPERTS = 4096, 1536, 64, 8
L2_BYTES = 129 * 1024 * 1024
WORKLOAD = (f"q4_8expert_decode: 8 experts x (gate/up [{D_FF},{D_MODEL}] + down [{D_MODEL},{D_FF}]), "
            f"Q4 group {GROUP}, f32 scales, one f32 token")


def q_bytes(bits, rows, cols, group):
    return rows * cols * bits // 8 + rows * (cols // group) * 4


def expert_bytes(bits, d_model=D_MODEL, d_ff=D_FF, group=GROUP):
    return 2 * q_bytes(bits, d_ff, d_model, group) + q_bytes(bits, d_model, d_ff, group)


def step_bytes(bits, n_experts=N_EXPERTS, d_model=D_MODEL, d_ff=D_FF, group=GROUP):
    """Algorithmic bytes of one token through n experts: every expert's codes
    and scales, x once, the [n, d_model] outputs (hidden not counted)."""
    return n_experts * expert_bytes(bits, d_model, d_ff, group) + d_model * 4 + n_experts * d_model * 4


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock/throttle sampling while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [c.strip() for c in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------ distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world, dev=None):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_step, steps, world, seconds):
    """Whole-job throughput: every rank runs `steps` steps of `bytes_per_step`
    (weak scaling); `seconds` is the slowest rank's time (max_over_ranks)."""
    return bytes_per_step * steps * world / seconds / 1e9


# ------------------------------------------------------------ the GPU arm

class DecodeWorkload:
    """n_copies independent sets of 8 experts (bits = 4 or 2) resident on the
    device, one captured graph per copy, plus the token and outputs."""

    def __init__(self, smoe, dev, bits, seed, n_copies, grouped=False, fused=False):
        import torch
        self.smoe, self.dev, self.bits, self.grouped, self.fused = smoe, dev, bits, grouped, fused
        self.ffn = smoe.smoe_experts_ffn_q4 if bits == 4 else smoe.smoe_experts_ffn_q2
        self.gate_up = smoe.smoe_gate_up_q4 if bits == 4 else smoe.smoe_gate_up_q2
        self.down = smoe.smoe_down_q4 if bits == 4 else smoe.smoe_down_q2
        self.g_gate_up = smoe.smoe_experts_gate_up_q4 if bits == 4 else smoe.smoe_experts_gate_up_q2
        self.g_down = smoe.smoe_experts_down_q4 if bits == 4 else smoe.smoe_experts_down_q2
        self.copies = []
        for c in range(n_copies):
            ex = []
            for e in range(N_EXPERTS):
                h = inp.expert(bits, D_MODEL, D_FF, GROUP, seed + 1000 * c, e)
                ex.append({k: torch.from_numpy(v).to(dev) for k, v in h.items()})
            self.copies.append(ex)
        self.x = torch.from_numpy(inp.activations(D_MODEL, seed)).to(dev)
        self.hidden = torch.empty((N_EXPERTS, D_FF), device=dev)
        self.out = torch.empty((N_EXPERTS, D_MODEL), device=dev)
        # workspace of the one-call path: counters (zero) + hidden
        self.ws_bytes = smoe.smoe_experts_ffn_workspace_bytes(N_EXPERTS, D_FF)
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.stream = torch.cuda.Stream(device=dev)
        self.graphs = []

    def calls(self, c, stream):
        if self.fused:
            ex = self.copies[c]
            self.ffn(*[[t[k] for t in ex] for k in ("gate_codes", "gate_scales", "up_codes", "up_scales",
                                                    "down_codes", "down_scales")],
                     self.x, self.out, D_MODEL, D_FF, GROUP, self.ws, self.ws_bytes, stream=stream)
            return
        if self.grouped:
            ex = self.copies[c]
            self.g_gate_up([t["gate_codes"] for t in ex], [t["gate_scales"] for t in ex],
                           [t["up_codes"] for t in ex], [t["up_scales"] for t in ex], self.x, self.hidden,
                           D_FF, D_MODEL, GROUP, stream=stream)
            self.g_down([t["down_codes"] for t in ex], [t["down_scales"] for t in ex], self.hidden, self.out,
                        D_MODEL, D_FF, GROUP, stream=stream)
            return
        for i, t in enumerate(self.copies[c]):
            self.gate_up(t["gate_codes"], t["gate_scales"], t["up_codes"], t["up_scales"], self.x,
                         self.hidden[i], D_FF, D_MODEL, GROUP, stream=stream)
            self.down(t["down_codes"], t["down_scales"], self.hidden[i], self.out[i], D_MODEL, D_FF,
                      GROUP, stream=stream)

    def capture(self):
        """One graph per copy (one step each) and one graph for a whole
        rotation (len(copies) steps), so that host-side replay cost stays far
        below the device time of the steps it launches."""
        import torch
        s = self.stream
        with torch.cuda.stream(s):
            for c in range(len(self.copies)):
                self.calls(c, s)
        s.synchronize()
        for c in range(len(self.copies)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                self.calls(c, s)
            self.graphs.append(g)
        self.cycle = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.cycle, stream=s):
            for c in range(len(self.copies)):
                self.calls(c, s)
        s.synchronize()

    def run(self, steps):
        """`steps` consecutive steps, each on the next weight copy."""
        import torch
        n = len(self.copies)
        with torch.cuda.stream(self.stream):
            for _ in range(steps // n):
                self.cycle.replay()
            for i in range(steps % n):
                self.graphs[i].replay()


def hold_stream(stream, launches):
    """Enqueues a spin kernel (about 2 ms + 100 us per launch to follow) so
    that the launches enqueued after it wait on the device, not on the host:
    the events around them then time device work only (the blocking-kernel
    method of GPU benchmarking harnesses).  Not used for end-to-end timing."""
    import torch
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(4e6 + 2e5 * launches))


def time_steps(fn, steps, stream, hold=0):
    """Device time of fn(steps) between two events on `stream`; hold > 0:
    the stream is held (hold_stream) for that many launches first."""
    import torch
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if hold:
        hold_stream(stream, hold)
    e0.record(stream)
    fn(steps)
    e1.record(stream)
    e1.synchronize()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1000.0


def kernel_alone_seconds(launch, n, stream):
    """Average device time of one launch, each bracketed by its own events.
    A spin kernel holds the stream while the n launches are enqueued, so the
    device never waits on the host between an event and its launch (a C-ABI
    call through ctypes takes longer to enqueue than the kernel runs)."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    torch.cuda.synchronize()
    hold_stream(stream, n)
    with torch.cuda.stream(stream):
        for i, (a, b) in enumerate(evs):
            a.record(stream)
            launch(i)
            b.record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs) / n / 1000.0


def kernel_chain_seconds(launch, n, stream, reps=20):
    """Average device time of one launch in a CUDA graph of n back-to-back
    launches (as in a decode step, where each launch follows another kernel
    with programmatic dependent launch), timed with events over `reps`
    replays of the graph."""
    import torch
    with torch.cuda.stream(stream):
        for i in range(n):
            launch(i)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(n):
            launch(i)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        t = time_steps(lambda k: [g.replay() for _ in range(k)], reps, stream)
    return t / (reps * n)


def roofline_traffic(kernel_name):
    """dram read+write bytes per launch from the committed ncu summary, only
    while the kernel sources still hash to the value the counters were taken at."""
    try:
        with open(os.path.join(ROOT, "profiles", "roofline_traffic.json")) as f:
            rec = json.load(f).get(kernel_name)
    except Exception:
        return None
    if not rec:
        return None
    h = hashlib.sha256()
    for rel in rec["sources"]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return rec["traffic_bytes"] if h.hexdigest() == rec["sha256"] else None


def gpu_arm(args, rank, world, local):
    import torch
    import __graft_entry__
    __graft_entry__.build_library()
    import moe_expert_ffn_smoe_gb300 as smoe

    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    n_copies = max(2, -(-4 * L2_BYTES // step_bytes(4)))  # working set >= 4x L2
    wl = DecodeWorkload(smoe, dev, 4, 5, n_copies, grouped=True)
    wl.capture()
    wl.run(max(3, args.warmup))
    wl.stream.synchronize()
    # the same step as 16 single-expert calls (8 x gate/up + down)
    calls = DecodeWorkload(smoe, dev, 4, 5, 0, grouped=False)
    calls.copies = wl.copies
    calls.x, calls.hidden, calls.out = wl.x, wl.hidden, wl.out
    calls.capture()
    calls.run(max(3, args.warmup))
    calls.stream.synchronize()
    # the same step as one call (smoe_experts_ffn_q4: one launch)
    one = DecodeWorkload(smoe, dev, 4, 5, 0, fused=True)
    one.copies = wl.copies
    one.x, one.out = wl.x, wl.out
    one.capture()
    one.run(max(3, args.warmup))
    one.stream.synchronize()

    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.2)
    # the stream is held while the steps' graph replays are enqueued, so the
    # events time the device work of the K steps, not the host's submission
    replays = args.steps // len(wl.copies) + args.steps % len(wl.copies)
    t = time_steps(lambda k: wl.run(k), args.steps, wl.stream, hold=replays)
    clock_rec = clocks.stop()
    # the same K steps submitted without the hold (host enqueue gaps included)
    t_unheld = max_over_ranks(time_steps(lambda k: wl.run(k), args.steps, wl.stream), world, dev)
    barrier(world)
    t = max_over_ranks(t, world, dev)
    # distribution: each replay of the rotation graph (len(copies) steps back
    # to back, as in the timed region) between its own events; the stream is
    # held while they are enqueued, so no replay waits on the host
    n_dist = max(3, min(args.steps // len(wl.copies), 100))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_dist)]
    torch.cuda.synchronize()
    hold_stream(wl.stream, n_dist * len(wl.copies))
    with torch.cuda.stream(wl.stream):
        for a, b in evs:
            a.record(wl.stream)
            wl.cycle.replay()
            b.record(wl.stream)
    torch.cuda.synchronize()
    per = sorted(a.elapsed_time(b) * 1e3 / len(wl.copies) for a, b in evs)
    per_step = {"median": round(statistics.median(per), 3), "p10": round(per[len(per) // 10], 3),
                "p90": round(per[(9 * len(per)) // 10], 3), "n": n_dist,
                "how": f"us per step over each replay of {len(wl.copies)} back-to-back steps, "
                       f"each replay between its own events"}
    t_calls = time_steps(lambda k: calls.run(k), args.steps, calls.stream)
    t_calls = max_over_ranks(t_calls, world, dev)
    t_one = time_steps(lambda k: one.run(k), args.steps, one.stream)
    t_one = max_over_ranks(t_one, world, dev)

    sb = step_bytes(4)
    value = job_gbs(sb, args.steps, world, t)
    ms = t / args.steps * 1e3
    hbm_peak, peak_kind = peaks()

    # Dominant kernel: the grouped gate/up launch (2/3 of the bytes), timed alone.
    gu_bytes = N_EXPERTS * 2 * q_bytes(4, D_FF, D_MODEL, GROUP) + D_MODEL * 4 + N_EXPERTS * D_FF * 4
    nlaunch = 4 * len(wl.copies)
    ptrs = [[[t[k] for t in ex] for k in ("gate_codes", "gate_scales", "up_codes", "up_scales")]
            for ex in wl.copies]

    def gu_launch(i):
        smoe.smoe_experts_gate_up_q4(*ptrs[i % len(wl.copies)], wl.x, wl.hidden, D_FF, D_MODEL, GROUP,
                                     stream=wl.stream)

    kernel_alone_seconds(gu_launch, nlaunch, wl.stream)  # warm
    t_gu_alone = kernel_alone_seconds(gu_launch, nlaunch, wl.stream)
    t_gu = kernel_chain_seconds(gu_launch, nlaunch, wl.stream)
    achieved = gu_bytes / t_gu / 1e9
    roof = {"kernel": "qgemv_reg<Q4,gate_up> (smoe_experts_gate_up_q4, 8 experts x 1536x4096)",
            "bound": "hbm",
            "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
            "frac": round(achieved / hbm_peak, 4), "traffic": roofline_traffic("gate_up_q4"),
            "algorithmic_bytes_per_launch": gu_bytes, "us_per_launch": round(t_gu * 1e6, 3),
            "timing": f"{nlaunch} launches on rotating weight copies in one CUDA graph, events around "
                      f"graph replays; one launch bracketed by its own events, the stream held so the host "
                      f"is ahead: {t_gu_alone * 1e6:.3f} us",
            "peak_kind": f"{peak_kind} burst HBM copy bandwidth"}

    # The other kernel of the step, timed the same way.
    dn_ptrs = [[[t[k] for t in ex] for k in ("down_codes", "down_scales")] for ex in wl.copies]
    t_dn = kernel_chain_seconds(lambda i: smoe.smoe_experts_down_q4(*dn_ptrs[i % len(wl.copies)], wl.hidden, wl.out,
                                                                    D_MODEL, D_FF, GROUP, stream=wl.stream),
                                nlaunch, wl.stream)
    dn_bytes = N_EXPERTS * q_bytes(4, D_MODEL, D_FF, GROUP) + N_EXPERTS * D_FF * 4 + N_EXPERTS * D_MODEL * 4
    down_kernel = {"kernel": "qgemv_reg<Q4,down> (smoe_experts_down_q4, 8 experts x 4096x1536)",
                   "us_per_launch": round(t_dn * 1e6, 3), "GB/s": round(dn_bytes / t_dn / 1e9, 1),
                   "frac": round(dn_bytes / t_dn / 1e9 / hbm_peak, 4), "algorithmic_bytes_per_launch": dn_bytes}

    # End to end: token in from pinned host memory, outputs back to pinned host memory.
    x_host = torch.from_numpy(inp.activations(D_MODEL, 5)).pin_memory()
    out_host = torch.empty((N_EXPERTS, D_MODEL)).pin_memory()
    h2d, d2h = D_MODEL * 4, N_EXPERTS * D_MODEL * 4

    # (1) one CUDA graph per weight copy holds the whole step: smoe_copy of
    # the token into device memory (every CTA of gate/up reads it), the two
    # grouped calls, the down projection writing its outputs straight into
    # the pinned host buffer (each output crosses the host link once)
    def e2e_body(c, s):
        ex = wl.copies[c]
        smoe.smoe_copy(wl.x, x_host, h2d, stream=s)
        wl.g_gate_up([t["gate_codes"] for t in ex], [t["gate_scales"] for t in ex], [t["up_codes"] for t in ex],
                     [t["up_scales"] for t in ex], wl.x, wl.hidden, D_FF, D_MODEL, GROUP, stream=s)
        wl.g_down([t["down_codes"] for t in ex], [t["down_scales"] for t in ex], wl.hidden, out_host,
                  D_MODEL, D_FF, GROUP, stream=s)

    with torch.cuda.stream(wl.stream):
        for c in range(len(wl.copies)):
            e2e_body(c, wl.stream)
    wl.stream.synchronize()
    e2e_graphs = []
    for c in range(len(wl.copies)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=wl.stream, capture_error_mode="thread_local"):
            e2e_body(c, wl.stream)
        e2e_graphs.append(g)

    def e2e_steps(k):
        for i in range(k):
            e2e_graphs[i % len(e2e_graphs)].replay()

    # (2) through the copy engines (cudaMemcpyAsync) around the step's graph
    def e2e_ce_steps(k):
        for i in range(k):
            wl.x.copy_(x_host, non_blocking=True)
            wl.graphs[i % len(wl.graphs)].replay()
            out_host.copy_(wl.out, non_blocking=True)

    e2e_n = max(3, min(args.steps, 2000))
    with torch.cuda.stream(wl.stream):
        e2e_steps(3)
        t_e2e = time_steps(e2e_steps, e2e_n, wl.stream)
        # the last step's outputs, written to host memory by the down
        # projection, against the same step computed into device memory
        torch.cuda.synchronize()
        host_out = out_host.clone()
        wl.calls((e2e_n - 1) % len(wl.copies), wl.stream)
        torch.cuda.synchronize()
        if not torch.equal(host_out, wl.out.cpu()):
            raise RuntimeError("end-to-end step: the outputs written to host memory differ from the device's")
        e2e_ce_steps(3)
        t_ce = time_steps(e2e_ce_steps, e2e_n, wl.stream)
    t_e2e = max_over_ranks(t_e2e, world, dev)
    t_ce = max_over_ranks(t_ce, world, dev)
    torch.cuda.synchronize()
    if not torch.equal(out_host, wl.out.cpu()):
        raise RuntimeError("end-to-end step: the outputs copied to host memory differ from the device's")
    e2e = {"value": round(sb * e2e_n * world / t_e2e / 1e9, 2), "unit": "GB/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "us_per_step": round(t_e2e / e2e_n * 1e6, 3),
           "launch": "one CUDA graph replay per step: smoe_copy of the token from pinned host memory, "
                     "the 2 grouped C-ABI calls, the down projection writing the outputs straight into "
                     "pinned host memory (over the host link, chained with programmatic dependent launch)",
           "copy_engine": {"us_per_step": round(t_ce / e2e_n * 1e6, 3),
                           "launch": "per step: cudaMemcpyAsync in, one graph replay, cudaMemcpyAsync out"}}

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32+f32",
        "arithmetic": "per 32-column chunk x is rounded to a power-of-two grid with its largest |x| in "
                      "[2^22, 2^23) (three signed-byte digits); code x digit products summed exactly in "
                      "int32 (dp4a, codes minus 8); per-chunk scale fold, row sum and SiLU in f32",
        "data": "synthetic (seeded uniform codes, U[0.01,0.05] scales, N(0,1) token)",
        "config": {"workload": WORKLOAD, "bytes_per_step": sb,
                   "l2": f"{len(wl.copies)} rotating weight copies ({len(wl.copies) * sb / 1e6:.0f} MB) "
                         f"> {L2_BYTES >> 20} MB L2",
                   "launch": "2 grouped C-ABI calls per step (smoe_experts_gate_up_q4 over the 8 "
                             "experts, then smoe_experts_down_q4), captured in a CUDA graph, "
                             "programmatic dependent launch between kernels",
                   "parallelism": f"replicas x{world} (experts are independent; no collective)"},
        "us_per_8expert_ffn": round(ms * 1e3, 3),
        "per_step_us": per_step,
        "submission_inclusive": {"ms_per_step": round(t_unheld / args.steps * 1e3, 6),
                                 "how": "the same K steps with the host enqueueing graph replays while "
                                        "the device runs them (no stream hold before the start event)"},
        "one_call": {"GB/s": round(sb * args.steps * world / t_one / 1e9, 2),
                     "us_per_8expert_ffn": round(t_one / args.steps * 1e6, 3),
                     "launch": "1 C-ABI call per step (smoe_experts_ffn_q4: one launch for gate/up and "
                               "down of the 8 experts) in a CUDA graph"},
        "per_expert_calls": {"GB/s": round(sb * args.steps * world / t_calls / 1e9, 2),
                             "us_per_8expert_ffn": round(t_calls / args.steps * 1e6, 3),
                             "launch": "16 single-expert calls (8 x smoe_gate_up_q4 + smoe_down_q4) per "
                                       "step in a CUDA graph"},
        "hbm_frac": round(value / world / hbm_peak, 4),
        "roofline": roof, "down_kernel": down_kernel, "e2e": e2e, "gpu_launches": 2 * args.steps,
        "clocks": clock_rec,
    }
    return result, wl, smoe, dev


# ------------------------------------------------------------ other rows

def rows_breakdown(smoe, dev, steps, pattern=""):
    """Each remaining row of the hot path, timed with events on its own stream
    over `steps` launches with rotating inputs larger than L2.  `pattern`
    keeps only the rows whose name contains it."""
    import torch
    hbm_peak, _ = peaks()
    out = {}
    s = torch.cuda.Stream(device=dev)

    def timed(launch, n, calls_per=1):
        """calls_per: C-ABI calls one launch(i) makes (sizes the stream hold)."""
        with torch.cuda.stream(s):
            for i in range(3):
                launch(i)
            return time_steps(lambda k: [launch(i) for i in range(k)], n, s, hold=n * calls_per)

    if pattern in "q2_8expert_decode":
        q2_row(smoe, dev, steps, out, hbm_peak)
    for (rows, cols), seed in zip(inp.CONFIGS["bf16_matvec"]["shapes"], inp.CONFIGS["bf16_matvec"]["seeds"]):
        if pattern in f"bf16_{rows}x{cols}":
            bf16_row(smoe, dev, steps, out, hbm_peak, timed, s, rows, cols, seed)
    if pattern in "bf16_batch_8x512x4096":
        bf16_batch_row(smoe, dev, steps, out, hbm_peak, timed, s)
    # the workload's token counts, plus 2, 4 and 8 (the decode-slot path
    # below the measured crossover with the tensor cores)
    for T in sorted(set(inp.CONFIGS["q4_token_batch"]["tokens"]) | {2, 4, 8}):
        if pattern in f"q4_token_batch_T{T}":
            batch_row(smoe, dev, steps, out, hbm_peak, timed, s, T)
    for T in (16, 256):
        if pattern in f"q2_token_batch_T{T}":
            batch_row(smoe, dev, steps, out, hbm_peak, timed, s, T, bits=2)
    if pattern in "q4_experts_batch_8xT16":
        experts_batch_row(smoe, dev, steps, out, hbm_peak, timed, s)
    if pattern in "route_128x4096_top8":
        route_row(smoe, dev, steps, out, timed, s)
    for bits in (4, 2):
        if pattern in f"q{bits}_gate_up_38experts_sustained":
            sustained_row(smoe, dev, steps, out, hbm_peak, bits)
    if pattern in "moe_layer_routed_128e_top8":
        routed_layer_row(smoe, dev, steps, out, s)
    if pattern in "q4_ffn_256":
        small_row(smoe, dev, steps, out, timed, s)
    return out


def q2_row(smoe, dev, steps, out, hbm_peak):
    """Q2 8-expert decode with the grouped calls, timed like the headline step."""
    import torch
    n_copies = max(2, -(-4 * L2_BYTES // step_bytes(2)))
    q2 = DecodeWorkload(smoe, dev, 2, 6, n_copies, grouped=True)
    q2.capture()
    q2.run(5)
    n = max(50, steps // 4)
    nc = len(q2.copies)
    t = time_steps(lambda k: q2.run(k), n, q2.stream, hold=n // nc + n % nc)
    sb = step_bytes(2)
    # each grouped kernel alone, in a chain of launches on rotating copies
    nc = len(q2.copies)
    gu = [[[t[k] for t in ex] for k in ("gate_codes", "gate_scales", "up_codes", "up_scales")] for ex in q2.copies]
    dn = [[[t[k] for t in ex] for k in ("down_codes", "down_scales")] for ex in q2.copies]
    t_gu = kernel_chain_seconds(lambda i: smoe.smoe_experts_gate_up_q2(*gu[i % nc], q2.x, q2.hidden, D_FF, D_MODEL,
                                                                       GROUP, stream=q2.stream), 4 * nc, q2.stream)
    t_dn = kernel_chain_seconds(lambda i: smoe.smoe_experts_down_q2(*dn[i % nc], q2.hidden, q2.out, D_MODEL, D_FF,
                                                                    GROUP, stream=q2.stream), 4 * nc, q2.stream)
    b_gu = N_EXPERTS * 2 * q_bytes(2, D_FF, D_MODEL, GROUP)
    b_dn = N_EXPERTS * q_bytes(2, D_MODEL, D_FF, GROUP)
    out["q2_8expert_decode"] = {"GB/s": round(sb * n / t / 1e9, 1), "us_per_step": round(t / n * 1e6, 3),
                                "frac": round(sb * n / t / 1e9 / hbm_peak, 4), "bytes_per_step": sb,
                                "gate_up_us": round(t_gu * 1e6, 3),
                                "gate_up_frac": round(b_gu / t_gu / 1e9 / hbm_peak, 4),
                                "down_us": round(t_dn * 1e6, 3),
                                "down_frac": round(b_dn / t_dn / 1e9 / hbm_peak, 4)}
    del q2
    torch.cuda.empty_cache()


def bf16_row(smoe, dev, steps, out, hbm_peak, timed, s, rows, cols, seed):
    """One dense bf16 matvec shape."""
    import torch
    wbytes = rows * cols * 2
    ncp = max(1, min(8, -(-2 * L2_BYTES // wbytes)))
    ws = [torch.from_numpy(inp.bf16_rows(rows, cols, seed, 1 + c).view(np.int16)).to(dev) for c in range(ncp)]
    x = torch.from_numpy(inp.activations(cols, seed)).to(dev)
    y = torch.empty(rows, device=dev)
    nl = max(20, min(steps // 4, int(2e9 // wbytes)))
    t = timed(lambda i: smoe.matvec_bf16(ws[i % ncp], x, y, rows, cols, stream=s), nl)
    b = wbytes + cols * 4 + rows * 4
    out[f"bf16_{rows}x{cols}"] = {"GB/s": round(b * nl / t / 1e9, 1), "us_per_call": round(t / nl * 1e6, 3),
                                  "frac": round(b * nl / t / 1e9 / hbm_peak, 4), "bytes_per_call": b}
    del ws
    torch.cuda.empty_cache()


def bf16_batch_row(smoe, dev, steps, out, hbm_peak, timed, s, n=8, rows=512, cols=4096, seed=3):
    """n small bf16 matvecs in one matvec_bf16_batch submission, against the
    same matvecs as n matvec_bf16 calls."""
    import torch
    wbytes = n * rows * cols * 2
    ncp = max(2, -(-4 * L2_BYTES // wbytes))
    ws = [[torch.from_numpy(inp.bf16_rows(rows, cols, seed, 1 + 100 * c + i).view(np.int16)).to(dev)
           for i in range(n)] for c in range(ncp)]
    xs = [torch.from_numpy(inp.activations(cols, seed + i)).to(dev) for i in range(n)]
    ys = [torch.empty(rows, device=dev) for _ in range(n)]
    nl = max(20, min(steps // 4, 400))
    t_b = timed(lambda i: smoe.matvec_bf16_batch(ws[i % ncp], xs, ys, [rows] * n, [cols] * n, stream=s), nl)

    def singles(i):
        for j in range(n):
            smoe.matvec_bf16(ws[i % ncp][j], xs[j], ys[j], rows, cols, stream=s)

    t_s = timed(singles, nl, calls_per=n)
    b = n * (rows * cols * 2 + cols * 4 + rows * 4)
    out[f"bf16_batch_{n}x{rows}x{cols}"] = {
        "GB/s": round(b * nl / t_b / 1e9, 1), "us_per_call": round(t_b / nl * 1e6, 3),
        "frac": round(b * nl / t_b / 1e9 / hbm_peak, 4), "bytes_per_call": b,
        "single_calls_us": round(t_s / nl * 1e6, 3)}
    del ws
    torch.cuda.empty_cache()


def batch_row(smoe, dev, steps, out, hbm_peak, timed, s, T, bits=4):
    """Token-batch FFN of one expert for T tokens (16 rotating experts)."""
    import torch
    ncp = 16
    experts = [{k: torch.from_numpy(v).to(dev)
                for k, v in inp.expert(bits, D_MODEL, D_FF, GROUP, 7 + bits % 4 + 1000 * c).items()}
               for c in range(ncp)]
    fn = smoe.ffn_batch_q4 if bits == 4 else smoe.ffn_batch_q2
    X = torch.from_numpy(inp.activations((T, D_MODEL), 7)).to(dev)
    Y = torch.empty((T, D_MODEL), device=dev)
    need = smoe.smoe_ffn_batch_workspace_bytes(T, D_MODEL, D_FF, GROUP)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)

    def launch(i):
        e = experts[i % ncp]
        fn(e["gate_codes"], e["gate_scales"], e["up_codes"], e["up_scales"], e["down_codes"],
           e["down_scales"], X, Y, T, D_MODEL, D_FF, GROUP, ws, need, stream=s)
    nl = max(20, min(steps // 8, 400))
    t = timed(launch, nl)
    b = expert_bytes(bits) + 2 * T * D_MODEL * 4
    flops = 2 * T * 3 * D_FF * D_MODEL
    out[f"q{bits}_token_batch_T{T}"] = {"GB/s": round(b * nl / t / 1e9, 1), "us_per_call": round(t / nl * 1e6, 3),
                                   "frac": round(b * nl / t / 1e9 / hbm_peak, 4),
                                   "TFLOP/s": round(flops * nl / t / 1e12, 2), "bytes_per_call": b}
    del experts
    torch.cuda.empty_cache()


def experts_batch_row(smoe, dev, steps, out, hbm_peak, timed, s, n=8, T=16):
    """Token batches of n experts (T tokens each) in one smoe_experts_ffn_batch_q4
    call, against the same batches as n ffn_batch_q4 calls."""
    import torch
    ncp = 4  # weight sets of n experts, rotated: 4 x 8 x 10.6 MB > L2
    sets = [[{k: torch.from_numpy(v).to(dev) for k, v in inp.expert(4, D_MODEL, D_FF, GROUP, 9 + 1000 * c, e).items()}
             for e in range(n)] for c in range(ncp)]
    Xs = [torch.from_numpy(inp.activations((T, D_MODEL), 9 + e)).to(dev) for e in range(n)]
    Ys = [torch.empty((T, D_MODEL), device=dev) for _ in range(n)]
    Ts = [T] * n
    need = smoe.smoe_experts_ffn_batch_workspace_bytes(Ts, D_MODEL, D_FF, GROUP)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    key = ("gate_codes", "gate_scales", "up_codes", "up_scales", "down_codes", "down_scales")

    def grouped(i):
        ex = sets[i % ncp]
        smoe.smoe_experts_ffn_batch_q4(*[[x[k] for x in ex] for k in key], Xs, Ys, Ts, D_MODEL, D_FF, GROUP,
                                       ws, need, stream=s)

    need1 = smoe.smoe_ffn_batch_workspace_bytes(T, D_MODEL, D_FF, GROUP)
    ws1 = torch.empty(need1, dtype=torch.uint8, device=dev)

    def singles(i):
        for e, x in enumerate(sets[i % ncp]):
            smoe.ffn_batch_q4(*[x[k] for k in key], Xs[e], Ys[e], T, D_MODEL, D_FF, GROUP, ws1, need1, stream=s)

    nl = max(20, min(steps // 8, 200))
    t_g = timed(grouped, nl)
    t_s = timed(singles, nl, calls_per=n)
    b = n * (expert_bytes(4) + 2 * T * D_MODEL * 4)
    out[f"q4_experts_batch_{n}xT{T}"] = {
        "GB/s": round(b * nl / t_g / 1e9, 1), "us_per_call": round(t_g / nl * 1e6, 3),
        "frac": round(b * nl / t_g / 1e9 / hbm_peak, 4), "bytes_per_call": b,
        "single_calls_us": round(t_s / nl * 1e6, 3)}
    del sets
    torch.cuda.empty_cache()


def route_row(smoe, dev, steps, out, timed, s, n=128, d=D_MODEL, k=N_EXPERTS):
    """Router of one token (bf16 gate 128 x 4096, top-8 with weights) and the
    combine of 8 expert outputs."""
    import torch
    ncp = 8
    gs = [torch.from_numpy(inp.bf16_rows(n, d, 10, 1 + c).view(np.int16)).to(dev) for c in range(ncp)]
    x = torch.from_numpy(inp.activations(d, 10)).to(dev)
    logits = torch.empty(n, device=dev)
    idx = torch.empty(k, dtype=torch.int32, device=dev)
    w = torch.empty(k, device=dev)
    eo = torch.from_numpy(inp.activations((k, d), 11)).to(dev)
    y = torch.empty(d, device=dev)
    nl = max(20, min(steps // 4, 400))
    t_r = timed(lambda i: smoe.smoe_route_topk_bf16(gs[i % ncp], x, n, d, k, logits, idx, w, stream=s), nl)
    t_l = timed(lambda i: smoe.matvec_bf16(gs[i % ncp], x, logits, n, d, stream=s), nl)
    t_c = timed(lambda i: smoe.smoe_combine(k, eo, w, y, d, stream=s), nl)
    out[f"route_{n}x{d}_top{k}"] = {"us_per_route": round(t_r / nl * 1e6, 3),
                                    "us_per_logits_matvec": round(t_l / nl * 1e6, 3),
                                    "us_per_combine": round(t_c / nl * 1e6, 3)}
    del gs
    torch.cuda.empty_cache()


def routed_layer_row(smoe, dev, steps, out, s, n=128, k=N_EXPERTS, ntok=16):
    """A whole MoE layer per token with the selection on the device: router
    (bf16 gate n x 4096, top-k), the routed FFN of the k selected Q4 experts
    (smoe_experts_ffn_routed_q4 out of device pointer tables), combine.  One
    CUDA graph holds the layers of ntok different tokens back to back; the
    device time per layer is timed with the stream held.  End to end: the
    token copied in from pinned host memory and the layer output copied back
    (smoe_copy), one graph replay per token, host submission included."""
    import torch
    keys = ("gate_codes", "gate_scales", "up_codes", "up_scales", "down_codes", "down_scales")
    ex = [{kk: torch.from_numpy(v).to(dev) for kk, v in inp.expert(4, D_MODEL, D_FF, GROUP, 12, e).items()}
          for e in range(n)]
    tabs = [smoe.pointer_table([t[kk] for t in ex], dev) for kk in keys]
    gate = torch.from_numpy(inp.bf16_rows(n, D_MODEL, 12, 1).view(np.int16)).to(dev)
    X = torch.from_numpy(inp.activations((ntok, D_MODEL), 12)).to(dev)
    logits = torch.empty(n, device=dev)
    idx = torch.empty(k, dtype=torch.int32, device=dev)
    w = torch.empty(k, device=dev)
    wsb = smoe.smoe_experts_ffn_routed_workspace_bytes(k, D_FF)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    eo = torch.empty((k, D_MODEL), device=dev)
    y = torch.empty(D_MODEL, device=dev)

    def layer(x, out=None):
        smoe.smoe_route_topk_bf16(gate, x, n, D_MODEL, k, logits, idx, w, stream=s)
        smoe.smoe_experts_ffn_routed_q4(n, k, *tabs, idx, x, eo, D_MODEL, D_FF, GROUP, ws, wsb, stream=s)
        smoe.smoe_combine(k, eo, w, y if out is None else out, D_MODEL, stream=s)

    with torch.cuda.stream(s):
        for i in range(ntok):
            layer(X[i])
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(ntok):
            layer(X[i])
    reps = max(4, min(steps // ntok, 200))
    with torch.cuda.stream(s):
        g.replay()
        t = time_steps(lambda r: [g.replay() for _ in range(r)], reps, s, hold=reps * ntok)
    per = t / (reps * ntok)
    layer_bytes = n * D_MODEL * 2 + D_MODEL * 4 + k * expert_bytes(4, D_MODEL, D_FF, GROUP) + k * D_MODEL * 4 \
        + D_MODEL * 4
    # end to end: token in from pinned host memory (smoe_copy), the combine
    # writing the layer output straight into pinned host memory
    x_host = torch.from_numpy(inp.activations(D_MODEL, 13)).pin_memory()
    y_host = torch.empty(D_MODEL).pin_memory()
    xd = torch.empty(D_MODEL, device=dev)

    def e2e_body():
        smoe.smoe_copy(xd, x_host, D_MODEL * 4, stream=s)
        layer(xd, y_host)

    with torch.cuda.stream(s):
        e2e_body()
    s.synchronize()
    ge = torch.cuda.CUDAGraph()
    with torch.cuda.graph(ge, stream=s, capture_error_mode="thread_local"):
        e2e_body()
    ne = max(20, min(steps, 500))
    with torch.cuda.stream(s):
        ge.replay()
        te = time_steps(lambda r: [ge.replay() for _ in range(r)], ne, s)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        layer(xd)  # the same token's layer into device memory
    torch.cuda.synchronize()
    if not torch.equal(y_host, y.cpu()):
        raise RuntimeError("routed layer: the output written to host memory differs from the device's")
    out[f"moe_layer_routed_{n}e_top{k}"] = {
        "us_per_layer": round(per * 1e6, 3), "GB/s": round(layer_bytes / per / 1e9, 1),
        "bytes_per_layer": layer_bytes, "launches_per_layer": 6,
        "e2e": {"us_per_layer": round(te / ne * 1e6, 3), "h2d_bytes": D_MODEL * 4, "d2h_bytes": D_MODEL * 4,
                "launch": "one graph replay per token: smoe_copy in, route, routed FFN, combine into pinned "
                          "host memory"},
        "how": f"{ntok} layers on {ntok} tokens in one CUDA graph, {reps} replays, stream held; "
               f"{n} experts x {D_FF}x{D_MODEL} Q4 resident ({n * expert_bytes(4, D_MODEL, D_FF, GROUP) / 1e9:.2f} GB)"}
    del ex, tabs
    torch.cuda.empty_cache()


def sustained_row(smoe, dev, steps, out, hbm_peak, bits=4, n=38):
    """The grouped gate/up kernel over n experts in one launch (n = 38: four
    CTAs per expert, 384 rows each, about 32 stages per warp), so that the
    launch's ramp and tail are a small part of it: the kernel's streaming
    rate in steady state.  Two weight copies alternate (> 2 x L2)."""
    import torch
    ncp = 2
    sets = [[{k: torch.from_numpy(v).to(dev) for k, v in inp.expert(bits, D_MODEL, D_FF, GROUP, 13 + 1000 * c, e).items()
              if k.startswith(("gate", "up"))} for e in range(n)] for c in range(ncp)]
    x = torch.from_numpy(inp.activations(D_MODEL, 13)).to(dev)
    hid = torch.empty((n, D_FF), device=dev)
    fn = smoe.smoe_experts_gate_up_q4 if bits == 4 else smoe.smoe_experts_gate_up_q2
    st = torch.cuda.Stream(device=dev)
    ptrs = [[[t[k] for t in ex] for k in ("gate_codes", "gate_scales", "up_codes", "up_scales")] for ex in sets]
    t = kernel_chain_seconds(lambda i: fn(*ptrs[i % ncp], x, hid, D_FF, D_MODEL, GROUP, stream=st), 4, st)
    b = n * 2 * q_bytes(bits, D_FF, D_MODEL, GROUP) + D_MODEL * 4 + n * D_FF * 4
    out[f"q{bits}_gate_up_{n}experts_sustained"] = {"us_per_launch": round(t * 1e6, 3), "GB/s": round(b / t / 1e9, 1),
                                                   "frac": round(b / t / 1e9 / hbm_peak, 4),
                                                   "bytes_per_launch": b}
    del sets
    torch.cuda.empty_cache()


def small_row(smoe, dev, steps, out, timed, s):
    """The small 256/256 expert (latency bound)."""
    import torch
    small = [{k: torch.from_numpy(v).to(dev) for k, v in inp.expert(4, 256, 256, 64, c).items()} for c in range(4)]
    xs = torch.from_numpy(inp.activations(256, 0)).to(dev)
    hs = torch.empty(256, device=dev)
    ys = torch.empty(256, device=dev)

    def small_launch(i):
        e = small[i % 4]
        smoe.smoe_gate_up_q4(e["gate_codes"], e["gate_scales"], e["up_codes"], e["up_scales"], xs, hs,
                             256, 256, 64, stream=s)
        smoe.smoe_down_q4(e["down_codes"], e["down_scales"], hs, ys, 256, 256, 64, stream=s)
    nl = max(50, min(steps // 4, 2000))
    t = timed(small_launch, nl)
    out["q4_ffn_256"] = {"us_per_ffn": round(t / nl * 1e6, 3), "bytes_per_ffn": expert_bytes(4, 256, 256, 64)}


# ------------------------------------------------------------ the CPU arm

def cpu_sample(seconds, frac=None):
    """Times the oracle on the host cores on whole or sliced 8-expert steps.
    Returns (GB/s by the step's byte formula, threads, description, sec/step)."""
    import oracle
    threads = oracle.host_threads()
    oracle.set_threads(threads)
    experts = [inp.expert(4, D_MODEL, D_FF, GROUP, 5, e) for e in range(N_EXPERTS)]
    x = inp.activations(D_MODEL, 5).astype(np.float64)
    gu_rows = D_FF if frac is None else max(1, int(D_FF * frac))
    dn_rows = D_MODEL if frac is None else max(1, int(D_MODEL * frac))
    hidden = np.zeros(D_FF)

    def one_step():
        for e in experts:
            r = oracle.gate_up(4, e["gate_codes"], e["gate_scales"], e["up_codes"], e["up_scales"],
                               D_FF, D_MODEL, GROUP, x, 0, gu_rows)
            hidden[:gu_rows] = r["hidden"]
            oracle.qgemv(4, e["down_codes"], e["down_scales"], D_MODEL, D_FF, GROUP, hidden, 0, dn_rows)

    steps, t0 = 0, time.perf_counter()
    while True:
        one_step()
        steps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    b = (N_EXPERTS * (2 * q_bytes(4, gu_rows, D_MODEL, GROUP) + q_bytes(4, dn_rows, D_FF, GROUP))
         + D_MODEL * 4 + N_EXPERTS * dn_rows * 4)
    desc = (f"{steps} oracle step(s) of the 8-expert decode"
            + ("" if frac is None else f", each on rows [0,{gu_rows}) of gate/up and [0,{dn_rows}) of down")
            + f"; {el:.1f} s wall")
    return b * steps / el / 1e9, threads, desc, el / steps, b


def reference_arm(args, rank, world):
    """The oracle, as it stands, on this host's cores: K steps after W warm-up
    steps, each step a row slice of the 8-expert decode sized so the whole run
    stays within about a minute and a half."""
    if rank != 0:
        return None
    # size the slice: one probe step on 1/64 of the rows
    _, _, _, per, _ = cpu_sample(0.0, frac=1 / 64)
    budget = 90.0 / max(1, args.steps + args.warmup)
    frac = max(1 / D_FF, min(1.0, (1 / 64) * budget / max(per, 1e-9)))
    import oracle
    experts = [inp.expert(4, D_MODEL, D_FF, GROUP, 5, e) for e in range(N_EXPERTS)]
    x = inp.activations(D_MODEL, 5).astype(np.float64)
    gu_rows, dn_rows = max(1, int(D_FF * frac)), max(1, int(D_MODEL * frac))
    hidden = np.zeros(D_FF)

    def step():
        for e in experts:
            r = oracle.gate_up(4, e["gate_codes"], e["gate_scales"], e["up_codes"], e["up_scales"],
                               D_FF, D_MODEL, GROUP, x, 0, gu_rows)
            hidden[:gu_rows] = r["hidden"]
            oracle.qgemv(4, e["down_codes"], e["down_scales"], D_MODEL, D_FF, GROUP, hidden, 0, dn_rows)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    t = time.perf_counter() - t0
    b = (N_EXPERTS * (2 * q_bytes(4, gu_rows, D_MODEL, GROUP) + q_bytes(4, dn_rows, D_FF, GROUP))
         + D_MODEL * 4 + N_EXPERTS * dn_rows * 4)
    v = b * args.steps / t / 1e9
    sample = (f"each step: the 8-expert Q4 decode on rows [0,{gu_rows}) of every gate/up and "
              f"[0,{dn_rows}) of every down matrix ({b} algorithmic bytes)")
    return {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(t / args.steps * 1e3, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "bytes_per_step": b},
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": oracle.get_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-rows", action="store_true", help="skip the per-row breakdown")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--rows", default="", help="run only the breakdown rows whose name contains this")
    ap.add_argument("--rows-only", action="store_true",
                    help="run only the breakdown rows (no headline step): for profiling one row's kernels")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        # rank 0 alone times the oracle; the other ranks exit without work
        rank = int(os.environ.get("RANK", "0"))
        res = reference_arm(args, rank, int(os.environ.get("WORLD_SIZE", "1")))
        if rank == 0:
            print(json.dumps(res), flush=True)
        return
    rank, world, local = dist_setup()
    if args.rows_only:
        import torch
        import __graft_entry__
        __graft_entry__.build_library()
        import moe_expert_ffn_smoe_gb300 as smoe
        dev = torch.device(f"cuda:{local}")
        torch.cuda.set_device(dev)
        if rank == 0:
            print(json.dumps({"rows": rows_breakdown(smoe, dev, args.steps, args.rows)}), flush=True)
        return

    res, wl, smoe, dev = gpu_arm(args, rank, world, local)
    if rank == 0 and world == 1 and not args.no_cpu:
        v, threads, desc, _, _ = cpu_sample(args.cpu_seconds)
        res["cpu_baseline"] = {"value": round(v, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                               "sample": desc}
    if rank == 0 and world == 1 and not args.no_rows:
        del wl
        res["rows"] = rows_breakdown(smoe, dev, args.steps, args.rows)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
