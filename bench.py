#!/usr/bin/env python3
"""Throughput of the ONNX-semantics recurrent operator on GB300.

One step = one rnn_run (weight pack, input projection, state set-up,
persistent recurrence, mask epilogue) over one batch of the workload, inputs
resident in HBM.  The default workload is the largest one that fits one GPU:
the LSTM bidirectional layer (seq 512, batch 128, input 1024, hidden 1024,
clip 3, HardSigmoid / LeakyRelu / ScaledTanh forward, sequence_lens), in
fast mode (fp32: fused multiply-adds, within 1e-5 of the exact arithmetic).
The metric is cell-steps per second (seq * batch * dirs per step),
aggregated over ranks; each rank runs an independent replica (the operator
has no exchange between GPUs).  The value comes from the median step time
over the K timed steps (the mean is reported beside it).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--mode exact|fast|tf32|bf16]
                  [--workload NAME] [--impl ours|reference]

The L2 (129 MB) is flushed between timed steps by writing a 256 MiB buffer
outside the timed events.  Per-kernel times come from CUDA events the library
records on its own stream around each kernel during the timed steps.  The
recurrent kernel's roofline is the per-step one: each step is bounded below by
the largest of its FP32 work over the ALU peak, its resident R bytes over the
shared-memory bandwidth, and the R bytes that cannot stay in shared memory
over the L2 bandwidth (measured here with an elementwise kernel over a
buffer pair that fits in L2).  The
reference arm (--impl reference) times the CPU oracle on the host, one batch
row of the workload per step.
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "cell-steps/sec (seq*batch*dirs per s) at 1 GB300; % of roofline per kernel"
UNIT = "cell-steps/s"
DEFAULT_WORKLOAD = "lstm_bidi_s512_b128_i1024_h1024"
DEFAULT_MODE = "fast"
FLUSH_BYTES = 256 << 20


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--lbr", type=int, default=0)
    ap.add_argument("--mode", default=DEFAULT_MODE, choices=["exact", "fast", "tf32", "bf16"])
    ap.add_argument("--io", default="f32", choices=["f32", "f16", "bf16"],
                    help="element type of X, initial states and outputs")
    ap.add_argument("--launch", default=None,
                    help="recurrent launch override unit_groups,rows_per_thread,r_resident,row_groups,kernel "
                         "(rnn_plan_set_launch; 0 / -1 = the planner's choice)")
    ap.add_argument("--layer-by-layer", action="store_true",
                    help="stack workloads: run the layers one after another")
    ap.add_argument("--wavefront", action="store_true",
                    help="stack workloads: one wavefront launch whenever the stack qualifies "
                         "(default: where the library measures it faster)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--out", default=None, help="also append the JSON line to this file")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(values, dist, device):
    """Each value's maximum over the ranks (the slowest replica sets the
    job's time); `dist` is torch.distributed with a process group up."""
    import torch
    t = torch.tensor([float(v) for v in values], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_value(units_per_rank, steps, world_size, total_ms):
    """Whole-job throughput: every rank's units over the slowest rank's time."""
    return units_per_rank * steps * world_size / (total_ms / 1e3)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f)
    return {}


def emit(obj, out=None):
    line = json.dumps(obj)
    print(line, flush=True)
    if out:
        with open(out, "a") as f:
            f.write(line + "\n")


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.dev)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9], parts[4]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"],
                    "samples": 0}
        inside = [r for r in rows if t0 <= r[0] <= t1] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
                "samples": len(inside)}


# ------------------------------------------------------------- roofline

def algorithmic(case):
    """FLOPs of the recurrent and projection products, per run."""
    G, H, I, D = case.gates, case.hidden_size, case.input_size, case.dirs
    valid_rows_steps = case.valid_cell_steps()           # sum of lengths * dirs
    rec = 2.0 * valid_rows_steps * G * H * H
    proj = 2.0 * case.seq * case.batch * D * G * H * I
    proj_bytes = 4.0 * (case.seq * case.batch * I + D * G * H * I + case.seq * case.batch * D * G * H)
    return rec, proj, proj_bytes


def live_rows_per_step(case):
    """Rows still running at each step the recurrent kernel takes (it runs
    max(len) steps; a row of length L is live in steps 0..L-1)."""
    import numpy as np
    if case.sequence_lens is None:
        return [case.batch] * case.seq
    L = np.asarray(case.sequence_lens, np.int64)
    steps = int(L.max(initial=0))
    return [int((L > s).sum()) for s in range(steps)]


# Dependent-issue latency of an FP32 add or fused multiply-add on one
# accumulator (cycles): 4 nominal; 4.24 measured on this GPU by a chain of
# 8192 dependent adds in one warp (the chain bound below uses 4).
FP32_CHAIN_CYCLES = 4.0


def step_roofline(case, mode, rec_ms, sms, clock_mhz, l2_gbs, smem_per_sm, h_bytes=0.0, tensor_tflops=None):
    """The recurrent kernel's per-step roofline (per launch): every step takes
    at least the largest of
      alu   2 * live rows * D * G * H^2 FLOP over the FP32 peak (fused
            multiply-add in the fast modes, separate multiply and add in exact),
            or over `tensor_tflops` for the tensor-core recurrence;
      smem  the R slices read once from shared memory, D * 4 * G * H^2 bytes
            (2 per element on the tensor cores), over SMs * 128 bytes per clock;
      l2    the part of R that cannot stay resident in the SMs' shared memory
            (D * 4 * G * H^2 - SMs * smem_per_sm, if positive), streamed from L2
            every step, over the measured L2 copy bandwidth;
      h     the copies of h that the launch's CTAs need from L2 (every CTA
            holding a slice of R needs h of every row it multiplies): `h_bytes`
            for all rows, counted for the live rows only, over the same
            bandwidth;
      chain every output is one accumulator over k = 0..H-1 in order (exact
            and fast mode alike), H dependent adds a step (2H for GRU with
            linear_before_reset = 0, whose second product needs the first's
            result) at FP32_CHAIN_CYCLES each (not on the tensor cores).
    Returns the terms per step (microseconds, averaged over the steps), the
    binding term, the roofline time of the launch and its fraction of the
    measured time."""
    G, H, D = case.gates, case.hidden_size, case.dirs
    live = live_rows_per_step(case)
    clock = clock_mhz * 1e6
    alu_peak = (tensor_tflops * 1e12 if tensor_tflops else sms * 128 * (1 if mode == "exact" else 2) * clock)
    smem_bw = sms * 128 * clock
    r_bytes = (2.0 if tensor_tflops else 4.0) * D * G * H * H
    streamed = max(0.0, r_bytes - float(sms) * smem_per_sm)
    t_smem = r_bytes / smem_bw
    t_l2 = streamed / (l2_gbs * 1e9) if l2_gbs else 0.0
    t_h_all = h_bytes / (l2_gbs * 1e9) if l2_gbs else 0.0
    two = case.op == "GRU" and case.linear_before_reset == 0
    t_chain = 0.0 if tensor_tflops else (2 if two else 1) * H * FP32_CHAIN_CYCLES / clock
    roof, terms = 0.0, {"alu": 0.0, "smem": 0.0, "l2": 0.0, "h": 0.0, "chain": 0.0}
    for n in live:
        t_alu = 2.0 * n * D * G * H * H / alu_peak
        t_h = t_h_all * n / case.batch
        roof += max(t_alu, t_smem, t_l2, t_h, t_chain)
        terms["alu"] += t_alu
        terms["smem"] += t_smem
        terms["l2"] += t_l2
        terms["h"] += t_h
        terms["chain"] += t_chain
    steps = max(1, len(live))
    binding = max(terms, key=terms.get)
    return {"terms_us_per_step": {k: round(v / steps * 1e6, 4) for k, v in terms.items()},
            "binding": binding, "steps": len(live), "roof_ms": round(roof * 1e3, 5),
            "measured_ms": round(rec_ms, 5), "frac": round(roof * 1e3 / rec_ms, 4) if rec_ms else 0.0,
            "peaks": {"alu_tflops": round(alu_peak / 1e12, 3), "smem_tbs": round(smem_bw / 1e12, 3),
                      "l2_gbs": round(l2_gbs, 1) if l2_gbs else None, "chain_cycles": FP32_CHAIN_CYCLES,
                      "note": "alu and smem derived (SMs x 128 lanes or bytes per clock x max SM clock); "
                              "l2 measured by an elementwise kernel over a buffer pair that fits in L2; "
                              "chain: H dependent FP32 adds a step at the pipe's latency"},
            "r_bytes_per_step": r_bytes, "r_streamed_bytes_per_step": streamed, "h_bytes_per_step": h_bytes}


def h_bytes_per_step(geometry, case):
    """Bytes of h the recurrent launch's CTAs read from L2 each step: every CTA
    of a direction copies the h of the rows it multiplies (the staged kernel
    all rows, the dataflow kernel its row group's, the tensor-core kernel all
    rows in fp16); the in-cluster exchange moves h through shared memory."""
    def up(a, b):
        return (a + b - 1) // b * b
    k = geometry.get("kernel")
    D, H, N = case.dirs, case.hidden_size, case.batch
    ctas = geometry.get("unit_groups", 0)
    if k == 1:
        return float(D * ctas * up(N, 8) * H * 4)
    if k == 2:
        cr = max(1, geometry.get("row_groups", 1))
        nrp = up((N + cr - 1) // cr, 4 if (cr == 1 and N <= 4) else 8)   # rows per group, padded
        return float(D * ctas * cr * nrp * H * 4)
    if k == 3:
        return float(D * ctas * up(N, 8) * H * 2)
    return 0.0


def measure_l2_gbs(torch, nbytes=32 << 20, reps=10, trials=5):
    """Bandwidth (read + write bytes per second) of an elementwise kernel over
    a buffer pair that fits in the L2 (b = a * 1, so the SMs move the data),
    timed with CUDA events after warm-up passes; the best of a few trials
    (a peak for the roofline, not a mean disturbed by whatever else runs).
    55 launches in all (5 warm-up, 5 x 10 timed)."""
    a = torch.empty(nbytes // 4, device="cuda")
    b = torch.empty_like(a)
    a.fill_(1.0)
    for _ in range(5):
        torch.mul(a, 1.0, out=b)
    best = 0.0
    for _ in range(trials):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            torch.mul(a, 1.0, out=b)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        best = max(best, 2.0 * nbytes * reps / (ms / 1e3) / 1e9)
    return best


# The sources each kernel is compiled from (its translation units and the
# headers its code comes from; the staged kernel's units also include the
# dataflow header, none of whose code the staged kernel uses): a committed
# traffic figure is keyed by their digest, so it stays valid while that
# kernel's code is unchanged.
_COMMON = ["tma.cuh", "exact_math.cuh", "io_types.cuh", "rnn_internal.h"]
KERNEL_SOURCES = {
    "rnn_recurrent_kernel": ["k_recur.cuh", "k_recur_rnn.cu", "k_recur_gru.cu", "k_recur_lstm.cu"] + _COMMON,
    "rnn_dataflow_kernel": ["k_recur.cuh", "k_recur2.cuh", "k_recur_rnn.cu", "k_recur_gru.cu", "k_recur_lstm.cu",
                            "k_clus_rnn.cu", "k_clus_gru.cu", "k_clus_lstm.cu"] + _COMMON,
    "rnn_tc_kernel": ["k_recur_tc.cu", "k_recur.cuh"] + _COMMON,
    "rnn_wavefront_kernel": ["k_wave.cuh", "k_wave_rnn.cu", "k_wave_gru.cu", "k_wave_lstm.cu",
                             "k_recur.cuh"] + _COMMON,
    "proj_tma_kernel": ["k_proj.cu", "exact_math.cuh", "tma.cuh", "rnn_internal.h"],
    "proj_tc_kernel": ["k_proj_tc.cu", "tma.cuh", "rnn_internal.h"],
    "rnn_cell_kernel": ["k_cell.cu", "exact_math.cuh", "rnn_internal.h"],
}


def code_only(text):
    """C/C++/CUDA source without its comments and blank space: two sources
    that differ only there build the same kernels (line numbers aside)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"' or c == "'":                      # a string or character literal, kept whole
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            while i < n and text[i] != "\n":
                i += 1
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def source_digest(kernel, read=None):
    """Digest of the code a kernel (by its name) is built from, comments and
    blank space dropped: a committed ncu traffic figure applies only while
    it is unchanged.  `read(name)` supplies a source's text (default: the
    tree's file)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "onnx_recurrent_gb300", "csrc")
    if read is None:
        def read(name):
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                return f.read()
    for name in KERNEL_SOURCES[kernel]:
        h.update(name.encode() + code_only(read(name)).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel, workload, mode, digest):
    """DRAM bytes per launch from a committed ncu summary of the same sources."""
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    for name in sorted(os.listdir(pdir)):
        if not name.endswith(".md"):
            continue
        with open(os.path.join(pdir, name)) as f:
            text = f.read()
        for m in re.finditer(r"traffic_key:\s*(\S+)\s+(\S+)\s+(\S+)\s+(\S+)\s+(\d+)", text):
            if m.group(1) == kernel and m.group(2) == workload and m.group(3) == mode and m.group(4) == digest:
                return int(m.group(5))
    return None


# ------------------------------------------------------------ our arm

class SequenceJob:
    """One rnn_run of a sequence-operator workload per step."""

    def __init__(self, args, orc, torch):
        from onnx_recurrent_gb300.synth import PROFILE_WORKLOADS, WORKLOADS, workload
        self.case = c = workload(args.workload, lbr=args.lbr)
        self.host = {k: v for k, v in c.tensors().items() if v is not None}
        self.plan = orc.rnn_plan_create(c.op, c.direction, c.hidden_size, c.input_size,
                                        activations=c.activations, alpha=c.alpha, beta=c.beta,
                                        clip=c.clip, layout=c.layout,
                                        linear_before_reset=c.linear_before_reset,
                                        input_forget=c.input_forget)
        self.out_shapes = [c.y_shape(), c.state_shape()] + ([c.state_shape()] if c.op == "LSTM" else [])
        self.cells = c.cell_steps()
        self.rec_flops, self.proj_flops, _ = algorithmic(c)
        desc = WORKLOADS.get(args.workload, PROFILE_WORKLOADS.get(args.workload, ""))
        self.config = {"workload": args.workload, "description": desc,
                       "op": c.op, "direction": c.direction, "seq": c.seq, "batch": c.batch,
                       "input": c.input_size, "hidden": c.hidden_size,
                       "valid_cell_steps_per_step": c.valid_cell_steps()}
        self.orc = orc

    def run(self, dv, outs, stream):
        Yc = outs[2] if len(outs) > 2 else None
        self.orc.rnn_run(self.plan, dv["X"], dv["W"], dv["R"], dv.get("B"), dv.get("sequence_lens"),
                         dv.get("initial_h"), dv.get("initial_c"), dv.get("P"), outs[0], outs[1], Yc, stream)

    def cpu_baseline(self):
        return cpu_baseline(self.case)


class CellJob:
    """One rnn_cell_run (RNNCell-3, a single step of batch rows) per step."""

    def __init__(self, args, orc, torch):
        from onnx_recurrent_gb300.synth import CELL_WORKLOADS, cell_workload
        self.case = c = cell_workload(args.workload)
        self.host = c.tensors()
        self.plan = orc.rnn_cell_plan_create(c.hidden_size, c.input_size, activation=c.activation, clip=c.clip)
        self.out_shapes = [(c.batch, c.hidden_size)]
        self.cells = c.batch
        self.rec_flops = 2.0 * c.batch * c.hidden_size * c.hidden_size
        self.proj_flops = 2.0 * c.batch * c.hidden_size * c.input_size
        self.config = {"workload": args.workload, "description": CELL_WORKLOADS[args.workload],
                       "op": "RNNCell", "batch": c.batch, "input": c.input_size, "hidden": c.hidden_size,
                       "activation": c.activation}
        self.orc = orc

    def run(self, dv, outs, stream):
        self.orc.rnn_cell_run(self.plan, dv["X"], dv["H"], dv["W"], dv["R"], dv["B"], outs[0], stream)

    def cpu_baseline(self, budget_s=12.0):
        """The oracle's cell, single-threaded, whole batch per call, repeated
        while the time spent stays under about `budget_s`."""
        import oracle
        c = self.case
        oracle.build()
        calls = 0
        t0 = time.perf_counter()
        while True:
            oracle.rnn_cell(c.hidden_size, c.input_size, c.X, c.H, c.W, c.R, c.B, activation=c.activation,
                            clip=float("inf") if c.clip is None else c.clip)
            calls += 1
            dt = time.perf_counter() - t0
            if dt + dt / calls > budget_s:
                break
        return {"value": round(calls * c.batch / dt, 2), "unit": UNIT, "cores": 1, "kind": "oracle",
                "sample": f"{calls} calls over all {c.batch} batch rows, {dt:.1f} s"}


class StackJob:
    """One rnn_stack_run of a stack workload per step; the metric counts every
    layer's cell-steps."""

    def __init__(self, args, orc, torch):
        from onnx_recurrent_gb300.synth import STACK_WORKLOADS, stack_workload
        self.cases = cs = stack_workload(args.workload)
        self.case = cs[0]
        self.host = {"X": cs[0].X}
        if cs[0].sequence_lens is not None:
            self.host["sequence_lens"] = cs[0].sequence_lens
        for i, c in enumerate(cs):
            for k in ("W", "R", "B", "P", "initial_h", "initial_c"):
                v = getattr(c, k)
                if v is not None:
                    self.host[f"{k}{i}"] = v
        self.layer_plans = [orc.rnn_plan_create(c.op, c.direction, c.hidden_size, c.input_size, clip=c.clip,
                                                layout=c.layout, linear_before_reset=c.linear_before_reset)
                            for c in cs]
        # the first layer's plan carries a wavefront run's timing, geometry and status
        self.plan = self.layer_plans[0]
        self.stack = None
        last = cs[-1]
        self.out_shapes = [last.y_shape()] + [c.state_shape() for c in cs] + \
                          [c.state_shape() for c in cs if c.op == "LSTM"]
        self.cells = sum(c.cell_steps() for c in cs)
        rows_steps = cs[0].valid_cell_steps() // cs[0].dirs      # the shared lengths, summed
        self.rec_flops = sum(2.0 * rows_steps * c.dirs * c.gates * c.hidden_size ** 2 for c in cs)
        self.proj_flops = sum(algorithmic(c)[1] for c in cs)
        # a wavefront run forms every layer's input product but the first inside
        # the recurrent launch (the valid steps only, as for the recurrent product)
        self.wave_rec_flops = self.rec_flops + sum(2.0 * rows_steps * c.dirs * c.gates * c.hidden_size * c.input_size
                                                   for c in cs[1:])
        self.wave_proj_flops = algorithmic(cs[0])[1]
        self.config = {"workload": args.workload, "description": STACK_WORKLOADS[args.workload],
                       "layers": [{"op": c.op, "direction": c.direction, "input": c.input_size,
                                   "hidden": c.hidden_size} for c in cs],
                       "seq": cs[0].seq, "batch": cs[0].batch,
                       "valid_cell_steps_per_step": sum(rows_steps * c.dirs for c in cs)}
        self.orc = orc

    def set_mode(self, mode, io):
        for p in self.layer_plans:
            self.orc.rnn_plan_set_mode(p, mode)
            self.orc.rnn_plan_set_io_type(p, io)
        self.stack = self.orc.rnn_stack_create(self.layer_plans)

    def run(self, dv, outs, stream):
        cs = self.cases
        L = len(cs)
        g = lambda k: [dv.get(f"{k}{i}") for i in range(L)]
        yh = outs[1:1 + L]
        lstm = [i for i, c in enumerate(cs) if c.op == "LSTM"]
        yc = [None] * L
        for j, i in enumerate(lstm):
            yc[i] = outs[1 + L + j]
        self.orc.rnn_stack_run(self.stack, dv["X"], g("W"), g("R"), g("B"), dv.get("sequence_lens"),
                               g("initial_h"), g("initial_c"), g("P"), outs[0], yh, yc, stream)

    def launches(self):
        return self.orc.rnn_stack_last_launch_count(self.stack)

    def wavefront(self):
        return self.orc.rnn_stack_last_wavefront(self.stack)

    def cpu_baseline(self):
        return {"value": None, "unit": UNIT, "cores": 1, "kind": "oracle",
                "sample": "not run for stacks (the single-layer workloads carry the oracle baseline)"}


def run_ours(args, ws, rank, local):
    import torch

    import onnx_recurrent_gb300 as orc
    from onnx_recurrent_gb300.synth import CELL_WORKLOADS, STACK_WORKLOADS

    torch.cuda.set_device(local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if rank == 0:
        orc.build()
    if dist:
        dist.barrier()
    orc.build()
    orc.load()

    job = (CellJob if args.workload in CELL_WORKLOADS else
           StackJob if args.workload in STACK_WORKLOADS else SequenceJob)(args, orc, torch)
    plan = job.plan
    if isinstance(job, StackJob):
        job.set_mode(args.mode, args.io)
        orc.rnn_stack_set_wavefront(job.stack, 0 if args.layer_by_layer else (2 if args.wavefront else 1))
        if args.launch:        # the first plan's override: its unit_groups cap the CTAs per wavefront layer
            orc.rnn_plan_set_launch(job.layer_plans[0], *[int(v) for v in args.launch.split(",")])
    else:
        orc.rnn_plan_set_mode(plan, args.mode)
        orc.rnn_plan_set_io_type(plan, args.io)
        if args.launch:
            orc.rnn_plan_set_launch(plan, *[int(v) for v in args.launch.split(",")])
    act = orc.rnn.io_dtype(plan)
    is_io = lambda k: k == "X" or k.startswith("initial_")   # the tensors in the I/O type (weights stay fp32)
    dev = {k: (torch.from_numpy(v).to(act) if is_io(k) else torch.from_numpy(v)).cuda()
           for k, v in job.host.items()}
    outs = [torch.empty(sh, device="cuda", dtype=act) for sh in job.out_shapes]
    flush = torch.empty(FLUSH_BYTES // 4, device="cuda")
    stream = torch.cuda.current_stream()
    l2_gbs = measure_l2_gbs(torch)

    def step():
        job.run(dev, outs, stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    orc.rnn_plan_sync(plan)
    launches_per_step = job.launches() if isinstance(job, StackJob) else orc.rnn_plan_last_launch_count(plan)
    geometry = orc.rnn_plan_get_launch(plan)
    if isinstance(job, StackJob):
        job.config["wavefront"] = job.wavefront()
        if job.config["wavefront"]:
            job.rec_flops, job.proj_flops = job.wave_rec_flops, job.wave_proj_flops

    # ---- timed region: inputs resident, L2 flushed between steps
    timed = job.layer_plans if isinstance(job, StackJob) else [plan]
    for p_ in timed:
        orc.rnn_plan_set_timing(p_, True)
    K = args.steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(K):
        flush.zero_()
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if dist:
        dist.barrier()
    if sampler:
        time.sleep(0.25)
        sampler.stop()
    orc.rnn_plan_sync(plan)
    step_ms = [a.elapsed_time(b) for a, b in evs]
    total_ms = sum(step_ms)
    median_ms = statistics.median(step_ms)
    kern_ms, runs = {}, 0
    for p_ in timed:                       # a stack: each kernel kind summed over the layers
        orc.rnn_plan_sync(p_)
        km, r_ = orc.rnn_plan_timing_totals(p_)
        runs = max(runs, r_)               # (a wavefront run is timed on the first layer's plan alone)
        for k_, v_ in km.items():
            kern_ms[k_] = kern_ms.get(k_, 0.0) + v_
        orc.rnn_plan_set_timing(p_, False)

    # ---- end to end: pinned host inputs -> device -> run -> host outputs,
    # every input (weights included) uploaded afresh each step, pipelined the
    # way a serving loop runs: uploads on one copy stream, runs on the compute
    # stream, downloads on another copy stream, with two sets of device
    # buffers, so batch i+1's upload and batch i-1's download ride the copy
    # engines while batch i computes
    host_in = {k: v.cpu().pin_memory() for k, v in dev.items()}
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    devs = [dev, {k: torch.empty_like(v) for k, v in dev.items()}]
    bufs = [outs, [torch.empty_like(t) for t in outs]]
    host_outs = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs] for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_outs[0])
    E = K
    ev = lambda: torch.cuda.Event()
    in_done, run_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    torch.cuda.synchronize()
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    s_in.wait_event(e_start)
    s_out.wait_event(e_start)
    for i in range(E):
        j = i % 2
        dv, ov = devs[j], bufs[j]
        if i >= 2:
            s_in.wait_event(run_done[j])       # the run of batch i-2 has read these inputs
            stream.wait_event(out_done[j])     # batch i-2's outputs have left these buffers
        with torch.cuda.stream(s_in):
            for k, v in host_in.items():
                dv[k].copy_(v, non_blocking=True)
        in_done[j].record(s_in)
        stream.wait_event(in_done[j])
        job.run(dv, ov, stream)
        run_done[j].record(stream)
        s_out.wait_event(run_done[j])
        with torch.cuda.stream(s_out):
            for h, d in zip(host_outs[j], ov):
                h.copy_(d, non_blocking=True)
        out_done[j].record(s_out)
    for j in range(2):
        stream.wait_event(out_done[j])
    e_end.record(stream)
    torch.cuda.synchronize()
    orc.rnn_plan_sync(plan)
    e2e_ms = e_start.elapsed_time(e_end)

    if dist:
        total_ms, median_ms, e2e_ms = max_over_ranks([total_ms, median_ms, e2e_ms], dist, "cuda")
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    cells = job.cells
    value = job_value(cells, 1, ws, median_ms)
    e2e_value = job_value(cells, E, ws, e2e_ms)
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    sms = props.multi_processor_count
    smem_per_sm = int(getattr(props, "shared_memory_per_block_optin", 232448))
    peaks = measured_peaks()
    clock_mhz = float(peaks.get("sm_max_mhz", 2070.0))
    exact = args.mode == "exact"
    alu_peak = sms * 128 * (1 if exact else 2) * clock_mhz * 1e6          # FLOP/s
    rec_flops, proj_flops = job.rec_flops, job.proj_flops
    avg = {k: (v / runs if runs else 0.0) for k, v in kern_ms.items()}
    if isinstance(job, CellJob):
        avg = {"cell": avg["recurrence"]}      # one kernel, timed in the recurrence slot
    dominant = max(avg, key=avg.get)

    traffic_name = args.workload + (f"-lbr{args.lbr}" if args.lbr else "")   # the workload as profiles name it
    if isinstance(job, StackJob) and not job.wavefront():
        traffic_name += "-layers"      # a stack run layer by layer (its launches summed), not its wavefront

    def roof(kernel):
        ms = avg[kernel]
        if kernel == "cell":
            flops = rec_flops + proj_flops
            ach = flops / (ms / 1e3) / 1e12 if ms else 0.0
            return {"bound": "alu", "achieved": round(ach, 3), "peak": round(alu_peak / 1e12, 3),
                    "unit": "TFLOP/s", "frac": round(ach / (alu_peak / 1e12), 4) if ms else 0.0,
                    "traffic": profiled_traffic(kernel, traffic_name, args.mode, source_digest("rnn_cell_kernel")),
                    "kernel": "rnn_cell_kernel", "avg_ms": round(ms, 5), "algorithmic_flops_per_launch": flops,
                    "peak_note": f"{'no' if exact else 'fused'} multiply-add: {sms} SMs x 128 FP32 "
                                 f"lanes x {'1' if exact else '2'} FLOP x {clock_mhz:.0f} MHz (derived)"}
        if kernel == "recurrence" and geometry.get("kernel") == 3:
            # fp16 tensor-core products (tcgen05 kind::f16): the measured bf16
            # burst peak, fp16 and bf16 having the same nominal dense rate
            peak = float(peaks.get("bf16_tflops", 1900.0))
            traffic = profiled_traffic(kernel, traffic_name, args.mode, source_digest("rnn_tc_kernel"))
            sr = (step_roofline(job.case, args.mode, ms, sms, clock_mhz, l2_gbs, smem_per_sm,
                                h_bytes_per_step(geometry, job.case), tensor_tflops=peak)
                  if isinstance(job, SequenceJob) else None)
            if sr and sr["binding"] == "h":
                # every CTA copies all of h (fp16) each step: those bytes over L2
                nbytes = sr["h_bytes_per_step"] * sr["steps"]
                ach = nbytes / (ms / 1e3) / 1e9 if ms else 0.0
                return {"bound": "l2", "achieved": round(ach, 1), "peak": round(l2_gbs, 1), "unit": "GB/s",
                        "frac": sr["frac"], "traffic": traffic, "kernel": "rnn_tc_kernel", "avg_ms": round(ms, 5),
                        "algorithmic_bytes_per_launch": nbytes, "step_roofline": sr,
                        "peak_note": "of measured L2 bandwidth (an elementwise kernel, read + write, a 32 MiB "
                                     "pair); the tensor-core products alone would take "
                                     f"{sr['terms_us_per_step']['alu']:.2f} us a step against the measured bf16 "
                                     f"burst ({peak:.0f} TFLOP/s)"}
            ach = rec_flops / (ms / 1e3) / 1e12 if ms else 0.0
            out = {"bound": "tensor", "achieved": round(ach, 3), "peak": round(peak, 3), "unit": "TFLOP/s",
                   "frac": round(ach / peak, 4) if ms else 0.0, "traffic": traffic,
                   "kernel": "rnn_tc_kernel", "avg_ms": round(ms, 5), "algorithmic_flops_per_launch": rec_flops,
                   "peak_note": "of measured bf16 burst (fp16 operands, same nominal rate)"}
            if sr:
                out["step_roofline"] = sr
            return out
        if kernel == "recurrence":
            # kernel 5: the dataflow kernel's in-cluster instance (same name)
            name = {2: "rnn_dataflow_kernel", 4: "rnn_wavefront_kernel",
                    5: "rnn_dataflow_kernel"}.get(geometry.get("kernel"), "rnn_recurrent_kernel")
            traffic = profiled_traffic(kernel, traffic_name, args.mode, source_digest(name))
            sr = (step_roofline(job.case, args.mode, ms, sms, clock_mhz, l2_gbs, smem_per_sm,
                                h_bytes_per_step(geometry, job.case))
                  if isinstance(job, SequenceJob) else None)
            if sr and sr["binding"] == "chain":
                # each output's dependent adds bound the step: their rate
                # against one add per FP32_CHAIN_CYCLES at the SM clock
                adds = (sr["terms_us_per_step"]["chain"] * 1e-6 * clock_mhz * 1e6 / FP32_CHAIN_CYCLES) * sr["steps"]
                rate = adds / (ms / 1e3) if ms else 0.0
                peak = clock_mhz * 1e6 / FP32_CHAIN_CYCLES
                return {"bound": "latency", "achieved": round(rate / 1e6, 2), "peak": round(peak / 1e6, 2),
                        "unit": "M dependent adds/s per output", "frac": sr["frac"], "traffic": traffic,
                        "kernel": name, "avg_ms": round(ms, 5), "algorithmic_flops_per_launch": rec_flops,
                        "step_roofline": sr,
                        "peak_note": f"one FP32 add (or fused multiply-add) per {FP32_CHAIN_CYCLES:.0f} cycles "
                                     f"on each output's chain (k ascending) at {clock_mhz:.0f} MHz; frac is the "
                                     "step roofline's (per-step max of the ALU, shared-memory, L2 and chain terms)"}
            if sr and sr["binding"] in ("l2", "h"):
                # R's streamed part (it does not fit in the SMs' shared memory)
                # or the copies of h bound the step: bytes from L2 against the
                # measured L2 copy rate
                nbytes = (sr["r_streamed_bytes_per_step"] if sr["binding"] == "l2"
                          else sr["h_bytes_per_step"]) * sr["steps"]
                ach = nbytes / (ms / 1e3) / 1e9 if ms else 0.0
                return {"bound": "l2", "achieved": round(ach, 1), "peak": round(l2_gbs, 1), "unit": "GB/s",
                        "frac": sr["frac"], "traffic": traffic, "kernel": name, "avg_ms": round(ms, 5),
                        "algorithmic_bytes_per_launch": nbytes, "step_roofline": sr,
                        "peak_note": "of measured L2 bandwidth (an elementwise kernel, read + write, a 32 MiB pair)"}
            ach = rec_flops / (ms / 1e3) / 1e12 if ms else 0.0
            out = {"bound": "alu", "achieved": round(ach, 3), "peak": round(alu_peak / 1e12, 3),
                   "unit": "TFLOP/s", "frac": round(ach / (alu_peak / 1e12), 4) if ms else 0.0,
                   "traffic": traffic, "kernel": name, "avg_ms": round(ms, 5),
                   "algorithmic_flops_per_launch": rec_flops,
                   "peak_note": f"{'no' if exact else 'fused'} multiply-add: {sms} SMs x 128 FP32 "
                                f"lanes x {'1' if exact else '2'} FLOP x {clock_mhz:.0f} MHz (derived)"}
            if sr:
                out["step_roofline"] = sr
            return out
        if kernel == "projection" and args.mode in ("tf32", "bf16"):
            # tensor cores: the measured bf16 burst peak, scaled by the nominal
            # TF32 : bf16 ratio (1.1 : 2.25 PFLOP/s dense) for TF32: the TF32
            # peak is derived from the bf16 measurement, not measured itself
            bf16 = float(peaks.get("bf16_tflops", 1900.0))
            peak = bf16 if args.mode == "bf16" else bf16 * 1.1 / 2.25
            ach = proj_flops / (ms / 1e3) / 1e12 if ms else 0.0
            return {"bound": "tensor", "achieved": round(ach, 3), "peak": round(peak, 3), "unit": "TFLOP/s",
                    "frac": round(ach / peak, 4) if ms else 0.0,
                    "traffic": profiled_traffic(kernel, traffic_name, args.mode, source_digest("proj_tc_kernel")),
                    "kernel": "proj_tc_kernel", "avg_ms": round(ms, 5), "algorithmic_flops_per_launch": proj_flops,
                    "peak_note": "of measured bf16 burst" + ("" if args.mode == "bf16" else
                                                             " x 1.1/2.25 (TF32: derived from the bf16 "
                                                             "measurement by the nominal dense-rate ratio)")}
        if kernel == "projection":
            ach = proj_flops / (ms / 1e3) / 1e12 if ms else 0.0
            return {"bound": "alu", "achieved": round(ach, 3), "peak": round(alu_peak / 1e12, 3),
                    "unit": "TFLOP/s", "frac": round(ach / (alu_peak / 1e12), 4) if ms else 0.0,
                    "traffic": profiled_traffic(kernel, traffic_name, args.mode, source_digest("proj_tma_kernel")),
                    "kernel": "proj_tma_kernel", "avg_ms": round(ms, 5),
                    "algorithmic_flops_per_launch": proj_flops}
        return {"kernel": kernel, "avg_ms": round(ms, 5)}

    clocks = sampler.summary(t0, t1) if sampler else None
    result = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(median_ms, 5),
        "ms_per_step_mean": round(total_ms / K, 5), "value_from": "median step time over the timed steps",
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": {"exact": "f32", "fast": "f32", "tf32": "f32 (tf32 projection)",
                  "bf16": "f32 (bf16 projection)"}[args.mode] + ("" if args.io == "f32" else f", {args.io} I/O"),
        "data": "synthetic (seeded, see synth.py)",
        "config": dict(job.config, mode=args.mode, io=args.io, l2="flushed between timed steps (256 MiB write)",
                       parallelism=f"replicas x{ws}", geometry=geometry),
        "roofline": roof(dominant),
        "kernels": {k: roof(k) for k in avg if avg[k] > 0},
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "pipeline": "uploads, runs and downloads on 3 streams, 2 buffer sets: "
                                                      "copies overlap compute; inputs re-uploaded every step"},
        "gpu_launches": launches_per_step * K,
        "clocks": clocks,
        "impl": "ours",
    }
    if not args.no_cpu_baseline and ws == 1:
        result["cpu_baseline"] = job.cpu_baseline()
    emit(result, args.out)
    if dist:
        dist.destroy_process_group()


def cpu_baseline(case, budget_s=12.0):
    """The oracle, as it stands, single-threaded on this host, on a bounded
    sample of the workload: its first batch rows, or whole passes over the
    batch repeated while the time spent stays under about `budget_s`; where
    one row alone would take longer, the first steps of row 0 (a sequence
    cut short: the same work per step).  The sample is sized from the time
    per valid step of the longest row, measured on its first steps."""
    import numpy as np

    import oracle
    from oracle import rnn as oracle_rnn
    a = case.attrs()
    full = case.tensors()
    S, N = case.seq, case.batch
    L = np.full(N, S, np.int64) if case.sequence_lens is None else np.asarray(case.sequence_lens, np.int64)

    def cut(steps):
        t = dict(full)
        t["X"] = full["X"][:steps] if case.layout == 0 else full["X"][:, :steps]
        if full["sequence_lens"] is not None:
            t["sequence_lens"] = np.minimum(full["sequence_lens"], steps).astype(full["sequence_lens"].dtype)
        return t

    def rows(t, b, e):
        return oracle_rnn(a["op"], a["direction"], a["hidden_size"], a["input_size"], t["X"], t["W"],
                          t["R"], B=t["B"], sequence_lens=t["sequence_lens"], initial_h=t["initial_h"],
                          initial_c=t["initial_c"], P=t["P"], activations=a["activations"],
                          alpha=a["alpha"], beta=a["beta"], clip=a["clip"], layout=a["layout"],
                          linear_before_reset=a["linear_before_reset"],
                          input_forget=a["input_forget"], rows=(b, e))
    oracle.build()
    k = int(np.argmax(L))
    s0 = int(min(S, 16))
    probe = cut(s0)
    rows(probe, k, k + 1)                           # first call: loads the compiled oracle
    t0 = time.perf_counter()
    rows(probe, k, k + 1)
    per_step = (time.perf_counter() - t0) / max(1, min(int(L[k]), s0))
    if per_step * max(1, int(L[k])) > budget_s:
        steps = int(max(1, min(S, budget_s / per_step)))
        t = cut(steps)
        t0 = time.perf_counter()
        rows(t, 0, 1)
        dt = time.perf_counter() - t0
        valid = int(min(L[0], steps)) * case.dirs
        return {"value": round(steps * case.dirs / dt, 2), "unit": UNIT, "cores": 1, "kind": "oracle",
                "sample": f"batch row 0, first {steps} of {S} steps ({valid} valid cell-steps), {dt:.1f} s"}
    est = np.cumsum(np.maximum(L, 1)) * per_step    # estimated time of rows 0..i
    n = int(min(N, max(1, np.searchsorted(est, budget_s, side="right"))))
    passes = 0
    t0 = time.perf_counter()
    while True:
        rows(full, 0, n)
        passes += 1
        dt = time.perf_counter() - t0
        if n < N or dt + dt / passes > budget_s:
            break
    valid = int(L[:n].sum()) * case.dirs
    what = (f"{passes} passes over all {n} batch rows" if passes > 1 else
            ("all batch rows" if n == N else f"batch rows 0..{n - 1}"))
    return {"value": round(passes * n * S * case.dirs / dt, 2), "unit": UNIT, "cores": 1,
            "kind": "oracle", "sample": f"{what} of the workload, all {S} steps "
                                        f"({passes * valid} valid cell-steps), {dt:.1f} s"}


# ------------------------------------------------------ reference arm

def run_reference(args, ws, rank):
    if rank != 0:
        return
    import oracle
    from onnx_recurrent_gb300.synth import CELL_WORKLOADS, WORKLOADS, cell_workload, workload
    if args.workload in CELL_WORKLOADS:
        return run_reference_cell(args, ws)
    case = workload(args.workload, lbr=args.lbr)
    a = case.attrs()
    t = case.tensors()
    oracle.build()

    def one_row(r):
        oracle.rnn(a["op"], a["direction"], a["hidden_size"], a["input_size"], t["X"], t["W"],
                   t["R"], B=t["B"], sequence_lens=t["sequence_lens"], initial_h=t["initial_h"],
                   initial_c=t["initial_c"], P=t["P"], activations=a["activations"],
                   alpha=a["alpha"], beta=a["beta"], clip=a["clip"], layout=a["layout"],
                   linear_before_reset=a["linear_before_reset"], input_forget=a["input_forget"],
                   rows=(r, r + 1))
    for i in range(args.warmup):
        one_row(i % case.batch)
    t0 = time.perf_counter()
    for i in range(args.steps):
        one_row(i % case.batch)
    dt = time.perf_counter() - t0
    per_step = case.seq * case.dirs
    value = per_step * args.steps / dt
    emit({"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
          "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 3),
          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
          "data": "synthetic (seeded, see synth.py)",
          "config": {"workload": args.workload, "description": WORKLOADS.get(args.workload, ""),
                     "mode": "exact", "sample": "one batch row per step"},
          "impl": "reference",
          "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": 1, "kind": "oracle",
                           "sample": f"one batch row ({case.seq} steps) of the workload per step"},
          "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0,
                  "d2h_bytes_per_step": 0},
          "gpu_launches": 0}, args.out)


def run_reference_cell(args, ws):
    """The oracle's cell on one batch row of the cell workload per step."""
    import oracle
    from onnx_recurrent_gb300.synth import CELL_WORKLOADS, cell_workload
    c = cell_workload(args.workload)
    oracle.build()
    clip = float("inf") if c.clip is None else c.clip

    def one_row(r):
        oracle.rnn_cell(c.hidden_size, c.input_size, c.X[r:r + 1], c.H[r:r + 1], c.W, c.R, c.B,
                        activation=c.activation, clip=clip)
    for i in range(args.warmup):
        one_row(i % c.batch)
    t0 = time.perf_counter()
    for i in range(args.steps):
        one_row(i % c.batch)
    dt = time.perf_counter() - t0
    value = args.steps / dt
    emit({"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
          "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 3),
          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
          "data": "synthetic (seeded, see synth.py)",
          "config": {"workload": args.workload, "description": CELL_WORKLOADS[args.workload],
                     "mode": "exact", "sample": "one batch row per step"},
          "impl": "reference",
          "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": 1, "kind": "oracle",
                           "sample": "one batch row of the cell workload per step"},
          "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
          "gpu_launches": 0}, args.out)


def main():
    args = parse_args()
    ws, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, ws, rank)
    else:
        run_ours(args, ws, rank, local)


if __name__ == "__main__":
    main()
