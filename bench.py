#!/usr/bin/env python3
"""Throughput of the SNACK sparse layer's hot path on GB300.

One step = forward (Y = X W^T), backward-input (dX = dY W) and
backward-weight (dW at the stored entries) of every layer of the workload at
every batch size of the workload, through the library's C ABI.  The metric
is effective GFLOP/s, 2 * nnz * batch per SpMM, three SpMMs per (layer,
batch).  Default workload: the 10000x10000 single-layer sweep (the paper's
§4.2 training cycle layer) at 90, 95 and 99 % sparsity (10 M, 5 M and 1 M
stored entries), batch 1, 4, 8, 16 and 64.

Timing: W warm-up steps, then K steps, each replayed from a CUDA graph of
the step and timed with CUDA events on the launching stream; between steps
a 256 MiB buffer (about twice the L2) is written and then read back, so
every step starts with a cold L2 holding only clean lines (the flush's own
write-backs are not charged to the step).  Barrier + synchronize on both
sides; the max over ranks is reported.  Under torchrun every rank runs its
own replica (weak scaling, no collective on the data path).

Also reported: the roofline of the dominant op (metric bytes / measured
duration against the measured HBM copy bandwidth) and of the ops at the
95 % / batch >= 8 operating point, an end-to-end number through the same
calls with host buffers (one pinned H2D copy of every X and dY, one D2H copy
of every Y, dX and dW, inside the timed region), the CPU oracle on the host
cores on a bounded sample (single-threaded, and its all-cores copy), the SM
clocks sampled during the timed region, and the kernel launches.  The per-op
table (each op replayed from its own CUDA graph, 10 untimed then 50 timed
replays, each after an L2 flush; mean and median microseconds) gives
GFLOP/s, GB/s of the metric's bytes, the fraction of the measured copy peak,
and gather_gbs: the 4 * B bytes per stored entry of operand rows every op
gathers (through L1 or shared memory), the bound that takes over from HBM as
B grows.  It also times the Adam step (snack_adam_step) of each layer and
batch, a training step (forward, backward-input, Adam step) on the 95 %
layer, and the forward / backward ops of the GPT-2 MLP layers and the skewed
8192x8192 layer; none of these are part of the metric.

`--impl reference` times the CPU oracle instead (the deliberately slow
reference arm), on a bounded sample of the same workload and metric.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "SpMM fwd+bwd GFLOP/s (2·nnz·B) and % of HBM roofline at 90–99% sparsity"
UNIT = "GFLOP/s"
FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------ ranks

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(backend: str):
    import torch.distributed as dist
    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        os.environ.setdefault("MASTER_PORT", "29533")
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return rank, world


def reduce_max(x: float, device=None) -> float:
    """Max of x over ranks (x itself at world size 1)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) >= 9 and p[1].replace(".", "").isdigit():
                    rows.append(p)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows]
        smax = max(float(r[2]) for r in rows)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(float(r[3]) for r in rows
                                                         if r[3].replace(".", "").isdigit())}


# ------------------------------------------------------------------ workload

def make_cases(workload_name: str, batches=None, seed: int = 0):
    """Host-side inputs of a workload: per layer the COO triple; per batch X, dY."""
    import workloads
    wl = workloads.workload(workload_name, seed)
    cases = []
    for L in wl.layers:
        row, col, val = L.coo()
        acts = {B: L.activations(B) for B in (batches or wl.batches)}
        cases.append(dict(layer=L, row=row, col=col, val=val, acts=acts))
    return wl, cases


def flops_per_step(cases) -> float:
    return float(sum(3 * 2 * c["layer"].nnz * B for c in cases for B in c["acts"]))


def metric_bytes(op: str, nnz: int, out: int, inp: int, B: int) -> int:
    """Minimal bytes of one op: nnz*12 + the dense operands it reads / writes."""
    if op == "fwd":
        return nnz * 12 + 4 * B * (inp + out)
    if op == "bwd_input":
        return nnz * 12 + 4 * B * (out + inp)
    if op == "adam_step":  # column 4 B, value and two moments read and written 24 B
        return nnz * 28 + 4 * B * (inp + out)
    return nnz * 12 + 4 * B * (inp + out)  # bwd_weight: X and dY read, dW in the 12


def flush_l2(buf):
    """Evict the workload from L2 before a timed step: write a buffer twice
    the size of L2, then read it back.  The read pass writes the dirty lines
    back to HBM and leaves L2 holding clean lines of the flush buffer, so the
    timed step starts cold without paying for the flush's own write-backs."""
    buf.fill_(1.0)
    buf.sum()


def read_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_sha(csrc: str | None = None) -> str:
    """Hash of the CUDA sources' code: comments and whitespace are removed
    first, so that an edit to a comment keeps recorded counters valid while
    any change to the code itself does not."""
    h = hashlib.sha256()
    csrc = csrc or os.path.join(ROOT, "coo_spmm_sparse_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                code = f.read()
            code = re.sub(r"/\*.*?\*/", " ", code, flags=re.S)
            code = re.sub(r"//[^\n]*", " ", code)
            code = " ".join(code.split())
            h.update(name.encode() + b"\0" + code.encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu capture, if the kernel
    sources are unchanged since it was taken; else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    for r in rec.get("entries", []):
        if r.get("op") == kernel and r.get("workload") == workload and \
                r.get("source_sha") == kernel_source_sha():
            return r.get("bytes_per_launch")
    return None


# ------------------------------------------------------------------ our arm

def _upload(cases, dev, stream, sn):
    import torch
    with torch.cuda.stream(stream):
        for c in cases:
            L = c["layer"]
            c["h"] = sn.snack_create(L.out, L.inp, c["row"], c["col"], c["val"], stream=stream)
            c["dev"] = {}
            for B, (X, dY) in c["acts"].items():
                c["dev"][B] = dict(X=torch.from_numpy(X).to(dev), dY=torch.from_numpy(dY).to(dev),
                                   Y=torch.empty(B, L.out, device=dev),
                                   dX=torch.empty(B, L.inp, device=dev),
                                   dW=torch.empty(L.nnz, device=dev))
    torch.cuda.synchronize()


def time_graph(fn, stream, flush, reps=50, warm=10):
    """Mean and median microseconds of `fn` replayed from a CUDA graph between
    events on `stream`, after an L2 flush each time."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            fn()
        for _ in range(warm):
            g.replay()
        ts = []
        for _ in range(reps):
            flush_l2(flush)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            ts.append((e0, e1))
    torch.cuda.synchronize()
    del g
    durs = [a.elapsed_time(b) * 1e3 for a, b in ts]
    return statistics.mean(durs), statistics.median(durs)


def op_rows(cases, sn, stream, flush, ops=("fwd", "bwd_input", "bwd_weight", "adam_step"),
            workload=None):
    """Per-op table of one workload's layers and batches."""
    import torch
    rows = []

    def run_op(op, c, d):
        if op == "fwd":
            sn.snack_forward(c["h"], d["X"], d["Y"], stream=stream)
        elif op == "bwd_input":
            sn.snack_backward_input(c["h"], d["dY"], d["dX"], stream=stream)
        elif op == "bwd_weight":
            sn.snack_backward_weight(c["h"], d["X"], d["dY"], d["dW"], stream=stream)
        else:  # Adam step (gradient + update); not part of the metric
            sn.snack_adam_step(c["h"], d["X"], d["dY"], lr=1e-3, step=1, stream=stream)

    for c in cases:
        L = c["layer"]
        for B, d in c["dev"].items():
            for op in ops:
                if op == "adam_step":  # its first call allocates the moments
                    with torch.cuda.stream(stream):
                        run_op(op, c, d)
                    torch.cuda.synchronize()
                us, med = time_graph(lambda: run_op(op, c, d), stream, flush)
                if op == "adam_step":  # the steps changed the values: re-derive
                    sn.snack_values_changed(c["h"])  # their column-ordered copy
                    torch.cuda.synchronize()
                nbytes = metric_bytes(op, L.nnz, L.out, L.inp, B)
                plan_op = {"fwd": 0, "bwd_input": 1}.get(op, 2)  # dW and Adam: rows
                bw, lanes, segs = sn.snack_plan(c["h"], plan_op, B)
                r = dict(op=op, layer=L.name, shape=f"{L.out}x{L.inp}", nnz=L.nnz, B=B,
                         us=round(us, 3), us_median=round(med, 3),
                         gflops=round(2 * L.nnz * B / us / 1e3, 2),
                         gbs=round(nbytes / us / 1e3, 1), bytes=nbytes,
                         gather_gbs=round(4 * B * L.nnz / us / 1e3, 1),
                         plan=dict(slice=bw, lanes=lanes, segments=segs))
                if workload:
                    r["workload"] = workload
                rows.append(r)
    return rows


def train_step_rows(case, sn, stream, flush, batches=(1, 16)):
    """One training step of a layer (forward, backward-input, Adam step), two
    ways: dX reading the values through the column permutation (the
    column-ordered copy left stale by the step) and dX reading the copy,
    re-derived right after the step.  Not part of the metric."""
    import torch
    rows = []
    c = case
    L = c["layer"]
    h = c["h"]
    for B in batches:
        d = c["dev"][B]
        for mode in ("permutation", "refreshed_copy"):
            def fn():
                sn.snack_forward(h, d["X"], d["Y"], stream=stream)
                sn.snack_backward_input(h, d["dY"], d["dX"], stream=stream)
                sn.snack_adam_step(h, d["X"], d["dY"], lr=1e-3, step=1, stream=stream)
                if mode == "refreshed_copy":
                    sn.snack_values_changed(h, stream=stream)
            with torch.cuda.stream(stream):
                sn.snack_adam_step(h, d["X"], d["dY"], lr=1e-3, step=1, stream=stream)
                if mode == "refreshed_copy":
                    sn.snack_values_changed(h, stream=stream)
            torch.cuda.synchronize()
            us, med = time_graph(fn, stream, flush)
            rows.append(dict(op="train_step", mode=mode, layer=L.name, shape=f"{L.out}x{L.inp}",
                             nnz=L.nnz, B=B, us=round(us, 3), us_median=round(med, 3),
                             gflops=round(3 * 2 * L.nnz * B / us / 1e3, 2)))
    sn.snack_values_changed(h)
    torch.cuda.synchronize()
    return rows


def run_ours(args):
    import numpy as np
    import torch

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    rank, world = dist_init("nccl")
    dev = torch.device("cuda", local)
    import coo_spmm_sparse_gb300 as sn

    wl, cases = make_cases(args.workload, args.batches, args.seed)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    _upload(cases, dev, stream, sn)

    def step():
        for c in cases:
            for B, d in c["dev"].items():
                sn.snack_forward(c["h"], d["X"], d["Y"], stream=stream)
                sn.snack_backward(c["h"], d["X"], d["dY"], d["dX"], d["dW"], stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            step()
    torch.cuda.synchronize()

    # CUDA graph of one step (the calls only launch kernels: capturable).
    n0 = sn.snack_launch_count()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    launches_per_step = sn.snack_launch_count() - n0
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(3):
            graph.replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for e0, e1 in evs:
            flush_l2(flush)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    step_ms = [e0.elapsed_time(e1) for e0, e1 in evs]
    total_ms = reduce_max(sum(step_ms), dev)
    fl = flops_per_step(cases)
    value = world * fl * args.steps / (total_ms / 1e3) / 1e9
    del graph

    # Per-op durations -> dominant op, roofline.  Each op is replayed from its
    # own CUDA graph between events on the launching stream, after an L2
    # flush that keeps the GPU busy while the host queues the replay.
    ops = op_rows(cases, sn, stream, flush)
    train = []
    c95 = next((c for c in cases if c["layer"].name == "large95"), None)
    if c95 is not None and not args.no_extra_ops:
        train = train_step_rows(c95, sn, stream, flush,
                                [B for B in (1, 16) if B in c95["dev"]])
    extra = []
    if not args.no_extra_ops:
        for name in [w for w in args.extra_ops.split(",") if w and w != args.workload]:
            _, xc = make_cases(name, None, args.seed)
            _upload(xc, dev, stream, sn)
            extra += op_rows(xc, sn, stream, flush, ops=("fwd", "bwd_input", "bwd_weight"),
                             workload=name)
            for c in xc:
                c["h"].close()
            del xc
    peak, peak_kind = read_peak()
    for o in ops + extra:
        o["frac"] = round(o["gbs"] / peak, 4)
    dom = max((o for o in ops if o["op"] != "adam_step"), key=lambda o: o["us"])
    tr = recorded_traffic(f"{dom['op']}:{dom['layer']}:B{dom['B']}", args.workload)
    target = {f"{o['op']} B={o['B']}": o["frac"] for o in ops
              if o["layer"] == "large95" and o["B"] >= 8 and o["op"] != "adam_step"}
    roofline = {"bound": "hbm", "achieved": dom["gbs"], "peak": peak, "unit": "GB/s",
                "frac": dom["frac"], "traffic": tr,
                "kernel": f"{dom['op']} {dom['shape']} nnz={dom['nnz']} B={dom['B']}",
                "peak_kind": f"{peak_kind} HBM copy bandwidth (burst)",
                "bytes": "metric bytes nnz*12 + dense operands, per launch",
                # the rate at which the op gathers operand rows (4 * B bytes per
                # stored entry, through L1 from L2): from batch ~8 on, this and
                # not DRAM is what the kernels' time follows
                "gather_gbs": dom["gather_gbs"],
                "at_95pct_batch_ge_8": target}

    # End to end through the same calls with host buffers: each step's inputs
    # (X, dY of every layer and batch) travel in one pinned buffer with one
    # H2D copy, and its results (Y, dX, dW) come back in one D2H copy; every
    # array sits at a 16-byte aligned offset of its buffer.
    pairs = [(c, B, d) for c in cases for B, d in c["dev"].items()]

    def layout(sizes):
        offs, n = [], 0
        for sz in sizes:
            offs.append(n)
            n += (sz + 3) & ~3
        return offs, n

    in_arrays = [(c["acts"][B][0], c["acts"][B][1]) for c, B, _ in pairs]
    out_shapes = [(d["Y"].shape, d["dX"].shape, d["dW"].shape) for _, _, d in pairs]
    in_off, n_in = layout([a.size for xs in in_arrays for a in xs])
    out_off, n_out = layout([int(np.prod(sh)) for shs in out_shapes for sh in shs])
    h_in = torch.empty(n_in, dtype=torch.float32).pin_memory()
    h_out = torch.empty(n_out, dtype=torch.float32).pin_memory()
    d_in = torch.empty(n_in, dtype=torch.float32, device=dev)
    d_out = torch.empty(n_out, dtype=torch.float32, device=dev)
    views = []
    for i, ((c, B, d), (X, dY), shs) in enumerate(zip(pairs, in_arrays, out_shapes)):
        h_in[in_off[2 * i]:in_off[2 * i] + X.size] = torch.from_numpy(X).reshape(-1)
        h_in[in_off[2 * i + 1]:in_off[2 * i + 1] + dY.size] = torch.from_numpy(dY).reshape(-1)

        def dview(buf, off, shape):
            n = int(np.prod(shape))
            return buf[off:off + n].view(*shape)
        views.append(dict(h=c["h"], X=dview(d_in, in_off[2 * i], X.shape),
                          dY=dview(d_in, in_off[2 * i + 1], dY.shape),
                          Y=dview(d_out, out_off[3 * i], shs[0]),
                          dX=dview(d_out, out_off[3 * i + 1], shs[1]),
                          dW=dview(d_out, out_off[3 * i + 2], shs[2])))
    h2d, d2h = n_in * 4, n_out * 4
    # Per (layer, batch) pair: its inputs and its outputs are contiguous
    # ranges of the two buffers.
    in_rng = [(in_off[2 * i], in_off[2 * i + 1] + X.size) for i, (X, dY) in
              enumerate(in_arrays)]
    out_rng = [(out_off[3 * i], out_off[3 * i + 2] + int(np.prod(shs[2]))) for i, shs in
               enumerate(out_shapes)]
    copy_in = torch.cuda.Stream(device=dev)
    copy_out = torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in pairs]
    ev_done = [torch.cuda.Event() for _ in pairs]

    def e2e_step():
        """One step with host buffers: every pair's inputs go up on one copy
        stream, its products run on `stream` once they have landed, and its
        results come back on a second copy stream while the next pair
        computes.  The step ends when the last result is on the host."""
        copy_in.wait_stream(stream)  # the previous step is done with d_in
        with torch.cuda.stream(copy_in):
            for (lo, hi), ev in zip(in_rng, ev_in):
                d_in[lo:hi].copy_(h_in[lo:hi], non_blocking=True)
                ev.record(copy_in)
        for v, (lo, hi), ei, ed in zip(views, out_rng, ev_in, ev_done):
            stream.wait_event(ei)
            sn.snack_forward(v["h"], v["X"], v["Y"], stream=stream)
            sn.snack_backward(v["h"], v["X"], v["dY"], v["dX"], v["dW"], stream=stream)
            ed.record(stream)
            copy_out.wait_event(ed)
            with torch.cuda.stream(copy_out):
                h_out[lo:hi].copy_(d_out[lo:hi], non_blocking=True)
        stream.wait_stream(copy_out)

    def time_e2e(run):
        """Milliseconds of args.steps e2e steps (max over ranks), each after
        an L2 flush, between events on `stream`; also this rank's per-step
        times (the host link is shared, so single steps can stall)."""
        evs = []
        barrier()
        with torch.cuda.stream(stream):
            for _ in range(args.steps):
                flush_l2(flush)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                run()
                e1.record(stream)
                evs.append((e0, e1))
        torch.cuda.synchronize()
        barrier()
        per = [a.elapsed_time(b) for a, b in evs]
        return reduce_max(sum(per), dev), per

    with torch.cuda.stream(stream):
        for _ in range(3):
            e2e_step()
    torch.cuda.synchronize()
    eager_ms, _ = time_e2e(e2e_step)
    # The same pipeline (its copies, events and library calls) captured once
    # and replayed from a CUDA graph, as the device-resident step is: every
    # replay moves the step's inputs and results between pinned host memory
    # and the device, without the host re-issuing ~100 calls per step.
    e2e_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(e2e_graph, stream=stream):
        e2e_step()
    with torch.cuda.stream(stream):
        for _ in range(3):
            e2e_graph.replay()
    torch.cuda.synchronize()
    h_out.zero_()  # what the check below reads must come from the timed replays
    e2e_ms, e2e_per = time_e2e(e2e_graph.replay)
    del e2e_graph
    # The host buffer holds the last step's results: one pair's Y must equal
    # a forward of the same (device-resident) X with the current values (the
    # per-op table's Adam steps have changed them since the timed step).
    c0, B0, d0 = pairs[0]
    want = torch.empty_like(d0["Y"])
    sn.snack_forward(c0["h"], d0["X"], want, stream=stream)
    torch.cuda.synchronize()
    got = h_out[out_off[0]:out_off[0] + want.numel()].view_as(want)
    if not torch.equal(got, want.cpu()):
        raise RuntimeError("e2e: the copied-back Y differs from a device-resident forward")
    barrier()
    e2e_value = world * fl * args.steps / (e2e_ms / 1e3) / 1e9
    eager_value = world * fl * args.steps / (eager_ms / 1e3) / 1e9

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(cases, budget_s=args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded uniform-random COO patterns, N(0,1) activations)",
            "config": {"workload": describe(wl, cases), "layers": [
                dict(name=c["layer"].name, out=c["layer"].out, inp=c["layer"].inp,
                     sparsity=c["layer"].sparsity, nnz=c["layer"].nnz) for c in cases],
                "batches": sorted({B for c in cases for B in c["acts"]}),
                "ops_per_step": "fwd + fused bwd (dX, dW) per layer per batch",
                "launch": "CUDA graph replay of the step",
                "l2": "flushed between timed steps (256 MiB write, then read back); "
                      "flush not timed",
                "parallelism": f"{world} independent replica(s)"},
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "eager_value": round(eager_value, 2),
                    "ms_per_step_min_median_max": [round(x, 4) for x in (
                        min(e2e_per), sorted(e2e_per)[len(e2e_per) // 2], max(e2e_per))],
                    "how": "per step and per layer/batch: pinned H2D copy of its X and dY "
                           "(one copy stream), snack_forward + snack_backward via the C ABI "
                           "once they have landed, D2H copy of its Y, dX, dW on a second copy "
                           "stream while the next layer/batch computes; the step ends when the "
                           "last result is on the host.  value: that pipeline captured once "
                           "and replayed from a CUDA graph each step (copies included); "
                           "eager_value: the same calls issued from Python each step"},
            "gpu_launches": int(launches_per_step * args.steps),
            "launches_per_step": int(launches_per_step),
            "clocks": clk,
            "wall_s_timed_region": round(wall, 4),
            "ops": ops,
            "train_step": train,
            "extra_ops": extra,
        }
        print(json.dumps(line), flush=True)


def describe(wl, cases):
    parts = [f"{c['layer'].out}x{c['layer'].inp}@{c['layer'].sparsity:g}% (nnz {c['layer'].nnz})"
             for c in cases]
    bs = sorted({B for c in cases for B in c["acts"]})
    if len(parts) > 4:
        parts = parts[:2] + [f"... {len(parts)} layers"]
    return f"{wl.name}: " + ", ".join(parts) + f"; batch {bs}; fwd+bwd"


# ------------------------------------------------------------------ oracle

SAMPLE_ENTRIES = 600_000  # stored entries per layer the oracle sample keeps at most


def prepare_oracle(cases, max_entries: int = SAMPLE_ENTRIES):
    """A bounded sample of every layer for the oracle: a stride of its rows
    (forward and dW: the sampled rows' entries, a layer of those rows) and
    the same stride of its columns (backward-input: the sampled columns'
    entries), each canonicalised once.  The stride keeps at most
    max_entries entries per layer; the flops are counted on the sample."""
    import numpy as np
    import oracle
    oracle.build()
    prepared = []
    for c in cases:
        L = c["layer"]
        ref = oracle.canonicalize(L.out, L.inp, c["row"], c["col"], c["val"])
        stride = max(1, -(-L.nnz // max_entries))
        rows = np.arange(0, L.out, stride)
        cols = np.arange(0, L.inp, stride)
        rmap = np.full(L.out, -1, np.int64)
        rmap[rows] = np.arange(rows.size)
        cmap = np.full(L.inp, -1, np.int64)
        cmap[cols] = np.arange(cols.size)
        rk = rmap[ref["row"]] >= 0
        ck = cmap[ref["col"]] >= 0
        rsub = oracle.canonicalize(rows.size, L.inp, rmap[ref["row"][rk]], ref["col"][rk],
                                   ref["val"][rk])
        csub = oracle.canonicalize(L.out, cols.size, ref["row"][ck], cmap[ref["col"][ck]],
                                   ref["val"][ck])
        acts = {B: (X, dY, np.ascontiguousarray(dY[:, rows]))
                for B, (X, dY) in c["acts"].items()}
        prepared.append(dict(out=L.out, inp=L.inp, nr=rows.size, nc=cols.size, rsub=rsub,
                             csub=csub, acts=acts, stride=stride))
    return prepared


def oracle_sample_flops(prepared) -> float:
    return float(sum(2 * B * (2 * p["rsub"]["row"].size + p["csub"]["row"].size)
                     for p in prepared for B in p["acts"]))


def oracle_step(prepared, omp_threads: int = 0):
    """One pass of the oracle over the sample: forward and dW on the sampled
    rows, backward-input on the sampled columns, every batch.  omp_threads > 0
    runs the all-cores copy of the same loops (bit-identical results)."""
    import oracle
    for p in prepared:
        r, cs = p["rsub"], p["csub"]
        for B, (X, dY, dYr) in p["acts"].items():
            if omp_threads:
                oracle.forward_omp(p["nr"], p["inp"], r, X, omp_threads)
                oracle.backward_input_omp(p["out"], p["nc"], cs, dY, omp_threads)
                oracle.backward_weight_omp(p["nr"], p["inp"], r, X, dYr, omp_threads)
            else:
                oracle.forward(p["nr"], p["inp"], r["row"], r["col"], r["val"], X)
                oracle.backward_input(p["out"], p["nc"], cs["row"], cs["col"], cs["val"], dY)
                oracle.backward_weight(p["nr"], p["inp"], r["row"], r["col"], X, dYr)


def _sample_text(prepared):
    ents = sum(p["rsub"]["row"].size + p["csub"]["row"].size for p in prepared)
    strides = sorted({p["stride"] for p in prepared})
    return (f"every {'/'.join(map(str, strides))}-th row (fwd, dW) and column (dX) of each "
            f"layer, all batches: {ents} sampled entries")


def _timed_passes(prepared, budget_s, omp_threads=0):
    t0 = time.perf_counter()
    n = 0
    while True:
        oracle_step(prepared, omp_threads)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or el / n * (n + 1) > 3 * budget_s:
            return n, el


def cpu_baseline(cases, budget_s: float = 10.0):
    """The oracle as it stands (single-threaded C, fp64 accumulation) on a
    bounded sample of the workload, ~budget_s of CPU work; then its all-cores
    copy (same loops split over the host's cores, bit-identical results) on
    the same sample."""
    import oracle
    prepared = prepare_oracle(cases)
    fl = oracle_sample_flops(prepared)
    n, el = _timed_passes(prepared, budget_s)
    res = {"value": round(fl * n / el / 1e9, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
           "sample": f"{_sample_text(prepared)}; {n} pass(es), {el:.1f} s, single thread"}
    try:
        cores = oracle.host_cores()
        oracle_step(prepared, cores)  # warm the threads
        n2, el2 = _timed_passes(prepared, budget_s / 2, cores)
        res["all_cores"] = {"value": round(fl * n2 / el2 / 1e9, 4), "unit": UNIT,
                            "cores": cores, "kind": "oracle loops on all cores (OpenMP)",
                            "sample": f"same sample; {n2} pass(es), {el2:.1f} s"}
    except Exception as e:  # no OpenMP build on this host
        res["all_cores"] = {"unavailable": str(e)[:200]}
    return res


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    wl, cases = make_cases(args.workload, args.batches, args.seed)
    prepared = prepare_oracle(cases)
    fl = oracle_sample_flops(prepared)
    for _ in range(args.warmup):
        oracle_step(prepared)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(prepared)
    el = time.perf_counter() - t0
    value = fl * args.steps / el / 1e9
    line = {"metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64 accumulate, f32 in/out",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": describe(wl, cases)},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"{_sample_text(prepared)}; one pass per step"},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_decoder_train(args):
    """The GPT-2-small-shaped decoder (all 48 attention / MLP projections
    SNACK layers at 99 %) trained on random tokens: plain SGD at lr 1e-2,
    30 % prune / regrow of every sparse layer every 100 steps.  One step =
    forward, backward and optimizer step of the whole model on 1 x 256
    tokens, run eagerly as a user's training loop would.  value = effective
    GFLOP/s of the sparse products (3 x 2 x nnz x 256 per layer per step)
    over the measured step time; tokens/s, the prune/regrow time (amortised
    over its 100-step period) and the sparse layers' share of the step are
    reported beside it."""
    import numpy as np
    import torch
    from coo_spmm_sparse_gb300.decoder import DecoderConfig, SparseDecoder, Trainer
    import coo_spmm_sparse_gb300 as sn

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    rank, world = dist_init("nccl")
    dev = torch.device("cuda", local)
    cfg = DecoderConfig(seed=args.seed)
    model = SparseDecoder(cfg, device=dev)
    tr = Trainer(model, lr=1e-2, prune_frac=0.30, prune_every=0)  # regrow timed apart
    lins = model.sparse_layers()
    g = torch.Generator(device="cpu").manual_seed(args.seed + 1)
    nbatch = 8
    host_tok = torch.randint(0, cfg.vocab, (nbatch, 1, cfg.ctx), generator=g).pin_memory()
    dev_tok = host_tok.to(dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    for i in range(max(args.warmup, 3)):
        tr.step(dev_tok[i % nbatch])
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    barrier()
    torch.cuda.synchronize()
    evs = []
    n0 = sn.snack_launch_count()
    for i in range(args.steps):
        flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        tr.step(dev_tok[i % nbatch])
        e1.record()
        evs.append((e0, e1))
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    launches = sn.snack_launch_count() - n0
    step_ms = reduce_max(sum(a.elapsed_time(b) for a, b in evs), dev) / args.steps

    # end to end: the token batch copied from pinned host memory and the loss
    # read back on the host every step
    evs2 = []
    for i in range(args.steps):
        flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        tok = host_tok[i % nbatch].to(dev, non_blocking=True)
        loss = tr.step(tok).item()
        e1.record()
        evs2.append((e0, e1))
    torch.cuda.synchronize()
    e2e_ms = reduce_max(sum(a.elapsed_time(b) for a, b in evs2), dev) / args.steps

    # one prune / regrow of all 48 layers (host-synchronising, every 100 steps)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    model.prune_regrow(0.30, 100)
    torch.cuda.synchronize()
    regrow_ms = (time.perf_counter() - t0) * 1e3

    # the sparse layers alone: forward + both backward products of each
    # layer on activations of the step's shapes, replayed from one graph
    s = torch.cuda.Stream(device=dev)
    bufs = []
    for l in lins:
        X = torch.randn(cfg.ctx, l.in_features, device=dev)
        dY = torch.randn(cfg.ctx, l.out_features, device=dev)
        bufs.append((l, X, dY, torch.empty(cfg.ctx, l.out_features, device=dev),
                     torch.empty(cfg.ctx, l.in_features, device=dev), torch.empty(l.nnz, device=dev)))

    def sparse_ops():
        for l, X, dY, Y, dX, dW in bufs:
            sn.snack_forward(l.handle, X, Y, stream=s)
            sn.snack_backward(l.handle, X, dY, dX, dW, stream=s)
    sparse_us, _ = time_graph(sparse_ops, s, flush, reps=20, warm=3)

    nnz = sum(l.nnz for l in lins)
    fl = 3 * 2 * nnz * cfg.ctx
    value = world * fl / (step_ms / 1e3) / 1e9
    mbytes = sum(3 * (l.nnz * 12 + 4 * cfg.ctx * (l.in_features + l.out_features)) for l in lins)
    peak, peak_kind = read_peak()
    achieved = mbytes / sparse_us / 1e3
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cases = []
        for l in lins:
            row, col, val = l.export()
            X = np.random.default_rng(0).standard_normal((cfg.ctx, l.in_features)).astype(np.float32)
            dY = np.random.default_rng(1).standard_normal((cfg.ctx, l.out_features)).astype(np.float32)
            lay = type("L", (), dict(name="", out=l.out_features, inp=l.in_features, nnz=l.nnz))
            cases.append(dict(layer=lay, row=row, col=col, val=val, acts={cfg.ctx: (X, dY)}))
        cpu = cpu_baseline(cases, budget_s=args.cpu_seconds)
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": round(step_ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (random tokens uniform in [0, 50257), random init)",
            "config": {"workload": "gpt2_decoder_train: 12 blocks, d 768, 12 heads, MLP 3072, "
                                   "ctx 256, vocab 50257 (tied head); 48 projections SNACK at "
                                   f"99 % ({nnz} stored entries); batch 1 x 256 tokens; SGD "
                                   "lr 1e-2; 30 % prune / regrow every 100 steps",
                       "ops_per_step": "model forward + backward + SGD step (eager)",
                       "l2": "flushed between timed steps", "parallelism": f"{world} replica(s)"},
            "tokens_per_s": round(world * cfg.ctx / (step_ms / 1e3), 1),
            "prune_regrow_ms": round(regrow_ms, 2),
            "ms_per_step_with_regrow_amortised": round(step_ms + regrow_ms / 100, 4),
            "sparse_layers_us": round(sparse_us, 2),
            "sparse_share_of_step": round(sparse_us / 1e3 / step_ms, 4),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": None,
                         "kernel": "all 48 sparse layers' forward + backward, back to back",
                         "peak_kind": f"{peak_kind} HBM copy bandwidth (burst)"},
            "cpu_baseline": cpu,
            "e2e": {"value": round(world * fl / (e2e_ms / 1e3) / 1e9, 2), "unit": UNIT,
                    "h2d_bytes_per_step": int(host_tok[0].numel() * 8), "d2h_bytes_per_step": 4,
                    "how": "token batch copied from pinned host memory and the loss read on the "
                           "host every step"},
            "last_loss": round(loss, 4),
            "gpu_launches": int(launches), "clocks": clk,
        }
        print(json.dumps(line), flush=True)


def run_only_op(args):
    """One op, a few launches, for an ncu capture of a single kernel."""
    import torch
    import coo_spmm_sparse_gb300 as sn
    wl, cases = make_cases(args.workload, args.batches, args.seed)
    c = cases[0]
    if args.layer:
        c = next(x for x in cases if x["layer"].name == args.layer)
    L = c["layer"]
    B = sorted(c["acts"])[0]
    X, dY = (torch.from_numpy(a).cuda() for a in c["acts"][B])
    h = sn.snack_create(L.out, L.inp, c["row"], c["col"], c["val"])
    Y = torch.empty(B, L.out, device="cuda")
    dX = torch.empty(B, L.inp, device="cuda")
    dW = torch.empty(L.nnz, device="cuda")
    flush = torch.empty(FLUSH_BYTES // 4, device="cuda")
    for _ in range(args.reps):
        flush_l2(flush)
        if args.only_op == "fwd":
            sn.snack_forward(h, X, Y)
        elif args.only_op == "bwd_input":
            sn.snack_backward_input(h, dY, dX)
        elif args.only_op == "bwd_weight":
            sn.snack_backward_weight(h, X, dY, dW)
        else:
            sn.snack_backward(h, X, dY, dX, dW)
    torch.cuda.synchronize()
    print(f"only-op {args.only_op} {L.name} {L.out}x{L.inp} nnz={L.nnz} B={B} reps={args.reps}")


def run_memory_sweep(args):
    """Memory headroom (SNACK §4.4, Figure 4): device bytes of one sparse layer
    against the dense W it replaces, at hidden size 10000 and input sizes
    5000-25000, sparsity 90 / 95 / 99 %.  Prints one JSON object.

    Per configuration: the handle's own accounting (snack_device_bytes:
    indices, values, CSR/CSC layouts, segment tables, workspace), the device
    memory the creation actually took (cudaMemGetInfo before / after, so
    allocation granularity included), and the training-time total with the
    nnz-long dW.  Dense references: W (4 B per cell), W + dW, and
    Dense+Mask = W + dW + a 1-byte mask per cell."""
    import torch
    import coo_spmm_sparse_gb300 as sn
    import workloads
    torch.cuda.init()
    hidden = 10000
    rows = []
    for inp in range(5000, 25001, 2500):
        for sp in (90, 95, 99):
            nnz = workloads.nnz_for(hidden, inp, sp)
            torch.cuda.synchronize()
            free0, _ = torch.cuda.mem_get_info()
            h, _ = sn.snack_create_random(hidden, inp, nnz, args.seed)
            torch.cuda.synchronize()
            free1, _ = torch.cuda.mem_get_info()
            acct = sn.snack_device_bytes(h)
            cells = hidden * inp
            rows.append(dict(inp=inp, hidden=hidden, sparsity=sp, nnz=nnz,
                             snack_bytes=acct, snack_measured=free0 - free1,
                             snack_train=acct + 4 * nnz,
                             dense_w=4 * cells, dense_train=8 * cells,
                             dense_mask_train=9 * cells))
            del h
    print(json.dumps({"metric": "device bytes of one layer vs dense", "hidden": hidden,
                      "unit": "bytes", "rows": rows}))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="large",
                    help="large (default: 10000x10000 at 90/95/99 %%), large90/95/99, gpt2_mlp, "
                         "toy256, skewed, gpt2_decoder (its sparse layers' products), "
                         "gpt2_decoder_train (the whole decoder trained)")
    ap.add_argument("--batches", type=lambda s: [int(x) for x in s.split(",")], default=None)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--extra-ops", default="gpt2_mlp,skewed",
                    help="workloads whose ops are timed too (per-op table only)")
    ap.add_argument("--no-extra-ops", action="store_true",
                    help="skip the extra workloads and the training-step timing")
    ap.add_argument("--only-op", choices=["fwd", "bwd_input", "bwd_weight", "bwd"], default=None,
                    help="profiling mode: run one op --reps times on one layer (--layer) and "
                         "the first batch of the workload (cold L2 before each), print no JSON")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--layer", default=None,
                    help="profiling mode: the workload's layer to run (default: its first)")
    ap.add_argument("--memory-sweep", action="store_true",
                    help="print the layer's device bytes against dense W at hidden 10000, "
                         "input 5000-25000, sparsity 90/95/99 %% (one JSON object)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.only_op:
        run_only_op(args)
        return
    if args.memory_sweep:
        run_memory_sweep(args)
        return
    if args.impl == "reference":
        if args.workload == "gpt2_decoder_train":  # the oracle on the decoder's sparse layers
            args.workload = "gpt2_decoder"
            args.batches = [256]
        run_reference(args)
    elif args.workload == "gpt2_decoder_train":
        run_decoder_train(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
