#!/usr/bin/env python3
"""Benchmark of the causal dot product (forward + backward) on GB300.

One step = causal_product_fwd_ckpt + causal_product_bwd_ckpt (the forward
leaves checkpoints of its state for the backward's dq scans, as the autograd
wrapper does) over one batch of the
bf16 workload B=8, H=16, N=4096, D=M=64 (inputs resident in HBM when the
timed region starts; every input is larger than the 129 MB L2, so no flush
is needed between iterations).  Prints ONE JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs the same per-GPU workload (weak scaling, no
collective on the data path); the timed region is bracketed by a barrier
and the maximum over ranks is reported.

--impl reference times the fp64 CPU oracle (the plain recurrence) on the
host cores, on a bounded sample of the same workload, in the same metric.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = "bf16_b8h16_n4096_d64"
METRIC = "causal-product fwd+bwd Mtokens/s·head"
UNIT = "Mtok·head/s"

# DRAM traffic of one launch of the tensor-core kernel measured by ncu
# (dram__bytes_read.sum + dram__bytes_write.sum) together with the SHA-256 of
# the kernel source it was measured on; a changed source reports null.
CAUSAL_SOURCES = ("cp_tc.cu", "cp_tc_causal.cuh", "cp_tc_common.cuh", "sm103_ptx.cuh")
BWD_SOURCES = ("cp_tc_dkdv.cu", "cp_tc_dkdv.cuh", "cp_tc_causal.cuh", "cp_tc_common.cuh",
               "sm103_ptx.cuh")
# Each figure is one launch of its kernel (the fourth of the run, after the
# three warm-up steps), from
# `ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum
# --clock-control none -k regex:<kernel> -s 3 -c 1` of `bench.py --steps 2
# --warmup 3 --no-e2e --no-extras --no-others --no-cpu-baseline`, one capture
# per kernel (the outputs a launch writes partly stay in the 126 MB L2 when
# it ends, so its write bytes undercount them).
PROFILED_TRAFFIC = {
    "source_sha256": "c55654417449854cafe01a3592c067a6cdc92527f23a3aed6e8214924ee78505",
    "bytes_per_launch": 211120896,  # 201.43 MB read + 9.69 MB written (forward launch)
}
PROFILED_TRAFFIC_BWD = {
    "source_sha256": "3d5f0084ac9e327b22b66036cc1d6f2f0bdbf42cd435297a677a8a2d36f1719d",
    "bytes_per_launch": 605626624,  # 463.83 MB read + 141.80 MB written (one backward launch)
}


def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def dist_setup():
    world = _env_int("WORLD_SIZE", 1)
    rank = _env_int("RANK", 0)
    local = _env_int("LOCAL_RANK", 0)
    if world > 1:
        import torch
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" \
        else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi sampling (every 5 ms) of SM clocks and throttle reasons.

    Each output line is stamped with the host time it arrives; summary()
    keeps the samples inside [t0, t1] (the timed region) and falls back to
    the surrounding loaded window when the region is shorter than a few
    sampling periods."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def _reader(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line))

    def __enter__(self):
        import threading
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "5"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._reader, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread is not None:
                self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float, loaded_from: float):
        def parse(window):
            rows = []
            for ts, line in self.lines:
                if not (window[0] <= ts <= window[1]):
                    continue
                r = [x.strip() for x in next(csv.reader(io.StringIO(line)), [])]
                if len(r) >= 9:
                    rows.append(r)
            return rows
        rows, window = parse((t0, t1 + 0.005)), "timed region"
        if len(rows) < 3:
            rows, window = parse((loaded_from, t1 + 0.005)), "timed region + loaded soak before it"
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        num = lambda x: x.replace(".", "", 1).isdigit()
        sm = [float(r[1]) for r in rows if num(r[1])]
        smax = [float(r[2]) for r in rows if num(r[2])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows), "window": window}


def kernel_sha(files=CAUSAL_SOURCES):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "prefix_sum_outer_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def back_to_back(fn, n, stream):
    """Total milliseconds of ``n`` calls of ``fn`` issued back to back on
    ``stream``, CUDA events at the two ends of the run only."""
    import torch

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(n):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def algorithmic_bytes(w):
    """Bytes the method must move per step: forward reads q, k, v and writes
    out; backward reads q, k, v, g and writes dq, dk, dv."""
    s = 2 if w.dtype == "bf16" else 4
    per_th = s * (2 * w.D + 2 * w.M) + s * (4 * w.D + 3 * w.M)
    return per_th * w.token_heads


def cpu_baseline(w, budget_s=10.0):
    """The oracle as it stands, all host cores, on a bounded sample of the
    workload: the first `n` (b,h) slices, forward + backward."""
    import oracle
    from prefix_sum_outer_gb300.workloads import make_inputs
    f = lambda t: t.float().numpy()
    # calibrate on one slice, then size the sample for ~budget_s
    q, k, v, g = make_inputs(1, 1, w.N, w.D, w.M, w.torch_dtype, seed=w.seed, feature=w.feature,
                             x_std=w.x_std)
    t0 = time.perf_counter()
    oracle.fwd(f(q), f(k), f(v))
    oracle.bwd(f(q), f(k), f(v), f(g))
    one = time.perf_counter() - t0
    cores = oracle.threads(0)
    n = int(max(1, min(w.B * w.H, round(budget_s * cores / max(one, 1e-6)))))
    q, k, v, g = make_inputs(1, n, w.N, w.D, w.M, w.torch_dtype, seed=w.seed, feature=w.feature,
                             x_std=w.x_std)
    qn, kn, vn, gn = f(q), f(k), f(v), f(g)
    # when the whole workload is shorter than the budget, repeat it (at most
    # 20 passes) so the figure rests on seconds of CPU work, not one short pass
    reps, dt = 0, 0.0
    while True:
        t0 = time.perf_counter()
        oracle.fwd(qn, kn, vn)
        oracle.bwd(qn, kn, vn, gn)
        dt += time.perf_counter() - t0
        reps += 1
        if dt >= 0.5 * budget_s or reps >= 20:
            break
    return {"value": reps * n * w.N / dt / 1e6, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n} of {w.B * w.H} (b,h) slices x N={w.N}, fwd+bwd, fp64 C oracle, "
                      f"{reps} pass(es), {dt:.1f} s"}


def run_reference(args, world, rank):
    from prefix_sum_outer_gb300.workloads import WORKLOADS
    if rank != 0:
        return 0
    import oracle
    w = WORKLOADS[args.workload]
    from prefix_sum_outer_gb300.workloads import make_inputs
    f = lambda t: t.float().numpy()
    cores = oracle.threads(0)
    # size one step at ~3 s of oracle work
    q, k, v, g = make_inputs(1, 1, w.N, w.D, w.M, w.torch_dtype, seed=w.seed, feature=w.feature,
                             x_std=w.x_std)
    t0 = time.perf_counter()
    oracle.fwd(f(q), f(k), f(v))
    oracle.bwd(f(q), f(k), f(v), f(g))
    one = time.perf_counter() - t0
    n = int(max(1, min(w.B * w.H, round(3.0 * cores / max(one, 1e-6)))))
    q, k, v, g = make_inputs(1, n, w.N, w.D, w.M, w.torch_dtype, seed=w.seed, feature=w.feature,
                             x_std=w.x_std)
    qn, kn, vn, gn = f(q), f(k), f(v), f(g)
    for _ in range(args.warmup):
        oracle.fwd(qn, kn, vn)
        oracle.bwd(qn, kn, vn, gn)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.fwd(qn, kn, vn)
        oracle.bwd(qn, kn, vn, gn)
    dt = (time.perf_counter() - t0) / max(args.steps, 1)
    value = n * w.N / dt / 1e6
    sample = f"{n} of {w.B * w.H} (b,h) slices x N={w.N} per step, fwd+bwd, fp64 C oracle"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N,
                                        "D": w.D, "M": w.M, "input_dtype": w.dtype},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, world, rank, local):
    import torch

    import prefix_sum_outer_gb300 as cp
    from prefix_sum_outer_gb300.workloads import WORKLOADS, make_inputs

    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device (the product has no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = WORKLOADS[args.workload]
    q, k, v, g = make_inputs(w.B, w.H, w.N, w.D, w.M, w.torch_dtype, seed=w.seed + 1000 * rank,
                             feature=w.feature, x_std=w.x_std, backward=True)
    qd, kd, vd, gd = (t.to(dev) for t in (q, k, v, g))
    out = torch.empty_like(vd)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    ws_f = torch.zeros(cp.causal_product_workspace_size(w.B, w.H, w.N, w.D, w.M, w.torch_dtype,
                                                        False), dtype=torch.uint8, device=dev)
    ws_b = torch.zeros(cp.causal_product_workspace_size(w.B, w.H, w.N, w.D, w.M, w.torch_dtype,
                                                        True), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    # the forward leaves checkpoints of its state for the backward's dq scans
    ckpt = torch.empty(max(cp.causal_product_checkpoint_size(w.B, w.H, w.N, w.D, w.M,
                                                             w.torch_dtype) // 4, 1),
                       dtype=torch.float32, device=dev)

    def fwd_call():
        cp.causal_product_fwd_ckpt(qd, kd, vd, out=out, ckpt=ckpt, workspace=ws_f, stream=stream)

    def bwd_call():
        cp.causal_product_bwd_ckpt(qd, kd, vd, gd, ckpt, dq, dk, dv, workspace=ws_b,
                                   stream=stream)

    def step():
        fwd_call()
        bwd_call()

    # kernels of ours launched per step: the library's own count for the
    # forward and the backward call of this shape
    launches_per_step = _launches_per_step(w)

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize()
    if cp.causal_product_status(ws_f) != cp.CP_OK or cp.causal_product_status(ws_b) != cp.CP_OK:
        raise RuntimeError("kernel status word reports an error after warm-up")

    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        # keep the GPU loaded for ~0.3 s so the sampler runs and clocks settle
        soak_from = time.time()
        while time.time() - soak_from < 0.3:
            step()
            torch.cuda.synchronize()
        torch.cuda.synchronize()
        t_start = time.time()
        # the K timed steps: fwd and bwd back to back, as a caller runs them
        # (nothing between the launches), events on the stream at both ends
        t0_ev, t1_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0_ev.record(stream)
        for _ in range(args.steps):
            step()
        t1_ev.record(stream)
        torch.cuda.synchronize()
        t_end = time.time()
        # then the per-launch figures for the roofline objects: K forward
        # calls back to back, then K backward calls back to back, events at
        # both ends of each run (an event between two launches would cut the
        # overlap of one launch's tail with the next one's start)
        fwd_ms = back_to_back(fwd_call, args.steps, stream)
        bwd_ms = back_to_back(bwd_call, args.steps, stream)
        # the same calls one at a time, each between its own events, for
        # comparison: a launch's start-up and drain are then not hidden
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
               torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for e0, e1, e2 in ev:
            e0.record(stream)
            fwd_call()
            e1.record(stream)
            bwd_call()
            e2.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    total_ms = t0_ev.elapsed_time(t1_ev)
    fwd_iso_ms = sum(a.elapsed_time(b) for a, b, _ in ev)
    bwd_iso_ms = sum(b.elapsed_time(c) for _, b, c in ev)
    total_ms = max_over_ranks(total_ms, world)
    fwd_ms, bwd_ms = max_over_ranks(fwd_ms, world), max_over_ranks(bwd_ms, world)
    ms_per_step = total_ms / args.steps
    value = w.token_heads * world * args.steps / (total_ms / 1e3) / 1e6

    # ---- end to end: pinned host buffers in, results back to the host.  The
    # step is cut into chunks of (b,h) slices, with copies and compute on
    # separate streams, so that the host-to-device copy of one chunk, the
    # fwd + bwd of the previous one and the device-to-host copy of the one
    # before overlap (and so do consecutive steps).
    e2e = None
    if not args.no_e2e:
        BH = w.B * w.H
        n_chunks = max(1, min(args.e2e_chunks, BH))
        while BH % n_chunks:
            n_chunks -= 1
        cb = BH // n_chunks
        hq, hk, hv, hg = (t.reshape(BH, w.N, -1).pin_memory() for t in (q, k, v, g))
        ho, hdq, hdk, hdv = (torch.empty((BH, w.N, t.shape[-1]), dtype=t.dtype).pin_memory()
                             for t in (out, dq, dk, dv))
        dev_in = [t.view(BH, w.N, -1) for t in (qd, kd, vd, gd)]
        dev_out = [t.view(BH, w.N, -1) for t in (out, dq, dk, dv)]
        host_in, host_out = (hq, hk, hv, hg), (ho, hdq, hdk, hdv)
        # one copy stream per tensor and direction, so that copies use
        # several copy engines at once
        s_ins = [torch.cuda.Stream(dev) for _ in range(4)]
        s_outs = [torch.cuda.Stream(dev) for _ in range(4)]
        s_cmp = torch.cuda.Stream(dev)
        ws_fc = torch.zeros(cp.causal_product_workspace_size(1, cb, w.N, w.D, w.M, w.torch_dtype,
                                                             False), dtype=torch.uint8, device=dev)
        ws_bc = torch.zeros(cp.causal_product_workspace_size(1, cb, w.N, w.D, w.M, w.torch_dtype,
                                                             True), dtype=torch.uint8, device=dev)
        # one checkpoint buffer per chunk would let chunks overlap; the
        # compute of the chunks runs on one stream, so they share one
        ckpt_c = torch.empty(max(cp.causal_product_checkpoint_size(1, cb, w.N, w.D, w.M,
                                                                   w.torch_dtype) // 4, 1),
                             dtype=torch.float32, device=dev)

        # cross-step hazards: a chunk's inputs are overwritten only after the
        # previous step's compute of that chunk, and its outputs only after
        # the previous step's copy back
        prev_cmp = [None] * n_chunks
        prev_out = [None] * n_chunks

        def e2e_step():
            done_in = []
            for c in range(n_chunks):
                sl = slice(c * cb, (c + 1) * cb)
                evs = []
                for s_i, d_t, h_t in zip(s_ins, dev_in, host_in):
                    if prev_cmp[c] is not None:
                        s_i.wait_event(prev_cmp[c])
                    with torch.cuda.stream(s_i):
                        d_t[sl].copy_(h_t[sl], non_blocking=True)
                    e = torch.cuda.Event()
                    e.record(s_i)
                    evs.append(e)
                done_in.append(evs)
            for c in range(n_chunks):
                sl = slice(c * cb, (c + 1) * cb)
                for e in done_in[c]:
                    s_cmp.wait_event(e)
                for e in prev_out[c] or ():
                    s_cmp.wait_event(e)
                cq, ck, cv, cg = (t[sl].view(1, cb, w.N, -1) for t in dev_in)
                co, cdq, cdk, cdv = (t[sl].view(1, cb, w.N, -1) for t in dev_out)
                cp.causal_product_fwd_ckpt(cq, ck, cv, out=co, ckpt=ckpt_c, workspace=ws_fc,
                                           stream=s_cmp)
                cp.causal_product_bwd_ckpt(cq, ck, cv, cg, ckpt_c, cdq, cdk, cdv, workspace=ws_bc,
                                           stream=s_cmp)
                e = torch.cuda.Event()
                e.record(s_cmp)
                prev_cmp[c] = e
            for c in range(n_chunks):
                sl = slice(c * cb, (c + 1) * cb)
                evs = []
                for s_o, d_t, h_t in zip(s_outs, dev_out, host_out):
                    s_o.wait_event(prev_cmp[c])
                    with torch.cuda.stream(s_o):
                        h_t[sl].copy_(d_t[sl], non_blocking=True)
                    e = torch.cuda.Event()
                    e.record(s_o)
                    evs.append(e)
                prev_out[c] = evs

        ref_out, ref_dk = out.view(BH, w.N, -1).cpu(), dk.view(BH, w.N, -1).cpu()
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        if cp.causal_product_status(ws_fc) != cp.CP_OK or cp.causal_product_status(ws_bc) != cp.CP_OK:
            raise RuntimeError("kernel status word reports an error in the end-to-end run")
        # chunks are split into scan segments, so they match the resident run
        # to rounding, not bitwise
        for got, ref in ((ho, ref_out), (hdk, ref_dk)):
            scale = ref.float().abs().max().item()
            if (got.float() - ref.float()).abs().max().item() > 2e-2 * scale:
                raise RuntimeError("end-to-end results differ from the resident-input run")
        barrier(world)
        n_e2e = max(3, min(args.steps, 10))
        t_start_ev, t_end_ev = (torch.cuda.Event(enable_timing=True) for _ in range(2))
        torch.cuda.synchronize()
        t_start_ev.record(stream)
        for st_ in s_ins + s_outs + [s_cmp]:
            st_.wait_stream(stream)
        for _ in range(n_e2e):
            e2e_step()
        for st_ in s_ins + s_outs + [s_cmp]:
            stream.wait_stream(st_)
        t_end_ev.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(t_start_ev.elapsed_time(t_end_ev), world)
        h2d = sum(t.numel() * t.element_size() for t in (q, k, v, g))
        d2h = sum(t.numel() * t.element_size() for t in (out, dq, dk, dv))
        e2e = {"value": w.token_heads * world * n_e2e / (e2e_ms / 1e3) / 1e6, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_e2e,
               "chunks": n_chunks,
               "timing": "CUDA events; copies and compute of successive chunks overlap"}

    # ---- the same step with a carried state: S_0 in, S_N out, dL/dS_N in,
    # dL/dS_0 out (the scans seed and hand on fp32 [B,H,D,M] states)
    st_shape = (w.B, w.H, w.D, w.M)
    if not args.no_extras:
        s0 = torch.randn(st_shape, device=dev)
        ds_n = torch.randn(st_shape, device=dev)
        s_n = torch.empty(st_shape, device=dev)
        ds_0 = torch.empty(st_shape, device=dev)

    def state_step():
        cp.causal_product_fwd(qd, kd, vd, out=out, workspace=ws_f, stream=stream, state_in=s0,
                              return_state=True, state_out=s_n)
        cp.causal_product_bwd(qd, kd, vd, gd, dq, dk, dv, workspace=ws_b, stream=stream,
                              state_in=s0, grad_state_out=ds_n, return_state_grad=True,
                              grad_state_in=ds_0)

    state_ms = None
    if not args.no_extras:
        for _ in range(3):
            state_step()
        torch.cuda.synchronize()
        n_st = max(3, min(args.steps, 10))
        st0, st1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        st0.record(stream)
        for _ in range(n_st):
            state_step()
        st1.record(stream)
        torch.cuda.synchronize()
        state_ms = max_over_ranks(st0.elapsed_time(st1), world) / n_st

    # ---- decoding step (one new row per (b,h), state updated in place) on a
    # serving-size batch whose fp32 state (128 MiB) exceeds L2
    dec = None
    if w.dtype == "bf16" and not args.no_extras:
        dB, dH = 512, w.H
        g_ = torch.Generator(device="cpu").manual_seed(77)
        dq_ = torch.randn((dB, dH, w.D), generator=g_).to(dev, w.torch_dtype)
        dk_ = torch.randn((dB, dH, w.D), generator=g_).to(dev, w.torch_dtype)
        dv_ = torch.randn((dB, dH, w.M), generator=g_).to(dev, w.torch_dtype)
        dst = torch.zeros((dB, dH, w.D, w.M), dtype=torch.float32, device=dev)
        dout = torch.empty((dB, dH, w.M), dtype=w.torch_dtype, device=dev)
        for _ in range(3):
            cp.causal_product_decode(dq_, dk_, dv_, dst, out=dout, stream=stream)
        torch.cuda.synchronize()
        n_dec = 20
        d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        d0.record(stream)
        for _ in range(n_dec):
            cp.causal_product_decode(dq_, dk_, dv_, dst, out=dout, stream=stream)
        d1.record(stream)
        torch.cuda.synchronize()
        dec_ms = max_over_ranks(d0.elapsed_time(d1), world) / n_dec
        s_ = 2
        dec_bytes = dB * dH * (8 * w.D * w.M + s_ * (2 * w.D + 2 * w.M))
        dec = {"B": dB, "H": dH, "D": w.D, "M": w.M, "us_per_step": dec_ms * 1e3,
               "tokens_per_s": dB * dH * world / (dec_ms / 1e3),
               "bytes_per_step": dec_bytes, "achieved_gbs": dec_bytes / (dec_ms / 1e3) / 1e9,
               "frac": dec_bytes / (dec_ms / 1e3) / 1e9 / load_peaks()[0],
               "kernel": "decode_kernel", "bound": "hbm"}

    # ---- normaliser z_i = q_i . sum_{j<=i} k_j of the same q, k, and its
    # backward (dq, dk from dL/dz); vector scans, bound by HBM
    norm = None
    if not args.no_extras:
        gz = torch.randn((w.B, w.H, w.N), generator=torch.Generator().manual_seed(78)).to(dev)
        zb = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
        nq, nk = torch.empty_like(qd), torch.empty_like(kd)
        ws_n = torch.zeros(cp.load_library().causal_product_normalizer_workspace_size(
            w.B, w.H, w.N, w.D, 1 if w.dtype == "bf16" else 0), dtype=torch.uint8, device=dev)

        def norm_fwd():
            cp.causal_product_normalizer(qd, kd, z=zb, workspace=ws_n, stream=stream)

        def norm_bwd():
            cp.causal_product_normalizer_bwd(qd, kd, gz, nq, nk, workspace=ws_n, stream=stream)

        def timed(fn, n=20):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(n):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            return max_over_ranks(e0.elapsed_time(e1), world) / n

        nf_ms, nb_ms = timed(norm_fwd), timed(norm_bwd)
        s_ = 2 if w.dtype == "bf16" else 4
        # forward reads q and k, writes z (fp32); backward reads k, q and
        # dL/dz twice and writes dq and dk
        nf_bytes = (2 * s_ * w.D + 4) * w.token_heads
        nb_bytes = (4 * s_ * w.D + 8) * w.token_heads
        peak = load_peaks()[0]
        norm = {"kernel": "z: norm_pp_kernel (one CTA per problem); dq, dk: norm_lb_kernel "
                          "(single pass, look-back)", "bound": "hbm",
                "fwd": {"us": nf_ms * 1e3, "bytes": nf_bytes,
                        "achieved_gbs": nf_bytes / (nf_ms / 1e3) / 1e9,
                        "frac": nf_bytes / (nf_ms / 1e3) / 1e9 / peak},
                "bwd": {"us": nb_ms * 1e3, "bytes": nb_bytes,
                        "achieved_gbs": nb_bytes / (nb_ms / 1e3) / 1e9,
                        "frac": nb_bytes / (nb_ms / 1e3) / 1e9 / peak},
                "timing": "CUDA events over 20 calls each; one launch per output (z; dq "
                          "then dk), after a workspace fill on the look-back kernel"}
        # the same with phi = elu + 1 applied to raw x ~ N(0, 1) in the kernel;
        # its backward streams q and k in both launches
        rq, rk, _, _ = make_inputs(w.B, w.H, w.N, w.D, 1, w.torch_dtype, seed=80,
                                   feature="normal", backward=False)
        rq, rk = rq.to(dev), rk.to(dev)
        ff_ms = timed(lambda: cp.causal_product_normalizer(rq, rk, z=zb, workspace=ws_n,
                                                           stream=stream, feature="elu1"))
        fb_ms = timed(lambda: cp.causal_product_normalizer_bwd(rq, rk, gz, nq, nk, workspace=ws_n,
                                                               stream=stream, feature="elu1"))
        fb_bytes = (6 * s_ * w.D + 8) * w.token_heads
        norm["feature_elu1"] = {
            "kernel": "z: norm_lb_kernel; dq, dk: norm_pp_kernel",
            "fwd": {"us": ff_ms * 1e3, "bytes": nf_bytes,
                    "frac": nf_bytes / (ff_ms / 1e3) / 1e9 / peak},
            "bwd": {"us": fb_ms * 1e3, "bytes": fb_bytes,
                    "frac": fb_bytes / (fb_ms / 1e3) / 1e9 / peak}}
        del rq, rk
        # out and z from one call: the product kernel writes z too where it
        # can (reads q, k, v once; writes out and z)
        fo_n = torch.empty_like(vd)
        ws_fn = torch.zeros(cp.load_library().causal_product_fwd_norm_workspace_size(
            w.B, w.H, w.N, w.D, w.M, cp._DTYPES[w.torch_dtype]), dtype=torch.uint8, device=dev)
        fn_ms = timed(lambda: cp.causal_product_fwd_norm(qd, kd, vd, out=fo_n, z=zb,
                                                         workspace=ws_fn, stream=stream))
        fn_bytes = (s_ * (2 * w.D + 2 * w.M) + 4) * w.token_heads
        norm["fused_with_forward"] = {
            "call": "causal_product_fwd_norm (out and z)",
            "launches": cp.causal_product_launch_count(w.B, w.H, w.N, w.D, w.M, w.torch_dtype,
                                                       norm=True),
            "us": fn_ms * 1e3, "bytes": fn_bytes,
            "achieved_gbs": fn_bytes / (fn_ms / 1e3) / 1e9,
            "frac": fn_bytes / (fn_ms / 1e3) / 1e9 / peak,
            "forward_alone_us": fwd_ms / args.steps * 1e3,
            "forward_then_normalizer_us": fwd_ms / args.steps * 1e3 + nf_ms * 1e3}
        del fo_n, ws_fn

    # ---- the forward with the feature map phi(x) = elu(x) + 1 applied to raw
    # x_q, x_k ~ N(0, 1) inside the product kernel (both branches of phi
    # taken); it moves the same bytes as the plain forward
    feat = None
    if not args.no_extras:
        xq_, xk_, _, _ = make_inputs(w.B, w.H, w.N, w.D, 1, w.torch_dtype, seed=79,
                                     feature="normal", backward=False)
        xq_, xk_ = xq_.to(dev), xk_.to(dev)
        fo = torch.empty_like(vd)

        def feat_fwd():
            cp.causal_product_fwd_feature(xq_, xk_, vd, "elu1", out=fo, workspace=ws_f,
                                          stream=stream)

        ff_ms = timed(feat_fwd)
        s_ = 2 if w.dtype == "bf16" else 4
        fb = s_ * (2 * w.D + 2 * w.M) * w.token_heads
        feat = {"kernel": "tc_causal_kernel, phi = elu + 1 applied in shared memory",
                "bound": "hbm", "us": ff_ms * 1e3, "bytes": fb,
                "achieved_gbs": fb / (ff_ms / 1e3) / 1e9,
                "frac": fb / (ff_ms / 1e3) / 1e9 / load_peaks()[0],
                "plain_fwd_us": fwd_ms / args.steps * 1e3,
                "timing": "CUDA events over 20 calls"}
        if w.backward:
            # the backward with respect to the raw rows: phi on the loaded
            # tiles, phi' on the stored gradients; the plain backward's bytes
            fdq, fdk, fdv = torch.empty_like(xq_), torch.empty_like(xk_), torch.empty_like(vd)
            ws_fb = torch.empty(cp.causal_product_feature_workspace_size(
                w.B, w.H, w.N, w.D, w.M, w.torch_dtype, backward=True), dtype=torch.uint8,
                device=dev)

            def feat_bwd():
                cp.causal_product_bwd_feature(xq_, xk_, vd, gd, "elu1", grad_q=fdq, grad_k=fdk,
                                              grad_v=fdv, workspace=ws_fb, stream=stream)

            fbw_ms = timed(feat_bwd)
            bb = s_ * (4 * w.D + 3 * w.M) * w.token_heads
            feat.update({"bwd_us": fbw_ms * 1e3, "bwd_bytes": bb,
                         "bwd_achieved_gbs": bb / (fbw_ms / 1e3) / 1e9,
                         "bwd_frac": bb / (fbw_ms / 1e3) / 1e9 / load_peaks()[0],
                         "plain_bwd_us": bwd_ms / args.steps * 1e3,
                         "bwd_kernels": ("D, M <= 64: the dk/dv scan and the dq scan of "
                                         "tc_bwd_kernel on raw rows (phi on the loaded tiles, "
                                         "phi' on the stored gradients); wider: three "
                                         "tc_causal_kernel products; no phi workspace")
                                        if w.dtype == "bf16" else "map, backward, chain rule"})
            if int(cp.causal_product_status(ws_fb, stream)) != 0:
                raise RuntimeError("kernel status word reports an error in the feature backward")
            del fdq, fdk, fdv, ws_fb
        del xq_, xk_, fo

    # ---- positive random features (the D = 256 workload's feature map) from
    # the raw rows: the forward with the map inside the product kernel, the
    # backward through the feature map kernels
    favor = None
    if not args.no_extras:
        favor = time_favor(cp, dev, stream, args.steps, args.warmup, world)

    # ---- the other four workloads, each as a step of its own pass (forward
    # for the fp32 ones, whose workload is forward only, with their
    # fwd + bwd beside it), same steps and warm-up, CUDA events
    others = None
    if not args.no_others:
        others = {}
        for name, w2 in WORKLOADS.items():
            if name == w.name:
                continue
            others[name] = time_workload(cp, w2, dev, stream, args.steps, args.warmup, world)

    # ---- roofline of the dominant kernel.  Unsplit problems on fewer than
    # the SMs: the single backward launch (dk/dv and dq scans; the backward
    # call is exactly that launch, timed by its own events); otherwise the
    # causal-product kernel (two launches per step, the forward call is one).
    hbm_gbs, bf16_tf, peak_src = load_peaks()
    s = 2 if w.dtype == "bf16" else 4
    fused = _fused_dkdv(w)
    segmented = _segmented(w)
    # one causal product over (BH, N) moves D' + D' + M' + M' columns per row
    # (q', k', v' read, out' written)
    fwd_bytes = s * (2 * w.D + 2 * w.M) * w.token_heads
    fwd_ms_launch = fwd_ms / args.steps
    fwd_traffic = None
    if not segmented and PROFILED_TRAFFIC["source_sha256"] == kernel_sha():
        fwd_traffic = PROFILED_TRAFFIC["bytes_per_launch"]
    fwd_entry = {"kernel": "tc_causal_kernel (one causal product per launch)", "bound": "hbm",
                 "bytes_per_launch": fwd_bytes, "avg_launch_ms": fwd_ms_launch,
                 "achieved": fwd_bytes / (fwd_ms_launch / 1e3) / 1e9,
                 "frac": fwd_bytes / (fwd_ms_launch / 1e3) / 1e9 / hbm_gbs,
                 "traffic": fwd_traffic,
                 "timing": "K forward calls (one launch each) back to back, CUDA events "
                           "on their stream at both ends"}
    bwd_entry = None
    if fused and not segmented:
        if _single_launch_bwd(w):
            # one launch: the fused dk/dv scans (read q, k, v, g; write dk,
            # dv) and the dq scans (read g, v, k; write dq).  The roofline
            # counts the backward's algorithmic bytes (read q, k, v, g once,
            # write dq, dk, dv); the kernel's own reads are reported beside it
            b_bytes = s * (4 * w.D + 3 * w.M) * w.token_heads
            impl_bytes = s * (5 * w.D + 5 * w.M) * w.token_heads
            b_ms = bwd_ms / args.steps
            b_traffic = None
            if PROFILED_TRAFFIC_BWD["source_sha256"] == kernel_sha(BWD_SOURCES):
                b_traffic = PROFILED_TRAFFIC_BWD["bytes_per_launch"]
            name, timing = ("tc_bwd_kernel", "K backward calls (one launch each) back to back, "
                            "CUDA events on their stream at both ends")
        else:
            # the fused dk/dv launch, timed as the backward call minus its
            # causal-product launch (dq, the same bytes as the forward when D = M)
            b_bytes = s * (3 * w.D + 3 * w.M) * w.token_heads
            impl_bytes = b_bytes
            b_ms = (bwd_ms - fwd_ms) / args.steps
            b_traffic = None
            name, timing = "tc_dkdv_kernel", "backward call minus one forward launch"
        bwd_entry = {"kernel": name, "bound": "hbm", "bytes_per_launch": b_bytes,
                     "implementation_bytes_per_launch": impl_bytes,
                     "avg_launch_ms": b_ms, "achieved": b_bytes / (b_ms / 1e3) / 1e9,
                     "frac": b_bytes / (b_ms / 1e3) / 1e9 / hbm_gbs, "traffic": b_traffic,
                     "timing": timing}
    if bwd_entry is not None and bwd_entry["kernel"] == "tc_bwd_kernel":
        dominant, kernels = bwd_entry, [fwd_entry]
    else:
        dominant, kernels = fwd_entry, [bwd_entry] if bwd_entry is not None else []
    step_roofline_ms = algorithmic_bytes(w) / (hbm_gbs * 1e9) * 1e3

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "D": w.D, "M": w.M,
                   "features": w.feature, "l2": "inputs larger than L2 (no flush)",
                   "fwd_ms": fwd_ms / args.steps, "bwd_ms": bwd_ms / args.steps,
                   "fwd_isolated_ms": fwd_iso_ms / args.steps,
                   "bwd_isolated_ms": bwd_iso_ms / args.steps,
                   "step_timing": "K back-to-back fwd+bwd steps, CUDA events at both ends; "
                                  "fwd_ms / bwd_ms: K forward calls back to back, then K "
                                  "backward calls, events at both ends of each run; "
                                  "*_isolated_ms: events around every call",
                   "step_hbm_roofline_frac": step_roofline_ms / ms_per_step,
                   "parallelism": f"replicas x{world} (b,h)-sharded, no collective"},
        "roofline": {"bound": "hbm", "achieved": dominant["achieved"], "peak": hbm_gbs,
                     "unit": "GB/s", "frac": dominant["frac"], "traffic": dominant["traffic"],
                     "kernel": dominant["kernel"], "peak_source": f"{peak_src} hbm_gbs",
                     "bytes_per_launch": dominant["bytes_per_launch"],
                     "implementation_bytes_per_launch": dominant.get(
                         "implementation_bytes_per_launch", dominant["bytes_per_launch"]),
                     "bytes_basis": "algorithmic bytes per launch: forward s(2D+2M), "
                                    "backward s(4D+3M) per token-head",
                     "avg_launch_ms": dominant["avg_launch_ms"], "timing": dominant["timing"],
                     "other_kernels": kernels},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks.summary(t_start, t_end, soak_from),
        "e2e": e2e,
        "decode": dec,
        "normalizer": norm,
        "feature_map": feat,
        "other_workloads": others,
        "favor": favor,
        "carried_state": None if state_ms is None else {
            "ms_per_step": state_ms, "value": w.token_heads * world / (state_ms / 1e3) / 1e6,
            "unit": UNIT, "note": "fwd with S_0 in and S_N out, bwd with dS_N in and dS_0 out"},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_budget)
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def step_bytes(w, backward=True):
    """Algorithmic bytes of one step: forward s(2D+2M), backward s(4D+3M)
    per token-head."""
    s = 2 if w.dtype == "bf16" else 4
    per_th = s * (2 * w.D + 2 * w.M) + (s * (4 * w.D + 3 * w.M) if backward else 0)
    return per_th * w.token_heads


def step_flops(w, backward=True):
    """Algorithmic flops of one step with the chunk convention C = 64:
    forward 4DM + C(D+M), backward 10DM + C(3D+2M) per token-head."""
    C = 64
    per_th = 4 * w.D * w.M + C * (w.D + w.M)
    if backward:
        per_th += 10 * w.D * w.M + C * (3 * w.D + 2 * w.M)
    return per_th * w.token_heads


def fp32_fma_peak_tflops():
    """FP32 FMA peak derived from unit counts and the clock (not measured):
    152 SMs x 128 lanes x 2 flop x the maximum SM clock."""
    mhz = 2070.0
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            mhz = float(json.load(f).get("sm_max_mhz", mhz))
    return 152 * 128 * 2 * mhz * 1e6 / 1e12


def time_workload(cp, w, dev, stream, steps, warmup, world):
    """Time one workload's step (its own pass) and its fwd + bwd step with
    CUDA events on `stream`, and report the step roofline."""
    import torch
    from prefix_sum_outer_gb300.workloads import make_inputs
    q, k, v, g = make_inputs(w.B, w.H, w.N, w.D, w.M, w.torch_dtype, seed=w.seed,
                             feature=w.feature, x_std=w.x_std, backward=True)
    qd, kd, vd, gd = (t.to(dev) for t in (q, k, v, g))
    out = torch.empty_like(vd)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    ws_f = torch.zeros(cp.causal_product_workspace_size(w.B, w.H, w.N, w.D, w.M, w.torch_dtype,
                                                        False), dtype=torch.uint8, device=dev)
    ws_b = torch.zeros(cp.causal_product_workspace_size(w.B, w.H, w.N, w.D, w.M, w.torch_dtype,
                                                        True), dtype=torch.uint8, device=dev)

    ckpt = torch.empty(max(cp.causal_product_checkpoint_size(w.B, w.H, w.N, w.D, w.M,
                                                             w.torch_dtype) // 4, 1),
                       dtype=torch.float32, device=dev)

    def fwd():
        cp.causal_product_fwd(qd, kd, vd, out=out, workspace=ws_f, stream=stream)

    def fwd_bwd():
        # the training step: the forward leaves checkpoints for the backward
        cp.causal_product_fwd_ckpt(qd, kd, vd, out=out, ckpt=ckpt, workspace=ws_f, stream=stream)
        cp.causal_product_bwd_ckpt(qd, kd, vd, gd, ckpt, dq, dk, dv, workspace=ws_b,
                                   stream=stream)

    def timed(fn):
        for _ in range(max(warmup, 3)):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(e0.elapsed_time(e1), world) / steps

    hbm_gbs = load_peaks()[0]
    res = {"B": w.B, "H": w.H, "N": w.N, "D": w.D, "M": w.M, "dtype": w.dtype,
           "features": w.feature, "pass": "fwd+bwd" if w.backward else "fwd"}
    for label, fn, bwd in (("fwd", fwd, False), ("fwd_bwd", fwd_bwd, True)):
        ms = timed(fn)
        nbytes, flops = step_bytes(w, bwd), step_flops(w, bwd)
        entry = {"ms_per_step": ms, "value": w.token_heads * world / (ms / 1e3) / 1e6,
                 "unit": UNIT, "bytes_per_step": nbytes,
                 "step_hbm_roofline_frac": nbytes / (hbm_gbs * 1e9) / (ms / 1e3),
                 "flops_per_step": flops}
        if w.dtype == "f32":
            peak = fp32_fma_peak_tflops()
            entry["bound"] = "alu"
            entry["step_alu_roofline_frac"] = flops / (peak * 1e12) / (ms / 1e3)
            entry["alu_peak_tflops"] = peak
            entry["alu_peak_source"] = "derived: 152 SMs x 128 FP32 lanes x 2 x max SM clock"
        else:
            entry["bound"] = "hbm"
        entry["launches"] = (_launch_count(w, True, ckpt=True) + _launch_count(w, False, ckpt=True)
                             if bwd else _launch_count(w, False))
        res[label] = entry
    if cp.causal_product_status(ws_f) != cp.CP_OK or cp.causal_product_status(ws_b) != cp.CP_OK:
        raise RuntimeError(f"kernel status word reports an error on {w.name}")
    res["timing"] = (f"CUDA events over {steps} back-to-back steps after "
                     f"{max(warmup, 3)} warm-up steps")
    del qd, kd, vd, gd, out, dq, dk, dv, ws_f, ws_b
    torch.cuda.empty_cache()
    return res


def time_favor(cp, dev, stream, steps, warmup, world):
    """Positive random features phi(x) = exp(W x - |x|^2/2)/sqrt(D) computed
    in the kernels from raw rows (B=4 H=8 N=8229, R=64, D=256, M=64: the
    D = 256 workload before its feature map), forward and backward."""
    import torch
    from prefix_sum_outer_gb300.workloads import favor_raw_inputs
    B, H, N, D, M = 4, 8, 8229, 256, 64
    W, xq, xk = favor_raw_inputs(B, H, N, D, 5)
    R = W.shape[1]
    gen = torch.Generator().manual_seed(6)
    v = torch.randn((B, H, N, M), generator=gen)
    g = torch.randn((B, H, N, M), generator=gen)
    xq, xk, v, g, W = (t.to(torch.bfloat16).to(dev) for t in (xq, xk, v, g, W))
    out, dxq, dxk, dv = (torch.empty_like(t) for t in (v, xq, xk, v))
    lib = cp.load_library()
    ws_f = torch.zeros(lib.causal_product_favor_workspace_size(B, H, N, R, D, M, 1, 0),
                       dtype=torch.uint8, device=dev)
    ws_b = torch.zeros(lib.causal_product_favor_workspace_size(B, H, N, R, D, M, 1, 1),
                       dtype=torch.uint8, device=dev)

    def fwd():
        cp.causal_product_fwd_favor(xq, xk, v, W, out=out, workspace=ws_f, stream=stream)

    def bwd():
        cp.causal_product_bwd_favor(xq, xk, v, W, g, dxq, dxk, dv, workspace=ws_b, stream=stream)

    def timed(fn):
        for _ in range(max(warmup, 3)):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(e0.elapsed_time(e1), world) / steps

    f_ms, b_ms = timed(fwd), timed(bwd)
    if cp.causal_product_status(ws_f) != cp.CP_OK or cp.causal_product_status(ws_b) != cp.CP_OK:
        raise RuntimeError("kernel status word reports an error in the feature-map run")
    th = B * H * N
    # algorithmic bytes: forward reads xq, xk (R), v (M) and writes out (M);
    # backward reads xq, xk, v, g and writes dxq, dxk, dv
    fb, bb = 2 * (2 * R + 2 * M) * th, 2 * (4 * R + 3 * M) * th
    peak = load_peaks()[0]
    return {"B": B, "H": H, "N": N, "R": R, "D": D, "M": M,
            "fwd": {"us": f_ms * 1e3, "kernel": "favor_causal_kernel (map fused into the product)",
                    "bytes": fb, "frac": fb / (f_ms / 1e3) / 1e9 / peak},
            "bwd": {"us": b_ms * 1e3, "bytes": bb, "frac": bb / (b_ms / 1e3) / 1e9 / peak,
                    "kernel": "favor_map_kernel, three products, favor_chain_kernel"},
            "value_fwd_bwd": th * world / ((f_ms + b_ms) / 1e3) / 1e6, "unit": UNIT,
            "timing": f"CUDA events over {steps} calls each"}


def _fused_dkdv(w):
    """bf16 with D, M <= 64: the backward computes dk and dv in one scan."""
    return w.dtype == "bf16" and w.D <= 64 and w.M <= 64


def _launch_count(w, backward, ckpt=False):
    import prefix_sum_outer_gb300 as cp
    c = cp.causal_product_launch_count(w.B, w.H, w.N, w.D, w.M, w.torch_dtype, backward,
                                       ckpt=ckpt)
    if c < 0:
        raise RuntimeError(f"shape of {w.name} rejected by the library")
    return c


def _segmented(w):
    """The forward scan is split into segments (sums, prefix, scan)."""
    return _launch_count(w, False) > 1


def _single_launch_bwd(w):
    """The whole backward (dk/dv and dq scans) is one launch."""
    return _fused_dkdv(w) and _launch_count(w, True, ckpt=True) == 1


def _launches_per_step(w):
    """Kernels one fwd + bwd step launches, as the library plans them (one per
    unsplit scan, three per split scan, one for the whole backward when it
    fits a single launch)."""
    return _launch_count(w, False, ckpt=True) + _launch_count(w, True, ckpt=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-chunks", type=int, default=2)
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the carried-state and decoding measurements")
    ap.add_argument("--no-others", action="store_true",
                    help="skip timing the other four workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    args = ap.parse_args(argv)
    world, rank, local = dist_setup()
    try:
        if args.impl == "reference":
            return run_reference(args, world, rank)
        return run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
