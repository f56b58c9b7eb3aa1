#!/usr/bin/env python
"""Benchmark of the Lightning Attention RNN mixer on GB300 (one JSON line).

Headline: hla_prefill over B=1, T=524288, H=16, d=128 bf16 (inputs resident in
HBM, 8 GiB, far larger than L2), reported as Mtok/s and as a fraction of the
HBM roofline.  The same line carries the batched decode step (B=64, H=32,
d=128, state from a 4096-token prefill, L2 flushed between steps) and the
distillation-shaped forward+backward (B=8, T=16384, H=32), the end-to-end
figure through the public API with pinned host buffers, the fp64 CPU oracle
timed on a bounded sample, and the SM clocks sampled during the timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs an independent replica (weak scaling); rank 0
prints the line.  ``--impl reference`` times the CPU oracle alone.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Lightning-attn prefill Mtok/s @512K + decode tok/s (B=64), % of roofline"
BF16 = 2


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-decode", action="store_true")
    p.add_argument("--no-backward", action="store_true")
    p.add_argument("--no-mma-bench", action="store_true")
    p.add_argument("--no-attention", action="store_true")
    p.add_argument("--no-layer", action="store_true",
                   help="skip the RNN layer with its projections (hla_project_in / _out)")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="target CPU time of the oracle sample")
    p.add_argument("--prefill-T", type=int, default=0,
                   help="override T of the prefill workload (small cases for ncu captures)")
    p.add_argument("--fb-recompute", action="store_true",
                   help="forward + backward without saved features (the backward "
                        "recomputes the q / k feature map)")
    p.add_argument("--backward-B", type=int, default=0,
                   help="override B of the forward+backward workload (small cases for ncu captures)")
    return p.parse_args()


def measured_traffic(record: str, sources, units: float):
    """DRAM bytes per launch of a kernel from a committed ncu summary
    (profiles/<record>: `bytes_per_unit` and the sha256 of the listed kernel
    sources), scaled to `units`; None when a source changed since the capture."""
    import hashlib
    import re
    path = os.path.join(ROOT, "profiles", record)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_b = re.search(r"bytes_per_(?:token_head|unit):\s*([0-9.]+)", text)
    m_s = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    if not (m_b and m_s):
        return None
    h = hashlib.sha256()
    for f in sources:
        h.update(open(os.path.join(ROOT, "rnn_sequence_mixer_gb300", "csrc", f), "rb").read())
    if h.hexdigest() != m_s.group(1):
        return None
    return float(m_b.group(1)) * units


def prefill_launches(api, B, T, H, chunk, gamma, passes=0) -> int:
    """Kernels one prefill call launches (the library's own plan, hla_prefill_launches)."""
    return api.prefill_launches(api.make_shape(B, T, H, 128, chunk=chunk, passes=passes), gamma)


def backward_launches(api, B, T, H, chunk, gamma, with_fwd_ws) -> int:
    return api.backward_launches(api.make_shape(B, T, H, 128, chunk=chunk), gamma, with_fwd_ws)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


# ----------------------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        if not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- oracle timing


def host_cpu_model() -> str:
    """The host CPU's model name (lscpu), else the machine type."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.machine()


def oracle_sample(w, seconds: float, threads: int = 0):
    """Time the fp64 oracle on a bounded sample of workload ``w`` (all H heads of
    one sequence, the first n tokens), growing n until the sample takes about
    ``seconds``; on ``threads`` cores (0: all).  Returns (tokens/s, n_tokens,
    threads, seconds)."""
    import numpy as np
    import torch

    import oracle
    from rnn_sequence_mixer_gb300 import inputs

    all_threads = oracle.threads()
    oracle.set_threads(threads or all_threads)
    try:
        return _oracle_sample(w, seconds, oracle, np, torch, inputs)
    finally:
        oracle.set_threads(all_threads)


def _oracle_sample(w, seconds, oracle, np, torch, inputs):
    gam = oracle.gamma(w.H).astype(np.float32).astype(np.float64)
    n, spent = 256, 0.0
    while True:
        inp = inputs.mixer_inputs(1, n, w.H, w.d, w.dtype, w.seed, device="cpu")
        arr = {k: v.to(torch.float64).numpy() for k, v in inp.items()}
        t0 = time.perf_counter()
        oracle.prefill(arr["q"], arr["k"], arr["v"], arr["gate"], gam, base=w.rope_base, eps=w.eps)
        dt = time.perf_counter() - t0
        spent += dt
        if dt >= seconds / 4 or n >= w.T or spent >= seconds:
            return n / dt, n, oracle.threads(), dt
        n = min(w.T, max(2 * n, int(n * (seconds / 4) / max(dt, 1e-3))))


def run_reference(args):
    """--impl reference: the CPU oracle on bounded samples of the headline workload."""
    from rnn_sequence_mixer_gb300 import workloads
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = workloads.PREFILL_512K
    per = max(1.0, min(20.0, 60.0 / max(1, args.steps + args.warmup)))
    tok_s, n, cores, _ = oracle_sample(w, per)
    times = []
    import numpy as np
    import torch

    import oracle
    from rnn_sequence_mixer_gb300 import inputs
    gam = oracle.gamma(w.H).astype(np.float32).astype(np.float64)
    inp = inputs.mixer_inputs(1, n, w.H, w.d, w.dtype, w.seed, device="cpu")
    arr = {k: v.to(torch.float64).numpy() for k, v in inp.items()}
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.prefill(arr["q"], arr["k"], arr["v"], arr["gate"], gam, base=w.rope_base, eps=w.eps)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    ms = 1e3 * statistics.mean(times)
    value = n / (ms / 1e3) / 1e6
    sample = f"first {n} tokens of sequence 0, all {w.H} heads, fp64"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "Mtok/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name, "sample_tokens": n},
        "cpu_baseline": {"value": value, "unit": "Mtok/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "Mtok/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }))


# ----------------------------------------------------------------------------- GPU arms


def timed(fn, steps, warmup, stream, dist_ctx, trace_count=0, step_events=False):
    """Run fn(i, trace) warmup + steps times; returns (ms per step, per-pass ms lists).
    With step_events the harness itself records a trace of two events around
    each step (fn gets None), so the per-pass lists hold each step's time."""
    import torch
    for i in range(warmup):
        fn(i, None)
    torch.cuda.synchronize()
    dist_ctx.barrier()
    torch.cuda.synchronize()
    traces = []
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(steps):
        tr = [torch.cuda.Event(enable_timing=True) for _ in range(trace_count)] or None
        if step_events:
            tr[0].record(stream)
            fn(warmup + i, None)
            tr[1].record(stream)
        else:
            fn(warmup + i, tr)
        traces.append(tr)
    end.record(stream)
    torch.cuda.synchronize()
    dist_ctx.barrier()
    ms = start.elapsed_time(end) / steps
    passes = []
    if trace_count:
        for tr in traces:
            passes.append([tr[j].elapsed_time(tr[j + 1]) for j in range(trace_count - 1)])
    return ms, passes


class Dist:
    """One process per GPU under torchrun (RANK / LOCAL_RANK / WORLD_SIZE /
    MASTER_* from the environment).  The bench runs an independent replica on
    every rank: no data moves between ranks, only the barrier around each timed
    region and the max of the per-rank times.  backend: "nccl" for GPU runs,
    "gloo" for host-only use (tests)."""

    def __init__(self, backend: str = "nccl"):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.backend = backend
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            if not dist.is_initialized():
                dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        """The largest x over all ranks (every rank gets it)."""
        if not self.pg:
            return x
        import torch
        dev = f"cuda:{self.local}" if self.backend == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())


def job_rate(units_per_rank: float, max_ms: float, world: int) -> float:
    """Whole-job throughput of `world` replicas, each processing units_per_rank
    units, bounded by the slowest rank (units per second)."""
    return world * units_per_rank / (max_ms / 1e3)


def run_ours(args):
    import torch

    import oracle  # noqa: F401  (cpu_baseline leg only)
    from rnn_sequence_mixer_gb300 import _lib, api, inputs, workloads

    D = Dist()
    torch.cuda.set_device(D.local)
    dev = torch.device(f"cuda:{D.local}")
    _lib.load()
    hbm_peak, tc_peak, peak_src = peaks()
    stream = torch.cuda.current_stream(dev)
    launches = 0
    out = {}

    # ---------------------------------------------------------------- prefill @512K
    w = workloads.PREFILL_512K
    if args.prefill_T:
        w = dataclasses.replace(w, T=args.prefill_T, name=f"prefill_B1_T{args.prefill_T}_H16_d128_bf16")
    gam = api.gamma_schedule(w.H)
    inp = inputs.mixer_inputs(w.B, w.T, w.H, w.d, w.dtype, w.seed + 1000 * D.rank, device=dev)
    y = torch.empty_like(inp["q"])
    st = torch.empty((w.B, w.H, w.d, w.d), dtype=torch.float32, device=dev)
    ws = torch.empty(api.prefill_workspace_size(api.make_shape(w.B, w.T, w.H, w.d, chunk=w.chunk)),
                     dtype=torch.uint8, device=dev)
    n_pass = 3
    n_launch = prefill_launches(api, w.B, w.T, w.H, w.chunk, gam)

    def prefill_step(i, trace):
        api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], gam, chunk=w.chunk,
                    rope_base=w.rope_base, eps=w.eps, y=y, state_out=st, workspace=ws, trace=trace)

    with ClockSampler(D.local) as clk:
        ms, passes = timed(prefill_step, args.steps, args.warmup, stream, D, n_pass + 1)
    launches += n_launch * args.steps
    ms = D.max(ms)
    tokens = w.B * w.T
    value = job_rate(tokens, ms, D.world) / 1e6
    pass_names = ["seg_state", "state_scan", "seg_output"]
    pass_ms = [statistics.mean(p[j] for p in passes) for j in range(n_pass)]
    dom = max(range(n_pass), key=lambda j: pass_ms[j])
    th = w.B * w.T * w.H
    nseg_bytes = ws.numel()
    alg = {  # algorithmic bytes per launch of each pass
        "seg_state": th * 2 * w.d * BF16 + nseg_bytes,
        "state_scan": 2 * nseg_bytes,
        "seg_output": th * 5 * w.d * BF16,
    }
    a_bytes = alg[pass_names[dom]]
    achieved = a_bytes / (pass_ms[dom] / 1e3) / 1e9
    whole = th * 5 * w.d * BF16 / (ms / 1e3) / 1e9
    traffic = (measured_traffic("traffic_tc_output.md", ("tc_prefill.cu", "tc_common.cuh", "umma.cuh"),
                                th) if pass_names[dom] == "seg_output" else None)
    roof = {"kernel": pass_names[dom], "bound": "hbm", "achieved": achieved, "peak": hbm_peak,
            "unit": "GB/s", "frac": achieved / hbm_peak,
            "traffic": traffic / 1e9 if traffic else None, "traffic_unit": "GB per launch",
            "peak_source": f"hbm_gbs of {peak_src}",
            "pass_ms": dict(zip(pass_names, pass_ms)),
            "whole_call": {"alg_bytes": th * 5 * w.d * BF16, "achieved": whole,
                           "frac": whole / hbm_peak}}
    # the same workload with each launch plan forced: one launch (every output
    # CTA forms its entering state from the decay window) and three passes
    # (local-state pass, scan, output pass); the headline above is the library's choice
    plans = {"library_choice_launches": n_launch}
    p_steps = max(3, args.steps // 2)
    for passes, key in ((1, "one_launch_ms"), (3, "three_pass_ms")):
        def plan_step(i, trace, passes=passes):
            api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], gam, chunk=w.chunk,
                        rope_base=w.rope_base, eps=w.eps, y=y, state_out=st, workspace=ws,
                        passes=passes)
        p_ms, _ = timed(plan_step, p_steps, args.warmup, stream, D)
        plans[key] = D.max(p_ms)
        launches += prefill_launches(api, w.B, w.T, w.H, w.chunk, gam, passes) * p_steps
    roof["launch_plans"] = plans
    config = {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "d": w.d, "chunk": w.chunk,
              "rope_base": w.rope_base, "l2": "inputs larger than L2 (8 GiB resident per step)",
              "replicas": D.world}

    # ---------------------------------------------------------------- e2e through the API
    # Inputs start in pinned host memory and y / the final state end there.  The
    # sequence is streamed through hla_prefill in chunks (state chained from one
    # call to the next, RoPE positions continued by pos_offset): the host-to-device
    # copy of chunk j + 1, the prefill of chunk j and the device-to-host copy of y
    # of chunk j - 1 run on three streams at once.
    e2e = None
    if not args.no_e2e:
        n_chunk = 16 if w.T % 16 == 0 else 1
        tc = w.T // n_chunk
        host = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in inp.items()}
        for k in host:
            host[k].copy_(inp[k])
        y_host = torch.empty(y.shape, dtype=y.dtype, pin_memory=True)
        st_host = torch.empty(st.shape, dtype=st.dtype, pin_memory=True)
        dbuf = {k: torch.empty_like(v) for k, v in inp.items()}
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        shp_c = api.make_shape(w.B, tc, w.H, w.d, chunk=w.chunk)
        ws_c = torch.empty(api.prefill_workspace_size(shp_c), dtype=torch.uint8, device=dev)

        def e2e_step(i, trace):
            start = torch.cuda.Event()
            start.record(stream)
            s_in.wait_event(start)
            s_out.wait_event(start)
            for j in range(n_chunk):
                sl = slice(j * tc, (j + 1) * tc)
                with torch.cuda.stream(s_in):
                    for k in dbuf:
                        dbuf[k][:, sl].copy_(host[k][:, sl], non_blocking=True)
                    copied = torch.cuda.Event()
                    copied.record(s_in)
                stream.wait_event(copied)
                api.prefill(dbuf["q"][:, sl], dbuf["k"][:, sl], dbuf["v"][:, sl], dbuf["gate"][:, sl],
                            gam, st if j else None, chunk=w.chunk, pos_offset=j * tc,
                            rope_base=w.rope_base, eps=w.eps, y=y[:, sl], state_out=st,
                            workspace=ws_c)
                done = torch.cuda.Event()
                done.record(stream)
                s_out.wait_event(done)
                with torch.cuda.stream(s_out):
                    y_host[:, sl].copy_(y[:, sl], non_blocking=True)
            with torch.cuda.stream(s_out):
                st_host.copy_(st, non_blocking=True)
            stream.wait_stream(s_in)
            stream.wait_stream(s_out)

        # ~44 ms a step: 20 steps keep a rare slow step (another GPU's traffic on the
        # shared host link) from dominating the mean
        e_steps = max(3, min(2 * args.steps, 20))
        e_ms, e_step_ms = timed(e2e_step, e_steps, 1, stream, D, trace_count=2, step_events=True)
        launches += prefill_launches(api, w.B, tc, w.H, w.chunk, gam) * n_chunk * e_steps
        e_ms = D.max(e_ms)
        e_step_ms = [p[0] for p in e_step_ms]
        # The host link is shared with the other GPUs of the machine: a step now
        # and then takes several times the others.  value uses the mean.
        e2e = {"value": job_rate(tokens, e_ms, D.world) / 1e6, "unit": "Mtok/s",
               "ms_per_step": e_ms, "ms_per_step_median": statistics.median(e_step_ms),
               "steps_ms": [round(x, 2) for x in e_step_ms], "chunks": n_chunk,
               "h2d_bytes_per_step": sum(v.numel() * v.element_size() for v in host.values()),
               "d2h_bytes_per_step": y_host.numel() * 2 + st_host.numel() * 4}
        del host, y_host, st_host, dbuf, ws_c
    del inp, y, ws
    torch.cuda.empty_cache()

    # ---------------------------------------------------------------- decode
    def decode_leg(wd, split=0, kernel="decode_kernel"):
        """256 decode steps of workload wd after a prefill of wd.prefill_T tokens;
        split = CTAs per (sequence, head) (0: the library's choice)."""
        gd = api.gamma_schedule(wd.H)
        pre = inputs.mixer_inputs(wd.B, wd.prefill_T, wd.H, wd.d, wd.dtype, wd.seed + 1000 * D.rank,
                                  device=dev)
        _, _, state = api.prefill(pre["q"], pre["k"], pre["v"], pre["gate"], gd, chunk=wd.chunk,
                                  rope_base=wd.rope_base, eps=wd.eps)
        del pre
        steps = inputs.decode_inputs(wd.steps, wd.B, wd.H, wd.d, wd.dtype, wd.seed + 100, device=dev)
        pos = torch.full((wd.B,), wd.prefill_T, dtype=torch.int64, device=dev)
        yd = torch.empty((wd.B, 1, wd.H, wd.d), dtype=wd.dtype, device=dev)
        flush = torch.empty(512 * 2**20 // 4, dtype=torch.float32, device=dev)
        torch.cuda.synchronize()
        D.barrier()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(wd.steps)]
        for s in range(wd.steps):
            flush.fill_(float(s))  # evict the state from L2 before each step
            ev[s][0].record(stream)
            api.decode_step(steps["q"][s], steps["k"][s], steps["v"][s], steps["gate"][s], gd,
                            state, pos, rope_base=wd.rope_base, eps=wd.eps, y=yd, split=split)
            ev[s][1].record(stream)
            pos.add_(1)
        torch.cuda.synchronize()
        per = [a.elapsed_time(b) for a, b in ev]
        nl = wd.steps
        us = D.max(1e3 * statistics.mean(per))
        # The same 256 steps (flush, decode, position update) captured once as a
        # CUDA graph and replayed: the library neither allocates nor synchronizes
        # inside a call, so a decode step is capturable.  Events inside a graph
        # cannot be timed, so a second graph without the decode steps is replayed
        # too and the difference is the decode time.
        graph_us = None
        try:
            def capture(with_decode):
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph):
                    for s in range(wd.steps):
                        flush.fill_(float(s))
                        if with_decode:
                            api.decode_step(steps["q"][s], steps["k"][s], steps["v"][s],
                                            steps["gate"][s], gd, state, pos,
                                            rope_base=wd.rope_base, eps=wd.eps, y=yd, split=split)
                        pos.add_(1)
                return graph

            def replay_ms(graph):
                graph.replay()  # warm
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                torch.cuda.synchronize()
                a.record(stream)
                graph.replay()
                b.record(stream)
                torch.cuda.synchronize()
                return a.elapsed_time(b)

            g_all, g_flush = capture(True), capture(False)
            graph_us = 1e3 * (replay_ms(g_all) - replay_ms(g_flush)) / wd.steps
            nl += 2 * wd.steps
            del g_all, g_flush
        except RuntimeError:
            graph_us = None
        bytes_step = wd.B * wd.H * (2 * wd.d * wd.d * 4 + 5 * wd.d * BF16)
        ach = bytes_step / (us / 1e6) / 1e9
        # the same roofline from the graph replay: steps back to back as in a
        # decode loop, without the launch overhead of each plain call
        graph_roof = None
        if graph_us and graph_us > 0:
            g_ach = bytes_step / (graph_us / 1e6) / 1e9
            graph_roof = {"us_per_step": graph_us, "achieved": g_ach, "frac": g_ach / hbm_peak}
        res = {"workload": wd.name, "tok_s": job_rate(wd.B, us / 1e3, D.world),
               "us_per_step": us, "us_per_step_median": 1e3 * statistics.median(per),
               "graph_us_per_step": graph_us, "decode_split": split or "library's choice",
               "steps": wd.steps, "l2": "flushed (512 MiB write) before every step",
               "roofline": {"kernel": kernel, "bound": "hbm", "achieved": ach,
                            "peak": hbm_peak, "unit": "GB/s", "frac": ach / hbm_peak,
                            "alg_bytes": bytes_step, "graph_replay": graph_roof,
                            # the record belongs to the one-CTA-per-head kernel
                            "traffic": measured_traffic(
                                "traffic_decode.md", ("decode.cu", "hla_internal.cuh"),
                                wd.B * wd.H) if kernel == "decode_kernel" else None}}
        del steps, state, flush
        torch.cuda.empty_cache()
        return res, nl

    if not args.no_decode:
        out["decode"], nl = decode_leg(workloads.DECODE_B64)
        launches += nl
        # batch 1 (time per output token of one sequence), one CTA per head (the
        # library's choice) and with each head's state columns split over a
        # cluster of four CTAs beside it
        b1, nl = decode_leg(workloads.DECODE_B1)
        b1_s4, nl4 = decode_leg(workloads.DECODE_B1, split=4, kernel="decode_split_kernel")
        launches += nl + nl4
        b1["split4"] = {k: b1_s4[k] for k in ("us_per_step", "us_per_step_median",
                                               "graph_us_per_step")}
        out["decode_b1"] = b1

    # ---------------------------------------------------------------- forward + backward
    if not args.no_backward:
        wb = workloads.FWD_BWD_16K
        if args.backward_B:
            wb = dataclasses.replace(wb, B=args.backward_B, name=f"{wb.name}_B{args.backward_B}")
        gb = api.gamma_schedule(wb.H)
        ib = inputs.mixer_inputs(wb.B, wb.T, wb.H, wb.d, wb.dtype, wb.seed + 1000 * D.rank,
                                 device=dev, with_dy=True)
        shp = api.make_shape(wb.B, wb.T, wb.H, wb.d, chunk=wb.chunk)
        wsb = torch.empty(api.backward_workspace_size(shp), dtype=torch.uint8, device=dev)
        wsf = torch.empty(api.prefill_workspace_size(shp), dtype=torch.uint8, device=dev)
        yb = torch.empty_like(ib["q"])
        # the features the forward saves for the backward (fp16 q~, k~ and the norms)
        svb = (None if args.fb_recompute else
               torch.empty(api.saved_bytes(shp), dtype=torch.uint8, device=dev))

        def fb_step(i, trace):
            api.prefill(ib["q"], ib["k"], ib["v"], ib["gate"], gb, chunk=wb.chunk,
                        rope_base=wb.rope_base, eps=wb.eps, y=yb, want_state=False, workspace=wsf,
                        trace=trace[:4] if trace else None, saved=svb)
            # the backward reads the segment states the forward left in its
            # workspace and the features it saved instead of recomputing them,
            # and, from the forward's y and the saved 1/RMS(o), the normalized
            # output instead of recomputing o
            api.prefill_backward(ib["q"], ib["k"], ib["v"], ib["gate"], gb, ib["dy"],
                                 chunk=wb.chunk, rope_base=wb.rope_base, eps=wb.eps, workspace=wsb,
                                 trace=trace[4:] if trace else None, fwd_workspace=wsf, saved=svb,
                                 y=yb if svb is not None else None)

        b_steps = max(1, min(args.steps, 5))
        b_ms, b_passes = timed(fb_step, b_steps, 1, stream, D, trace_count=11)
        # forward, then the backward without its own local-state pass and scan (fwd_ws)
        launches += (prefill_launches(api, wb.B, wb.T, wb.H, wb.chunk, gb) +
                     backward_launches(api, wb.B, wb.T, wb.H, wb.chunk, gb, True)) * b_steps
        b_ms = D.max(b_ms)
        b_names = ["fwd.seg_state", "fwd.state_scan", "fwd.seg_output", None, None, None,
                   "bwd.dq", "bwd.seg_gstate", "bwd.grad_scan", "bwd.dkdv"]
        b_pass_ms = {nm: statistics.median(p[j] for p in b_passes)
                     for j, nm in enumerate(b_names) if nm}
        thb = wb.B * wb.T * wb.H
        alg_b = thb * (5 * wb.d * BF16 + 9 * wb.d * BF16)  # fwd 5 d-rows + bwd 5 in / 4 out
        # tensor-core work: MMAs of 128 x 128 x 128 per 128-token tile and head
        # (forward: local state 1 + output 4; backward: dq pass 7, or 4 from the
        # forward's y, state-gradient sums 1, dk/dv pass 7)
        n_mma = 20 - (3 if svb is not None else 0)
        flops_b = n_mma * 2.0 * 128 ** 3 * thb / 128
        roof_ms = max(alg_b / (hbm_peak * 1e9), flops_b / (tc_peak * 1e12)) * 1e3
        out["fwd_bwd"] = {"workload": wb.name, "chunk": wb.chunk, "ms_per_step": b_ms,
                          "Mtok_s": job_rate(wb.B * wb.T, b_ms, D.world) / 1e6,
                          "alg_bytes": alg_b, "frac_hbm": alg_b / (b_ms / 1e3) / 1e9 / hbm_peak,
                          "tensor_flops": flops_b, "roofline_ms": roof_ms,
                          "frac_roofline": roof_ms / b_ms, "pass_ms": b_pass_ms,
                          "saved_features": svb is not None,
                          "saved_bytes": 0 if svb is None else svb.numel()}
        del ib, wsb, wsf, yb, svb
        torch.cuda.empty_cache()

    # ---------------------------------------------------------------- softmax attention
    # The hybrid's other mixer (hla_attention_prefill) on the HypeNet-2B
    # attention shape: 16 query heads over 8 key/value heads, 16K tokens.
    # Tensor-bound: the causal QK^T and PV products are 4 d T (T + 1) / 2 FLOPs
    # per query head; q, k, v, gate and y (256 MiB) exceed L2.
    if not args.no_attention:
        wa = workloads.ATTENTION_16K
        xa = inputs.mixer_inputs(wa.B, wa.T, wa.Hq, wa.d, torch.bfloat16, wa.seed + 1000 * D.rank,
                                 device=dev)
        kva = inputs.mixer_inputs(wa.B, wa.T, wa.Hkv, wa.d, torch.bfloat16,
                                  wa.seed + 1 + 1000 * D.rank, device=dev)
        ya = torch.empty_like(xa["q"])
        wsa = torch.empty(api.attention_workspace_size(
            api.make_attn_shape(wa.B, wa.T, wa.Hq, wa.Hkv, wa.d, a=wa.a)), dtype=torch.uint8,
            device=dev)

        def attn_step(i, trace):
            api.attention_prefill(xa["q"], kva["k"], kva["v"], xa["gate"], wa.a, eps=wa.eps, y=ya,
                                  workspace=wsa)

        a_ms, _ = timed(attn_step, args.steps, args.warmup, stream, D)
        launches += args.steps
        a_ms = D.max(a_ms)
        flops_a = 4.0 * wa.d * wa.T * (wa.T + 1) / 2 * wa.Hq * wa.B
        tf = flops_a / (a_ms / 1e3) / 1e12
        out["attention"] = {"workload": wa.name, "ms_per_step": a_ms,
                            "Mtok_s": job_rate(wa.B * wa.T, a_ms, D.world) / 1e6,
                            "roofline": {"kernel": "attention", "bound": "tensor",
                                         "achieved": tf, "peak": tc_peak, "unit": "TFLOP/s",
                                         "frac": tf / tc_peak, "alg_flops": flops_a,
                                         "peak_source": f"bf16_tflops of {peak_src}"}}
        del xa, kva, ya, wsa
        torch.cuda.empty_cache()

    # ---------------------------------------------------------------- RNN layer with projections
    # x [B, T, D] -> hla_project_in (x W_q,k,v,z, the feature map in the GEMM
    # epilogue) -> hla_prefill_features -> hla_project_out (W_o): HypeNet-2B's
    # RNN layer at 16K tokens.  The GEMMs are tensor-bound (2 M D 4 H d and
    # 2 M H d D FLOPs); the mixer between them is HBM-bound (1280 B per token-head).
    if not args.no_layer:
        wl = workloads.LAYER_16K
        li = inputs.layer_inputs(wl.B, wl.T, wl.D, wl.H, wl.d, wl.seed + 1000 * D.rank, device=dev)
        gl = api.gamma_schedule(wl.H)
        shp_l = api.make_shape(wl.B, wl.T, wl.H, wl.d, chunk=wl.chunk, rope_base=wl.rope_base)
        feat = torch.empty(api.saved_bytes(shp_l), dtype=torch.uint8, device=dev)
        vl = torch.empty((wl.B, wl.T, wl.H, wl.d), dtype=torch.bfloat16, device=dev)
        gatel = torch.empty_like(vl)
        yl = torch.empty_like(vl)
        outl = torch.empty((wl.B, wl.T, wl.D), dtype=torch.bfloat16, device=dev)
        wsl = torch.empty(api.prefill_workspace_size(shp_l), dtype=torch.uint8, device=dev)
        wsp = torch.empty(api.project_workspace_size(), dtype=torch.uint8, device=dev)

        def l_in(i, trace):
            api.project_in(li["x"], li["w_qkvz"], rope_base=wl.rope_base, eps=wl.eps, chunk=wl.chunk,
                           features=feat, v=vl, gate=gatel, workspace=wsp)

        def l_mix(i, trace):
            api.prefill_features(feat, vl, gatel, gl, chunk=wl.chunk, rope_base=wl.rope_base,
                                 eps=wl.eps, y=yl, want_state=False, workspace=wsl)

        def l_out(i, trace):
            api.project_out(yl, li["w_o"], out=outl, workspace=wsp)

        def l_all(i, trace):
            l_in(i, trace)
            l_mix(i, trace)
            l_out(i, trace)

        lm = {}
        for key, fn in (("project_in", l_in), ("prefill_features", l_mix), ("project_out", l_out),
                        ("layer", l_all)):
            t_ms, _ = timed(fn, args.steps, args.warmup, stream, D)
            lm[key] = D.max(t_ms)
        n_mix = prefill_launches(api, wl.B, wl.T, wl.H, wl.chunk, gl)
        launches += args.steps * (1 + n_mix + 1) * 2
        M = wl.B * wl.T
        f_in, f_out = 2.0 * M * wl.D * 4 * wl.H * wl.d, 2.0 * M * wl.H * wl.d * wl.D
        tf_in, tf_out = f_in / (lm["project_in"] / 1e3) / 1e12, f_out / (lm["project_out"] / 1e3) / 1e12
        mix_bytes = M * wl.H * 5 * wl.d * BF16
        out["layer"] = {
            "workload": wl.name, "ms_per_step": lm["layer"],
            "Mtok_s": job_rate(M, lm["layer"], D.world) / 1e6, "pass_ms": lm,
            "project_in": {"bound": "tensor", "achieved": tf_in, "peak": tc_peak, "unit": "TFLOP/s",
                           "frac": tf_in / tc_peak, "alg_flops": f_in,
                           "peak_source": f"bf16_tflops of {peak_src}"},
            "project_out": {"bound": "tensor", "achieved": tf_out, "peak": tc_peak, "unit": "TFLOP/s",
                            "frac": tf_out / tc_peak, "alg_flops": f_out,
                            "peak_source": f"bf16_tflops of {peak_src}"},
            "prefill_features": {"bound": "hbm", "alg_bytes": mix_bytes,
                                 "achieved": mix_bytes / (lm["prefill_features"] / 1e3) / 1e9,
                                 "peak": hbm_peak, "unit": "GB/s",
                                 "frac": mix_bytes / (lm["prefill_features"] / 1e3) / 1e9 / hbm_peak,
                                 "launches": n_mix}}
        del li, feat, vl, gatel, yl, outl, wsl, wsp
        torch.cuda.empty_cache()

    # ---------------------------------------------------------------- MMA ceiling
    # The output pass's four MMAs per 128-token tile, issued back to back on
    # shared-memory-resident operands, one CTA per SM: the tensor-core ceiling of
    # the pass (its own MMAs keep the tensor pipe ~16 % busy; CUDA-core work
    # bounds it).
    if not args.no_mma_bench:
        import ctypes
        from rnn_sequence_mixer_gb300 import build as libbuild
        mlib = ctypes.CDLL(libbuild.build_mmabench())
        mlib.hla_mmabench_run.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_float)]
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        iters = 4000
        ms_m = ctypes.c_float(0.0)
        rc = mlib.hla_mmabench_run(sms, iters, ctypes.byref(ms_m))
        if rc == 0 and ms_m.value > 0:
            flops = sms * iters * 4 * 2.0 * 128 ** 3
            tf = flops / (ms_m.value / 1e3) / 1e12
            # clock-derived dense rate: 8192 bf16/fp16 FLOP per clock per SM (4096 FMA) at the
            # maximum SM clock; the measured cuBLAS figure ran power-capped at a lower clock
            clock_mhz = float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))).get(
                "sm_max_mhz", 2070.0)) if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) else 2070.0
            clock_peak = sms * 8192 * clock_mhz * 1e6 / 1e12
            out["mma_rate"] = {"what": "MMA1-MMA4 of the output pass, 128x128x128 each, operands "
                                       "in shared memory, one CTA per SM",
                               "achieved": tf, "peak": tc_peak, "unit": "TFLOP/s",
                               "frac": tf / tc_peak, "peak_source": f"bf16_tflops of {peak_src}",
                               "clock_peak": clock_peak, "frac_clock_peak": tf / clock_peak,
                               "ms": ms_m.value}
        launches += 1

    # ---------------------------------------------------------------- CPU oracle
    cpu = None
    if D.rank == 0 and not args.no_cpu_baseline:
        tok_s, n, cores, dt = oracle_sample(w, args.cpu_seconds)
        tok_1, n_1, _, dt_1 = oracle_sample(w, max(1.0, args.cpu_seconds / 4), threads=1)
        cpu = {"value": tok_s / 1e6, "unit": "Mtok/s", "cores": cores, "kind": "oracle",
               "sample": f"first {n} tokens of sequence 0 of the 512K workload, all {w.H} heads, "
                         f"fp64, {dt:.1f} s",
               "value_1core": tok_1 / 1e6,
               "sample_1core": f"first {n_1} tokens, all {w.H} heads, one thread, {dt_1:.1f} s",
               "cpu_model": host_cpu_model()}

    if D.rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "Mtok/s", "n_gpus": D.world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic", "config": config, "roofline": roof, "cpu_baseline": cpu,
                "e2e": e2e, "gpu_launches": launches, "clocks": clk.summary()}
        line.update(out)
        print(json.dumps(line))
    if D.pg:
        D.pg.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
