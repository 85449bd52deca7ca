#!/usr/bin/env python
"""Benchmark of the decoder block: prefill tokens/s with attention and GEMM
TFLOP/s, and decode KV-cache GB/s, on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl tb|reference]

One step is one full prefill of the block (RMSNorm, QKV + RoPE, causal GQA
attention, Wo + residual, RMSNorm, SwiGLU, W2 + residual) over one batch of the
prefill workload (default gqa_8k: B=4, T=8192, d=4096, H=32, Hkv=8, dh=128,
f=14336).  The decode workload (gqa_decode: 32 sequences, cache lengths
uniform in [1024, 16383]) is timed after it and reported under "decode".

Inputs are seeded synthetic tensors resident in HBM before timing; each one is
larger than L2 (x 268 MB, weights 436 MB, decode KV 1.1 GB), so no L2 flush is
needed between steps.  Device time comes from CUDA events on the launching
stream; per-kernel times from the library's stage trace (events recorded
between launches on the same stream).  Under torchrun every rank runs its own
replica (the block has no exchange step) and the slowest rank's time counts.

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload on the host cores (the only reference that exists for this path).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Token count up to which each bf16 GEMM runs as the few-token GEMM (one
# launch each, its K split reduced inside a cluster).
FEW_TOKENS = 64


# The headline metric, the same string on both arms.
METRIC = "prefill tokens/s per block (attention TFLOP/s, GEMM TFLOP/s; decode KV GB/s)"


def decode_launches(B: int) -> int:
    """Kernels one bf16 decode step launches: the two attention kernels and
    the four GEMMs (the few-token GEMM, whose QKV instance also forms the row
    statistics, when the batch takes it; above that, the tile GEMMs and the
    row-statistics kernel)."""
    return 2 + 4 if B <= FEW_TOKENS else 3 + 4


def prefill_launches(tokens: int) -> int:
    """Kernels one bf16 prefill launches: the four GEMMs and the attention (the
    tile QKV GEMM forms the row statistics); with few tokens the
    row-statistics kernel runs first."""
    return 5 if tokens > FEW_TOKENS else 6


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 25 ms while running;
    samples drawing at least half the peak power count as under load."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "25"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")
        sm = [num(r[1]) for r in rows]
        mx = max(num(r[2]) for r in rows)
        power = [num(r[3]) for r in rows]
        pmax = max(power)
        loaded = [c for c, p in zip(sm, power) if p >= 0.5 * pmax] or sm
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(rows), "samples_under_load": len(loaded), "power_w_max": pmax}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The slowest rank's time: every rank contributes x, all get the maximum."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(world: int, units_per_rank_step: int, steps: int, ms_total_max: float) -> float:
    """Whole-job throughput of weak-scaled replicas: every rank processes the
    same units per step; the slowest rank's time bounds the job."""
    return world * units_per_rank_step * steps / (ms_total_max * 1e-3)


# ---------------------------------------------------------------------------
# CPU oracle timing (the reference arm and the cpu_baseline field)
# ---------------------------------------------------------------------------

def time_oracle_prefill(s, tokens: int, seed: int = 0):
    """The fp64 oracle on the first `tokens` tokens of sequence 0 of the
    workload (a causal prefix is a complete prefill of its own).  Returns
    (seconds, tokens)."""
    import oracle
    import workloads
    inp = workloads.make_block_inputs(s.with_(B=1), seed=seed, x_tokens=tokens)
    w = {n: workloads.to_f64(inp[n]) for n in workloads.WEIGHT_NAMES}
    cfg = oracle.Cfg(s.d, s.H, s.Hkv, s.dh, s.f, s.rope_base, s.eps)
    x = workloads.to_f64(inp["x"][0])
    t0 = time.perf_counter()
    oracle.block_prefill_seq(x, w, cfg)
    return time.perf_counter() - t0, tokens


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args, world, rank):
    import workloads
    if rank != 0:
        return
    s = workloads.CONFIGS[args.workload]
    tokens = args.ref_tokens
    times = []
    for i in range(args.warmup + args.steps):
        dt, _ = time_oracle_prefill(s, tokens)
        if i >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = tokens * len(times) / total
    sample = f"fp64 oracle prefill of the first {tokens} tokens of one sequence of {s.name}, per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(s),
        "cpu_baseline": {"value": value, "unit": "tok/s", "cores": cpu_cores(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


L2_BYTES = 129 << 20     # GB300 L2


def workload_config(s):
    from causal_gqa_attention_rmsnorm_gb300 import accounting as acc
    esz = 4 if s.dtype == "f32" else 2
    step_bytes = s.B * s.T * s.d * esz + acc.weight_bytes(s.d, s.H, s.Hkv, s.dh, s.f, esz)
    l2 = ("inputs larger than L2 (no flush)" if step_bytes > L2_BYTES
          else "inputs smaller than L2, not flushed: a parity workload, not a bench line")
    return {"workload": s.name, "B": s.B, "T": s.T, "d": s.d, "H": s.H, "Hkv": s.Hkv, "dh": s.dh, "f": s.f,
            "rope_base": s.rope_base, "eps": s.eps, "storage": s.dtype, "accumulate": "f32",
            "l2": l2, "parallelism": "replicas"}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def stage_stats(traces):
    """Mean ms of each stage over the traced calls."""
    acc = {}
    for tr in traces:
        for name, ms in tr:
            acc.setdefault(name, []).append(ms)
    return {k: sum(v) / len(v) for k, v in acc.items()}


def prefill_stage_work(s):
    from causal_gqa_attention_rmsnorm_gb300 import accounting as acc
    M = s.B * s.T
    g = acc.gemm_flops_each(s.d, s.H, s.Hkv, s.dh, s.f, M)
    return {
        "qkv": ("tensor", g["qkv"]), "attn": ("tensor", acc.causal_attn_flops(s.B, s.H, s.dh, s.T)),
        "wo": ("tensor", g["wo"]), "w13": ("tensor", g["w13"]), "w2": ("tensor", g["w2"]),
        "rms": ("hbm", M * s.d * 2 + M * 8),
    }


def bench_prefill(args, s, world, peaks):
    import torch
    import causal_gqa_attention_rmsnorm_gb300 as tb
    from causal_gqa_attention_rmsnorm_gb300 import binding
    import workloads

    inp = workloads.make_block_inputs(s, seed=0)
    dev = {n: t.cuda() for n, t in inp.items()}
    cfg = tb.BlockConfig(s.d, s.H, s.Hkv, s.dh, s.f, s.T, s.rope_base, s.eps, tb.TB_BF16)
    packed = tb.tb_pack_weights(cfg, dev)
    x = dev["x"]
    y = torch.empty((s.B, s.T, s.d), dtype=torch.float32, device="cuda")
    ws = torch.empty(tb.tb_workspace_bytes(cfg, s.B, s.T, 0), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        tb.tb_block_prefill(cfg, packed, x, y=y, ws=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert tb.tb_get_device_error(clear=True) == 0

    binding.tbx_trace_enable(args.steps)
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms_total = e0.elapsed_time(e1)
    clk = clocks.stop()
    traces = [binding.tbx_trace_read(i) for i in range(args.steps)]
    binding.tbx_trace_enable(0)
    assert tb.tb_get_device_error(clear=True) == 0
    assert torch.isfinite(y).all().item()
    ms_total = max_over_ranks(ms_total, world)
    stages = stage_stats(traces)

    # end to end through the public call with host buffers: every step copies its
    # x in from pinned host memory and its y back out.  Steps are pipelined the
    # way a serving loop runs them: two device buffers each for x and y and one
    # copy stream, on which step i+1's input copy is queued ahead of step i's
    # output copy, so both overlap the computation of a neighbouring step, and
    # events order every buffer's reuse.  One copy stream keeps the two
    # directions from running at once: on some hosts concurrent copies in and
    # out slowed the computation by about 15 %, while either alone cost little.
    e2e = None
    if not args.no_e2e:
        xh = inp["x"].pin_memory()
        yhs = [torch.empty((s.B, s.T, s.d), dtype=torch.float32).pin_memory() for _ in range(2)]
        xs, ys = [x, torch.empty_like(x)], [y, torch.empty_like(y)]
        cs = torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(2)]      # x buffer filled
        ev_done = [torch.cuda.Event() for _ in range(2)]    # step finished: x buffer free, y buffer ready
        ev_out = [torch.cuda.Event() for _ in range(2)]     # y buffer copied out: free

        def pipelined(n, start):
            cs.wait_event(start)
            with torch.cuda.stream(cs):
                xs[0].copy_(xh, non_blocking=True)
                ev_in[0].record(cs)
            for i in range(n):
                j = i % 2
                stream.wait_event(ev_in[j])
                if i >= 2:
                    stream.wait_event(ev_out[j])
                tb.tb_block_prefill(cfg, packed, xs[j], y=ys[j], ws=ws)
                ev_done[j].record(stream)
                with torch.cuda.stream(cs):
                    if i + 1 < n:
                        jn = (i + 1) % 2
                        if i >= 1:
                            cs.wait_event(ev_done[jn])       # step i-1 is done with that x buffer
                        xs[jn].copy_(xh, non_blocking=True)
                        ev_in[jn].record(cs)
                    cs.wait_event(ev_done[j])
                    yhs[j].copy_(ys[j], non_blocking=True)
                    ev_out[j].record(cs)
            stream.wait_stream(cs)

        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        pipelined(3, a)
        torch.cuda.synchronize()
        barrier(world)
        a.record(stream)
        pipelined(args.steps, a)
        b.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        assert tb.tb_get_device_error(clear=True) == 0
        assert torch.isfinite(yhs[(args.steps - 1) % 2]).all().item()
        e2e_ms = max_over_ranks(a.elapsed_time(b), world)
        e2e = {"value": world * s.B * s.T * args.steps / (e2e_ms * 1e-3), "unit": "tok/s",
               "h2d_bytes_per_step": xh.numel() * xh.element_size(),
               "d2h_bytes_per_step": yhs[0].numel() * yhs[0].element_size(), "ms_per_step": e2e_ms / args.steps,
               "pipelined": "x in and y out on one copy stream, overlapping neighbouring steps' compute"}
        del xs, ys
    del ws
    return {"ms_total": ms_total, "stages": stages, "clocks": clk, "e2e": e2e,
            "launches_per_step": prefill_launches(s.B * s.T)}


# DRAM read + write of one launch of the stage's kernel, from a one-pass ncu
# capture (dram__bytes_read.sum + dram__bytes_write.sum) of the benchmark's own
# launches: the mean of the two timed W1/W3 launches in
# profiles/prefill_gqa_8k_launches.md.  The reads vary from box to box
# (profiles/gemm_w13_gqa_8k.md).
NCU_TRAFFIC = {("gqa_8k", "w13"): (4454309888 + 4500537856 + 927719936 + 928212736) / 2}


def roofline_entry(stages, work, peaks, peak_src, workload):
    """The longest stage of the step against its roofline: algorithmic FLOPs
    (or bytes) per launch over the live mean launch time, against the measured
    burst bf16 peak or the HBM copy bandwidth.  The default 50-step run lasts
    about half a second and reaches the power cap, so a tensor-bound stage also
    carries its fraction of the measured sustained peak."""
    name = max(stages, key=lambda k: stages[k])
    bound, amount = work[name]
    ms = stages[name]
    if bound == "tensor":
        achieved = amount / (ms * 1e-3) / 1e12
        peak = peaks["bf16_tflops"]
        unit = "TFLOP/s"
        extra = {"frac_of_sustained": achieved / peaks["bf16_tflops_sustained"]}
    else:
        achieved = amount / (ms * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        unit = "GB/s"
        extra = {}
    out = {"kernel": name, "bound": "tensor" if bound == "tensor" else "hbm", "achieved": achieved, "peak": peak,
           "unit": unit, "frac": achieved / peak, "traffic": NCU_TRAFFIC.get((workload, name)), "ms": ms,
           "algorithmic": amount,
           "peak_source": f"{peak_src} ({'bf16 burst' if bound == 'tensor' else 'hbm copy'})"}
    out.update(extra)
    return out


def decode_shape(args):
    """The decode workload, with B overridden by --decode-batch (profiling runs)."""
    import workloads
    s = workloads.CONFIGS[args.decode_workload]
    return s.with_(name=f"{s.name}_b{args.decode_batch}", B=args.decode_batch) if args.decode_batch else s


def bench_decode(args, world, peaks):
    import torch
    import causal_gqa_attention_rmsnorm_gb300 as tb
    from causal_gqa_attention_rmsnorm_gb300 import accounting as acc
    from causal_gqa_attention_rmsnorm_gb300 import binding
    import workloads

    s = decode_shape(args)
    inp = workloads.make_block_inputs(s, seed=0)
    dev = {n: t.cuda() for n, t in inp.items()}
    lens = workloads.make_lens(s, seed=0)
    kc, vc = workloads.make_decode_cache(s, 0, lens, fill=0.0, device="cuda")
    lens0 = lens.cuda()
    kv = tb.KVCache(kc, vc, lens0.clone())
    cfg = tb.BlockConfig(s.d, s.H, s.Hkv, s.dh, s.f, s.T, s.rope_base, s.eps, tb.TB_BF16)
    packed = tb.tb_pack_weights(cfg, dev)
    y = torch.empty((s.B, 1, s.d), dtype=torch.float32, device="cuda")
    ws = torch.empty(tb.tb_workspace_bytes(cfg, s.B, s.T, 1), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        kv.lens.copy_(lens0, non_blocking=True)      # every step decodes at the same positions
        tb.tb_block_decode(cfg, packed, dev["x"], kv, y=y, ws=ws)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    assert tb.tb_get_device_error(clear=True) == 0
    n = max(args.steps, 20)
    binding.tbx_trace_enable(n)
    barrier(world)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(n):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b), world) / n
    stages = stage_stats([binding.tbx_trace_read(i) for i in range(n)])
    binding.tbx_trace_enable(0)
    assert torch.isfinite(y).all().item()
    # the same step captured once as a CUDA graph and replayed (no per-launch host work)
    graph_ms = None
    if not args.no_graph:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()                                    # warm the capture stream
        stream.wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            step()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        barrier(world)
        a.record(stream)
        for _ in range(n):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        graph_ms = max_over_ranks(a.elapsed_time(b), world) / n
        assert torch.isfinite(y).all().item()
    kv_bytes = acc.decode_kv_bytes(lens.tolist(), s.Hkv, s.dh, 2)
    w_bytes = acc.weight_bytes(s.d, s.H, s.Hkv, s.dh, s.f, 2)
    attn_ms = stages["attn"]
    kv_gbs = kv_bytes / (attn_ms * 1e-3) / 1e9
    return {
        "workload": s.name, "B": s.B, "T_max": s.T, "kv_bytes": kv_bytes, "weight_bytes": w_bytes,
        "kv_gbs": kv_gbs, "kv_frac_hbm": kv_gbs / peaks["hbm_gbs"], "attn_ms": attn_ms, "step_ms": ms,
        "tok_s": world * s.B / (ms * 1e-3), "stages_ms": stages, "gpu_launches": decode_launches(s.B) * n,
        "graph_step_ms": graph_ms,
        "graph_tok_s": None if graph_ms is None else world * s.B / (graph_ms * 1e-3),
        "step_hbm_gbs": (kv_bytes + w_bytes) / (ms * 1e-3) / 1e9,
    }


def bench_window(args, world, peaks):
    """The sliding-window path at W = args.window: one prefill of the benchmark
    workload and one decode step of the decode workload, each timed over
    args.steps live steps, with the windowed pair and byte counts."""
    import torch
    import causal_gqa_attention_rmsnorm_gb300 as tb
    from causal_gqa_attention_rmsnorm_gb300 import accounting as acc
    from causal_gqa_attention_rmsnorm_gb300 import binding
    import workloads

    W = args.window
    n = max(args.steps, 5)

    def timed(step):
        for _ in range(max(args.warmup, 3)):
            step()
        torch.cuda.synchronize()
        assert tb.tb_get_device_error(clear=True) == 0
        binding.tbx_trace_enable(n)
        barrier(world)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(n):
            step()
        b.record()
        torch.cuda.synchronize()
        stages = stage_stats([binding.tbx_trace_read(i) for i in range(n)])
        binding.tbx_trace_enable(0)
        assert tb.tb_get_device_error(clear=True) == 0
        return max_over_ranks(a.elapsed_time(b), world) / n, stages

    s = workloads.CONFIGS[args.workload]
    if args.batch:
        s = s.with_(B=args.batch)
    s = s.with_(window=W)
    inp = workloads.make_block_inputs(s, seed=0)
    dev = {k: t.cuda() for k, t in inp.items()}
    cfg = tb.BlockConfig(s.d, s.H, s.Hkv, s.dh, s.f, s.T, s.rope_base, s.eps, tb.TB_BF16, W)
    packed = tb.tb_pack_weights(cfg, dev)
    y = torch.empty((s.B, s.T, s.d), dtype=torch.float32, device="cuda")
    ws = torch.empty(tb.tb_workspace_bytes(cfg, s.B, s.T, 0), dtype=torch.uint8, device="cuda")
    ms, st = timed(lambda: tb.tb_block_prefill(cfg, packed, dev["x"], y=y, ws=ws))
    assert torch.isfinite(y).all().item()
    fl = acc.causal_attn_flops(s.B, s.H, s.dh, s.T, W)
    pre_tokens = s.B * s.T
    pre = {"workload": s.name, "ms_per_step": ms, "tok_s": world * s.B * s.T / (ms * 1e-3),
           "attn_ms": st["attn"], "attn_flops": fl, "attn_tflops": fl / (st["attn"] * 1e-3) / 1e12,
           "attn_frac_bf16": fl / (st["attn"] * 1e-3) / 1e12 / peaks["bf16_tflops"]}
    del dev, packed, y, ws

    s = workloads.CONFIGS[args.decode_workload].with_(window=W)
    inp = workloads.make_block_inputs(s, seed=0)
    dev = {k: t.cuda() for k, t in inp.items()}
    lens = workloads.make_lens(s, seed=0)
    kc, vc = workloads.make_decode_cache(s, 0, lens, fill=0.0, device="cuda")
    lens0 = lens.cuda()
    kv = tb.KVCache(kc, vc, lens0.clone())
    cfg = tb.BlockConfig(s.d, s.H, s.Hkv, s.dh, s.f, s.T, s.rope_base, s.eps, tb.TB_BF16, W)
    packed = tb.tb_pack_weights(cfg, dev)
    y = torch.empty((s.B, 1, s.d), dtype=torch.float32, device="cuda")
    ws = torch.empty(tb.tb_workspace_bytes(cfg, s.B, s.T, 1), dtype=torch.uint8, device="cuda")

    def dstep():
        kv.lens.copy_(lens0, non_blocking=True)
        tb.tb_block_decode(cfg, packed, dev["x"], kv, y=y, ws=ws)
    ms, st = timed(dstep)
    assert torch.isfinite(y).all().item()
    kv_bytes = acc.decode_kv_bytes(lens.tolist(), s.Hkv, s.dh, 2, W)
    dec = {"workload": s.name, "step_ms": ms, "tok_s": world * s.B / (ms * 1e-3), "attn_ms": st["attn"],
           "kv_bytes": kv_bytes, "kv_gbs": kv_bytes / (st["attn"] * 1e-3) / 1e9,
           "kv_frac_hbm": kv_bytes / (st["attn"] * 1e-3) / 1e9 / peaks["hbm_gbs"]}
    return {"window": W, "prefill": pre, "decode": dec,
            "gpu_launches": (prefill_launches(pre_tokens) + decode_launches(s.B)) * n}


def bench_paged(args, world, peaks):
    """A decode step of the decode workload through a paged cache: pages of
    args.page_size rows, the pool shuffled (sequence b's pages scattered over
    the pool by a seeded permutation), timed over args.steps eager steps."""
    import numpy as np
    import torch
    import causal_gqa_attention_rmsnorm_gb300 as tb
    from causal_gqa_attention_rmsnorm_gb300 import accounting as acc
    from causal_gqa_attention_rmsnorm_gb300 import binding
    import workloads

    ps = args.page_size
    s = workloads.CONFIGS[args.decode_workload]
    inp = workloads.make_block_inputs(s, seed=0)
    dev = {k: t.cuda() for k, t in inp.items()}
    lens = workloads.make_lens(s, seed=0)
    kc, vc = workloads.make_decode_cache(s, 0, lens, fill=0.0, device="cuda")
    per = s.T // ps
    num_pages = s.B * per
    perm = torch.tensor(np.random.default_rng(0).permutation(num_pages).reshape(s.B, per), dtype=torch.int32)
    kv = tb.KVCache.empty_paged(s.B, s.Hkv, s.T, s.dh, ps, num_pages, perm.cuda())
    for b in range(s.B):                             # the same rows, scattered into the pool
        kv.k[perm[b].long().cuda()] = kc[b].reshape(s.Hkv, per, ps, s.dh).transpose(0, 1)
        kv.v[perm[b].long().cuda()] = vc[b].reshape(s.Hkv, per, ps, s.dh).transpose(0, 1)
    del kc, vc
    lens0 = lens.cuda()
    cfg = tb.BlockConfig(s.d, s.H, s.Hkv, s.dh, s.f, s.T, s.rope_base, s.eps, tb.TB_BF16)
    packed = tb.tb_pack_weights(cfg, dev)
    y = torch.empty((s.B, 1, s.d), dtype=torch.float32, device="cuda")
    ws = torch.empty(tb.tb_workspace_bytes(cfg, s.B, s.T, 1), dtype=torch.uint8, device="cuda")

    def step():
        kv.lens.copy_(lens0, non_blocking=True)
        tb.tb_block_decode(cfg, packed, dev["x"], kv, y=y, ws=ws)
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    assert tb.tb_get_device_error(clear=True) == 0
    n = max(args.steps, 20)
    binding.tbx_trace_enable(n)
    barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(n):
        step()
    b.record()
    torch.cuda.synchronize()
    stages = stage_stats([binding.tbx_trace_read(i) for i in range(n)])
    binding.tbx_trace_enable(0)
    assert tb.tb_get_device_error(clear=True) == 0 and torch.isfinite(y).all().item()
    ms = max_over_ranks(a.elapsed_time(b), world) / n
    kv_bytes = acc.decode_kv_bytes(lens.tolist(), s.Hkv, s.dh, 2)
    return {"workload": s.name, "page_size": ps, "num_pages": num_pages, "step_ms": ms,
            "tok_s": world * s.B / (ms * 1e-3), "attn_ms": stages["attn"], "kv_bytes": kv_bytes,
            "kv_gbs": kv_bytes / (stages["attn"] * 1e-3) / 1e9,
            "kv_frac_hbm": kv_bytes / (stages["attn"] * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "gpu_launches": decode_launches(s.B) * n}


def bench_int8(args, world, peaks):
    """A decode step of the decode workload over an int8 cache: the same rows
    as the bf16 decode line, quantised into the cache through the C ABI's
    append, timed over args.steps eager steps and as a replayed CUDA graph."""
    import torch
    import causal_gqa_attention_rmsnorm_gb300 as tb
    from causal_gqa_attention_rmsnorm_gb300 import accounting as acc
    from causal_gqa_attention_rmsnorm_gb300 import binding
    import workloads

    s = decode_shape(args)
    inp = workloads.make_block_inputs(s, seed=0)
    dev = {k: t.cuda() for k, t in inp.items()}
    lens = workloads.make_lens(s, seed=0)
    kc, vc = workloads.make_decode_cache(s, 0, lens, fill=0.0, device="cuda")
    kv = tb.KVCache.empty_int8(s.B, s.Hkv, s.T, s.dh)
    tb.tb_kvcache_append(kv, kc, vc)                 # quantise every row of the bf16 cache
    del kc, vc
    lens0 = lens.cuda()
    cfg = tb.BlockConfig(s.d, s.H, s.Hkv, s.dh, s.f, s.T, s.rope_base, s.eps, tb.TB_BF16)
    packed = tb.tb_pack_weights(cfg, dev)
    y = torch.empty((s.B, 1, s.d), dtype=torch.float32, device="cuda")
    ws = torch.empty(tb.tb_workspace_bytes(cfg, s.B, s.T, 1), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        kv.lens.copy_(lens0, non_blocking=True)
        tb.tb_block_decode(cfg, packed, dev["x"], kv, y=y, ws=ws)
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    assert tb.tb_get_device_error(clear=True) == 0
    n = max(args.steps, 20)
    binding.tbx_trace_enable(n)
    barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(n):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    stages = stage_stats([binding.tbx_trace_read(i) for i in range(n)])
    binding.tbx_trace_enable(0)
    assert tb.tb_get_device_error(clear=True) == 0 and torch.isfinite(y).all().item()
    ms = max_over_ranks(a.elapsed_time(b), world) / n
    graph_ms = None
    if not args.no_graph:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            step()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        barrier(world)
        a.record(stream)
        for _ in range(n):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        graph_ms = max_over_ranks(a.elapsed_time(b), world) / n
        assert torch.isfinite(y).all().item()
    kv_bytes = acc.decode_kv_bytes(lens.tolist(), s.Hkv, s.dh, 1, scale_bytes=4)
    return {"workload": s.name, "step_ms": ms, "tok_s": world * s.B / (ms * 1e-3), "attn_ms": stages["attn"],
            "quant_ms": stages["quant"], "kv_bytes": kv_bytes, "kv_gbs": kv_bytes / (stages["attn"] * 1e-3) / 1e9,
            "kv_frac_hbm": kv_bytes / (stages["attn"] * 1e-3) / 1e9 / peaks["hbm_gbs"], "stages_ms": stages,
            "graph_step_ms": graph_ms,
            "graph_tok_s": None if graph_ms is None else world * s.B / (graph_ms * 1e-3),
            "gpu_launches": (decode_launches(s.B) + 1) * n}


def bench_stack(args, world, peaks):
    """An args.stack_layers-layer model of the prefill workload's block shape:
    the embedding gather, the stack, and the LM head's chunked per-token loss
    over every token (vocabulary args.vocab, head tied to the embedding); then
    one decode step through the same stack for the decode workload."""
    import torch
    import causal_gqa_attention_rmsnorm_gb300 as tb
    from causal_gqa_attention_rmsnorm_gb300 import accounting as acc
    import workloads

    L, V = args.stack_layers, args.vocab
    s = workloads.CONFIGS[args.workload]
    if args.batch:
        s = s.with_(B=args.batch)
    n = max(min(args.steps, 5), 2)
    sd = workloads.CONFIGS[args.decode_workload]
    cfg = tb.BlockConfig(s.d, s.H, s.Hkv, s.dh, s.f, max(s.T, sd.T), s.rope_base, s.eps, tb.TB_BF16)
    packed = []
    for l in range(L):
        w = {k: t.cuda() for k, t in workloads.make_block_inputs(s.with_(B=1, T=1), seed=100 + l).items()}
        packed.append(tb.tb_pack_weights(cfg, w))
        del w
    g = torch.Generator().manual_seed(7)
    table = (0.02 * torch.randn(V, s.d, generator=g)).to(torch.bfloat16).cuda()
    gain = (1 + 0.1 * torch.randn(s.d, generator=g)).to(torch.bfloat16).cuda()
    hcfg = tb.HeadConfig(s.d, V, s.eps, tb.TB_BF16)
    head = tb.tb_pack_lm_head(hcfg, gain, table, tied=True)
    ids = torch.randint(0, V, (s.B, s.T), generator=g, dtype=torch.int32).cuda()
    targets = torch.roll(ids, -1, dims=1).reshape(-1).contiguous()
    x = torch.empty((s.B, s.T, s.d), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((s.B, s.T, s.d), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(tb.binding.lib().tb_stack_workspace_bytes(ctypes_cfg(cfg), s.B, s.T, 0), dtype=torch.uint8,
                     device="cuda")
    hws = torch.empty(tb.binding.lib().tb_lm_head_workspace_bytes(ctypes_cfg(hcfg), 4096), dtype=torch.uint8,
                      device="cuda")
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]

    def step(record):
        if record:
            ev[0].record()
        tb.tb_embed(table, ids, x=x)
        y2 = tb.tb_stack_prefill(cfg, packed, x, y_dtype=tb.TB_BF16, ws=ws)
        if record:
            ev[1].record()
        _, nll = tb.tb_lm_head(hcfg, head, y2.reshape(-1, s.d), want_logits=False, targets=targets, row_chunk=4096,
                               ws=hws)
        if record:
            ev[2].record()
        return nll
    for _ in range(2):
        step(False)
    torch.cuda.synchronize()
    assert tb.tb_get_device_error(clear=True) == 0
    t_stack = t_head = 0.0
    for _ in range(n):
        nll = step(True)
        torch.cuda.synchronize()
        t_stack += ev[0].elapsed_time(ev[1])
        t_head += ev[1].elapsed_time(ev[2])
    assert tb.tb_get_device_error(clear=True) == 0 and torch.isfinite(nll).all().item()
    t_stack, t_head = t_stack / n, t_head / n
    tokens = s.B * s.T
    head_fl = acc.lm_head_flops(tokens, s.d, V)
    pre = {"workload": s.name, "layers": L, "vocab": V, "tokens": tokens, "stack_ms": t_stack,
           "stack_tok_s": world * tokens / (t_stack * 1e-3), "head_ms": t_head,
           "head_tflops": head_fl / (t_head * 1e-3) / 1e12, "head_frac_bf16": head_fl / (t_head * 1e-3) / 1e12 / peaks["bf16_tflops"],
           "model_tok_s": world * tokens / ((t_stack + t_head) * 1e-3), "mean_nll": float(nll.mean())}
    del x, y, ws, hws

    lens = workloads.make_lens(sd, seed=0)
    kvs = []
    for l in range(L):
        kc, vc = workloads.make_decode_cache(sd, l, lens, fill=0.0, device="cuda")
        kvs.append(tb.KVCache(kc, vc, lens.cuda()))
    lens0 = lens.cuda()
    ids1 = torch.randint(0, V, (sd.B, 1), generator=g, dtype=torch.int32).cuda()
    x1 = torch.empty((sd.B, 1, sd.d), dtype=torch.bfloat16, device="cuda")
    dws = torch.empty(tb.binding.lib().tb_stack_workspace_bytes(ctypes_cfg(cfg), sd.B, sd.T, 1), dtype=torch.uint8,
                      device="cuda")

    def dstep():
        for kv in kvs:
            kv.lens.copy_(lens0, non_blocking=True)
        tb.tb_embed(table, ids1, x=x1)
        h = tb.tb_stack_decode(cfg, packed, x1, kvs, y_dtype=tb.TB_BF16, ws=dws)
        return tb.tb_lm_head(hcfg, head, h.reshape(-1, sd.d))[0]
    for _ in range(3):
        dstep()
    torch.cuda.synchronize()
    m = max(args.steps, 10)
    ev[0].record()
    for _ in range(m):
        lg = dstep()
    ev[1].record()
    torch.cuda.synchronize()
    assert tb.tb_get_device_error(clear=True) == 0 and torch.isfinite(lg).all().item()
    dms = ev[0].elapsed_time(ev[1]) / m
    dec = {"workload": sd.name, "layers": L, "step_ms": dms, "tok_s": world * sd.B / (dms * 1e-3)}
    return {"prefill": pre, "decode": dec,
            "gpu_launches": n * (1 + prefill_launches(tokens) * L + 3 * (tokens + 4095) // 4096)
                            + m * (1 + decode_launches(sd.B) * L + 2)}


def ctypes_cfg(cfg):
    import ctypes
    return ctypes.byref(cfg.c())


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["tb", "reference"], default="tb")
    ap.add_argument("--workload", default="gqa_8k")
    ap.add_argument("--batch", type=int, default=0, help="override B of the prefill workload (profiling runs)")
    ap.add_argument("--decode-workload", default="gqa_decode")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--decode-batch", type=int, default=0, help="override B of the decode lines (profiling runs)")
    ap.add_argument("--no-prefill", action="store_true",
                    help="decode lines only (profiling runs); prints the decode and int8 objects")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay of the decode step")
    ap.add_argument("--window", type=int, default=4096, help="sliding-window width of the extra window line (0: skip)")
    ap.add_argument("--page-size", type=int, default=16, help="page size of the paged-cache decode line (0: skip)")
    ap.add_argument("--no-int8", action="store_true", help="skip the int8-cache decode line")
    ap.add_argument("--stack-layers", type=int, default=4, help="layers of the model line (0: skip)")
    ap.add_argument("--vocab", type=int, default=128256, help="vocabulary of the model line's LM head")
    ap.add_argument("--ref-tokens", type=int, default=512, help="oracle sample size per reference step")
    ap.add_argument("--cpu-tokens", type=int, default=6144, help="oracle sample size for cpu_baseline")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    import torch
    import workloads
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    peaks, peak_src = load_peaks()
    s = workloads.CONFIGS[args.workload]
    if args.batch:
        s = s.with_(name=f"{s.name}_b{args.batch}", B=args.batch)

    if args.no_prefill:
        dec = bench_decode(args, world, peaks)
        i8 = None if args.no_int8 else bench_int8(args, world, peaks)
        if rank == 0:
            print(json.dumps({"decode": dec, "int8_kv": i8}))
        return
    pre = bench_prefill(args, s, world, peaks)
    dec = None if args.no_decode else bench_decode(args, world, peaks)
    win = None if (args.window <= 0 or args.no_decode) else bench_window(args, world, peaks)
    pag = None if (args.page_size <= 0 or args.no_decode) else bench_paged(args, world, peaks)
    i8 = None if (args.no_int8 or args.no_decode) else bench_int8(args, world, peaks)
    stk = None if (args.stack_layers <= 0 or args.no_decode) else bench_stack(args, world, peaks)

    from causal_gqa_attention_rmsnorm_gb300 import accounting as acc
    tokens = s.B * s.T
    ms_step = pre["ms_total"] / args.steps
    value = aggregate_rate(world, tokens, args.steps, pre["ms_total"])
    work = prefill_stage_work(s)
    stages = pre["stages"]
    attn_tflops = work["attn"][1] / (stages["attn"] * 1e-3) / 1e12
    gemm_ms = sum(stages[k] for k in ("qkv", "wo", "w13", "w2"))
    gemm_tflops = sum(work[k][1] for k in ("qkv", "wo", "w13", "w2")) / (gemm_ms * 1e-3) / 1e12
    line = {
        "metric": METRIC,
        "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1) activations, N(0,0.02) weights, N(1,0.1) gains)",
        "config": workload_config(s),
        "attn_tflops": attn_tflops, "attn_frac_bf16": attn_tflops / peaks["bf16_tflops"],
        "attn_tflops_tile_count": acc.causal_attn_flops_tiles(s.B, s.H, s.dh, s.T) / (stages["attn"] * 1e-3) / 1e12,
        "attn_frac_bf16_sustained": attn_tflops / peaks["bf16_tflops_sustained"],
        "gemm_tflops": gemm_tflops, "gemm_frac_bf16": gemm_tflops / peaks["bf16_tflops"],
        "gemm_frac_bf16_sustained": gemm_tflops / peaks["bf16_tflops_sustained"],
        "stages_ms": stages,
        "stage_tflops": {k: work[k][1] / (stages[k] * 1e-3) / 1e12 for k in stages if work.get(k, ("", 0))[0] == "tensor"},
        "roofline": roofline_entry(stages, work, peaks, peak_src, s.name),
        "gpu_launches": pre["launches_per_step"] * args.steps,
        "clocks": pre["clocks"],
        "e2e": pre["e2e"],
        "decode": dec,
        "sliding_window": win,
        "paged_kv": pag,
        "int8_kv": i8,
        "model": stk,
        "peaks": {"source": peak_src, "bf16_tflops": peaks["bf16_tflops"],
                  "bf16_tflops_sustained": peaks["bf16_tflops_sustained"], "hbm_gbs": peaks["hbm_gbs"]},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        dt, n = time_oracle_prefill(s, args.cpu_tokens)
        line["cpu_baseline"] = {
            "value": n / dt, "unit": "tok/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"fp64 oracle prefill of the first {n} tokens of one sequence of {s.name} "
                      f"({dt:.1f} s; a causal prefix has less attention work per token than T={s.T})"}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
