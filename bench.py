#!/usr/bin/env python
"""Decode benchmark of the 33B-shaped bf16 GQA decoder on GB300.

Workload: the full 52-layer Nanbeige4.3-33B-shaped model with random-init bf16
weights (seed 21, ~61.7 GiB), an 8,192-token prompt of uniform-random ids (seed
22) prefilled in 2,048-row chunks, then batch-1 greedy decode: one step = one
decode row through all 52 layers + lm_head + argmax, the next id staying on the
device.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl tfl|reference]

--impl reference times the CPU oracle (the slow float64 reference) on the host
cores for the same metric.  With N > 1 (torchrun) every rank runs an independent
replica (the path has no data-parallel exchange: replicas only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gqa_decoder_forward_gb300 import synth  # noqa: E402

METRIC = "33B bf16 decode tok/s @1 stream + HBM GB/s vs peak; prefill tok/s"
SHAPE = synth.NANBEIGE_33B


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=64)
    p.add_argument("--warmup", type=int, default=8)
    p.add_argument("--impl", choices=["tfl", "reference"], default="tfl")
    p.add_argument("--context", type=int, default=8192)
    p.add_argument("--layers", type=int, default=SHAPE.layers)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--kv", choices=["prefill", "seeded"], default="prefill",
                   help="build the context by prefilling the prompt, or write seeded KV contents")
    p.add_argument("--op", default=None,
                   help="time one decode op (qkv_rope, attention, o_residual, gate_up, down_residual, attn_norm) "
                        "on a one-layer 33B-shaped model instead of the full step")
    p.add_argument("--rows", type=int, default=1, help="rows per step for --op")
    p.add_argument("--concurrent", type=int, default=0,
                   help="time decode steps of this many streams (1 row each, seeded caches of --context "
                        "positions) instead of the default line")
    p.add_argument("--prompt", action="store_true",
                   help="--op runs the prompt-chunk kernel of the op (rows up to 2,048)")
    p.add_argument("--concurrent-streams", type=int, default=16,
                   help="streams of the concurrent figures of the default line (0 = skip them)")
    p.add_argument("--drafted-tokens", type=int, default=64,
                   help="greedy tokens for the drafted-decode figures of the default line (0 = skip them)")
    return p.parse_args()


# ---- environment ---------------------------------------------------------------------

def dist_init(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if (args.impl == "tfl" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ---- algorithmic bytes --------------------------------------------------------------

def layer_weight_bytes(m) -> int:
    return sum(2 * int(torch.tensor(s).prod()) for s in synth.layer_tensor_shapes(m).values())


def step_bytes(m, ctx: int) -> int:
    """Bytes a batch-1 decode step must move: every weight but the embedding
    table (one embedding row), plus the keys and values of ctx positions."""
    w = m.layers * layer_weight_bytes(m) + 2 * m.hidden + m.vocab * m.hidden * 2 + m.hidden * 2
    kv = m.layers * 2 * m.n_kv * m.head_dim * 2 * ctx
    return w + kv


# ---- oracle (CPU) timing ----------------------------------------------------------------

def oracle_sample(context: int, min_seconds: float = 10.0):
    """Times the oracle on one 33B-shaped layer's decode step (one row at position
    `context` over a seeded cache) and on the lm_head of one row; returns
    (seconds per token for the 52-layer model, threads, description)."""
    import numpy as np

    import oracle
    oracle.build()
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    one = SHAPE.with_layers(1)
    w = {k: [synth.layer_weight(one, 21, 0, k, dev)] for k in synth.LAYER_KEYS}
    hw = {k: [synth.bits(w[k][0])] for k in synth.LAYER_KEYS}
    hw["embed"] = np.zeros(8, np.uint16)
    hw["final_norm"] = synth.bits(synth.global_weight(one, 21, "final_norm", dev))
    hw["lm_head"] = synth.bits(synth.global_weight(one, 21, "lm_head", dev))
    del w
    c = oracle.Config(one.hidden, 1, one.n_q, one.n_kv, one.head_dim, one.ffn, one.vocab, one.rope_theta,
                      one.rms_eps)
    om = oracle.Model(c, hw, context + 1)
    K, V = synth.kv_contents(one, 12, 0, context, dev)
    om.K[0, :context] = synth.bits(K)
    om.V[0, :context] = synth.bits(V)
    h = synth.bits(synth.hidden_rows(one, 13, 1, dev))
    pos = np.array([context], np.int32)
    om.layer(0, h, pos)  # warm
    t0 = time.perf_counter()
    reps = 0
    while True:
        out = om.layer(0, h, pos)
        reps += 1
        if time.perf_counter() - t0 >= min_seconds * 0.8:
            break
    t_layer = (time.perf_counter() - t0) / reps
    t1 = time.perf_counter()
    om.head(out)
    t_head = time.perf_counter() - t1
    per_token = SHAPE.layers * t_layer + t_head
    desc = (f"oracle: {reps} reps of one 33B-shaped layer decode step (1 row at position {context}, seeded KV) "
            f"= {t_layer * 1e3:.1f} ms, x{SHAPE.layers} layers + one lm_head row {t_head * 1e3:.0f} ms")
    return per_token, oracle.get_threads(), desc, t_layer, t_head


# ---- the two arms ---------------------------------------------------------------------

def decode_config(args, world):
    """The workload description both arms print (the driver compares them)."""
    return {"workload": f"Nanbeige4.3-33B-shaped decode, {args.layers} layers, 1 stream x 1 row, "
                        f"context {args.context} (+{args.warmup} warm-up)",
            "context_mean": args.context + args.warmup + (args.steps - 1) / 2.0, "rows": 1, "streams": 1,
            "layers": args.layers, "l2": "inputs larger than L2 (61.7 GiB of weights streamed per step)",
            "parallelism": "replicas" if world > 1 else "single GPU"}


def host_ram_gb() -> float:
    """Physical memory of this host, GB."""
    try:
        return os.sysconf("SC_PAGE_SIZE") * os.sysconf("SC_PHYS_PAGES") / 1e9
    except (ValueError, OSError, AttributeError):
        return float("nan")


def oracle_weight_gb(layers: int) -> float:
    """Bytes of bf16 weights a whole oracle model of `layers` layers holds, GB."""
    per_layer = 1_181_773_824
    return (layers * per_layer + 2 * SHAPE.vocab * SHAPE.hidden * 2) / 1e9


def run_reference(args, world, rank):
    """The oracle arm.  A timed step is a bounded sample of the decode step: one
    33B-shaped decoder layer of the oracle (one row at the benchmark's context,
    over a seeded cache), so the run ends in seconds.  --warmup untimed and
    --steps timed samples; ms_per_step is the measured time of one sample, and
    value extrapolates to the whole step: 1 / (layers x mean sample time + the
    time of one lm_head row, measured once outside the timed samples)."""
    if rank != 0:
        return
    import numpy as np

    import oracle
    oracle.build()
    ctx = args.context
    one = SHAPE.with_layers(1)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    w = {k: [synth.layer_weight(one, 21, 0, k, dev)] for k in synth.LAYER_KEYS}
    hw = {k: [synth.bits(w[k][0])] for k in synth.LAYER_KEYS}
    hw["embed"] = np.zeros(8, np.uint16)
    hw["final_norm"] = synth.bits(synth.global_weight(one, 21, "final_norm", dev))
    hw["lm_head"] = synth.bits(synth.global_weight(one, 21, "lm_head", dev))
    del w
    c = oracle.Config(one.hidden, 1, one.n_q, one.n_kv, one.head_dim, one.ffn, one.vocab, one.rope_theta,
                      one.rms_eps)
    om = oracle.Model(c, hw, ctx + 1)
    K, V = synth.kv_contents(one, 12, 0, ctx, dev)
    om.K[0, :ctx] = synth.bits(K)
    om.V[0, :ctx] = synth.bits(V)
    h = synth.bits(synth.hidden_rows(one, 13, 1, dev))
    pos = np.array([ctx], np.int32)
    for _ in range(args.warmup):
        out = om.layer(0, h, pos)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        out = om.layer(0, h, pos)
        times.append(time.perf_counter() - t0)
    t1 = time.perf_counter()
    om.head(out)
    t_head = time.perf_counter() - t1
    t_layer = sum(times) / len(times)
    per_token = args.layers * t_layer + t_head
    value = 1.0 / per_token
    cores = oracle.get_threads()
    desc = (f"oracle, {cores} threads: each timed step is one 33B-shaped decoder layer of the decode step (1 row at "
            f"position {ctx}, seeded KV), {args.steps} timed after {args.warmup} untimed, mean "
            f"{t_layer * 1e3:.1f} ms; value = 1 / ({args.layers} x that + one lm_head row {t_head * 1e3:.0f} ms)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_layer * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (random-init weights, seeded KV)",
        "config": decode_config(args, world),
        "reference_step": (f"one of {args.layers} layers per timed step; value extrapolated to the whole step "
                           f"(a whole {args.layers}-layer oracle step would hold about "
                           f"{oracle_weight_gb(args.layers):.0f} GB of bf16 weights in host memory; this host has "
                           f"{host_ram_gb():.0f} GB; sampled per layer so that the run ends within minutes)"),
        "host_ram_gb": round(host_ram_gb(), 1),
        "cpu_baseline": {"value": value, "unit": "tok/s", "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def ncu_traffic(kernel):
    """DRAM bytes per launch of a kernel family from the committed ncu summary
    (profiles/ncu_traffic.md), or None when its sources changed since the capture."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "ncu_traffic.md")
    if not os.path.exists(path):
        return None
    csrc = os.path.join(ROOT, "gqa_decoder_forward_gb300", "csrc")
    with open(path) as fh:
        for line in fh:
            cells = [c.strip() for c in line.strip().strip("|").split("|")]
            if len(cells) != 5 or cells[0] != kernel:
                continue
            m = hashlib.sha256()
            for f in cells[3].split():
                fp = os.path.join(csrc, f)
                if not os.path.exists(fp):
                    return None
                with open(fp, "rb") as src:
                    m.update(src.read())
            return int(cells[2]) if m.hexdigest()[:16] == cells[4] else None
    return None


def bf16_peak():
    """Dense bf16 tensor peak (TFLOP/s): the measured sustained cuBLAS figure (a
    prefill runs for about a second), else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return float(d["bf16_tflops_sustained"]), "measured (sustained)"
    return 1700.0, "fallback (sustained)"


def prefill_roofline(shape, ctx, prof):
    """Tensor roofline of the dominant prompt GEMM: algorithmic FLOPs (2 x rows x
    K x outputs per launch, over all launches) / its profiled time."""
    if not prof:
        return None
    H, QD, KD, F = shape.hidden, shape.n_q * shape.head_dim, shape.n_kv * shape.head_dim, shape.ffn
    per_row = {"gemm_qkv_rope": H * (QD + 2 * KD), "gemm_o_residual": QD * H,
               "gemm_gate_up_swiglu": 2 * H * F, "gemm_down_residual": F * H}
    best = max(per_row, key=lambda k: prof.get(k, (0.0, 0))[0])
    ms, n = prof[best]
    if not n:
        return None
    flops = 2.0 * ctx * per_row[best] * shape.layers     # every prompt row once per layer
    achieved = flops / (ms / 1e3) / 1e12
    peak, kind = bf16_peak()
    return {"bound": "tensor", "kernel": best, "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4), "peak_kind": kind, "launches": n,
            "ms_per_launch": round(ms / n, 4), "traffic": ncu_traffic(best)}


def run_tfl(args, world, rank, local):
    from gqa_decoder_forward_gb300 import build, tfl
    if rank == 0 or world == 1:
        build.build()
    barrier(world)
    tfl.lib()
    shape = SHAPE.with_layers(args.layers)
    ctx = args.context
    extra = args.warmup + args.steps + 16 + 16 + 18 + 8  # warm-up, timed, profiled, e2e, per-launch steps
    extra = max(extra, args.drafted_tokens + 17)       # the drafted-decode caches hold prompt + reply
    max_ctx = ctx + extra
    dev = torch.device("cuda", torch.cuda.current_device())

    weights = synth.model_weights(shape, 21, dev)
    torch.cuda.synchronize()
    model = tfl.Model(shape, weights, max_rows=2048, max_decode_rows=64, max_context=max_ctx)
    kv = model.kv(max_ctx)
    ids = synth.uniform_ids(22, ctx, shape.vocab, dev)
    st = torch.cuda.current_stream()
    logits = torch.empty((1, shape.vocab), dtype=torch.bfloat16, device=dev)
    nxt = torch.empty(1, dtype=torch.int32, device=dev)

    prefill_s = None
    prefill_prof = {}
    if args.kv == "prefill":
        # prefill (the prompt-chunk path), timed once
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for c in range(0, ctx, 2048):
            model.prefill_chunk(kv, ids[c:c + 2048].contiguous(), logits if c + 2048 >= ctx else None)
        e1.record(st)
        torch.cuda.synchronize()
        prefill_s = e0.elapsed_time(e1) / 1e3
        model.argmax(logits, nxt)
        first_id = int(nxt.item())
        # the same prefill once more on a second cache, every launch bracketed by events
        kv2 = model.kv(max_ctx)
        lg2 = torch.empty_like(logits)
        tfl.tfl_profile(model, True)
        for c in range(0, ctx, 2048):
            model.prefill_chunk(kv2, ids[c:c + 2048].contiguous(), lg2 if c + 2048 >= ctx else None)
        prefill_prof = tfl.tfl_profile_read(model)
        tfl.tfl_profile(model, False)
        del kv2, lg2
    else:
        for l in range(shape.layers):
            K, V = synth.kv_contents(shape, 22, l, ctx, dev)
            kv.write(l, 0, K, V)
        kv.reset(ctx)
        nxt.copy_(ids[-1:])

    def step():
        model.decode_step([kv], nxt, [1], logits)
        model.argmax(logits, nxt)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    ctx0 = kv.length

    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(st)
        for _ in range(args.steps):
            step()
        t1.record(st)
        torch.cuda.synchronize()
    barrier(world)
    ms = max_over_ranks(t0.elapsed_time(t1) / args.steps, world)
    status = model.status()
    mean_ctx = ctx0 + (args.steps - 1) / 2.0

    # per-kernel times (profiled pass: events around every launch)
    prof_steps = min(16, args.steps)
    tfl.tfl_profile(model, True)
    for _ in range(prof_steps):
        step()
    prof = tfl.tfl_profile_read(model)
    try:
        phases = tfl.tfl_step_phases(model)   # the last profiled step, when it ran persistent
    except tfl.TflError:
        phases = None
    tfl.tfl_profile(model, False)
    launches_per_step = sum(n for _, n in prof.values()) / prof_steps

    # the same steps with a launch per operation (the path larger steps take)
    model.set_persistent(False)
    for _ in range(2):
        step()
    torch.cuda.synchronize()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(st)
    for _ in range(prof_steps):
        step()
    a1.record(st)
    torch.cuda.synchronize()
    per_launch_ms = a0.elapsed_time(a1) / prof_steps
    model.set_persistent(True)

    # end to end through the C ABI with host buffers: id in (pinned, H2D), id out (D2H)
    e2e_steps = min(16, args.steps)
    host_in = torch.empty(1, dtype=torch.int32, pin_memory=True)
    host_out = torch.empty(1, dtype=torch.int32, pin_memory=True)
    host_in.copy_(nxt.cpu())
    dev_in = torch.empty(1, dtype=torch.int32, device=dev)
    torch.cuda.synchronize()
    w0 = time.perf_counter()
    for _ in range(e2e_steps):
        dev_in.copy_(host_in, non_blocking=True)
        model.decode_step([kv], dev_in, [1], logits)
        model.argmax(logits, nxt)
        host_out.copy_(nxt, non_blocking=True)
        st.synchronize()
        host_in.copy_(host_out)
    e2e_s = (time.perf_counter() - w0) / e2e_steps
    e2e_s = max_over_ranks(e2e_s, world)

    peak, peak_kind = measured_peaks()
    step_b = step_bytes(shape, int(round(mean_ctx)))
    step_gbs = step_b / (ms / 1e3) / 1e9
    dom = max(prof.items(), key=lambda kv_: kv_[1][0])
    dom_name, (dom_ms, dom_n) = dom
    H, F = shape.hidden, shape.ffn
    dom_bytes = {
        "matvec_gate_up_swiglu": 2 * F * H * 2 + H * 2 + F * 2,
        "matvec_down_residual": H * F * 2 + F * 2 + 2 * H * 2,
        "matvec_qkv_rope": (shape.n_q + 2 * shape.n_kv) * 128 * H * 2 + H * 2,
        "matvec_o_residual": H * H * 2 + 3 * H * 2,
        "matvec_lm_head": shape.vocab * H * 2 + H * 2 + shape.vocab * 2,
        # the whole step in one launch: every weight byte and the visible KV
        "decode_step_persistent": step_b,
    }.get(dom_name)
    roof = None
    if dom_bytes is not None:
        ach = dom_bytes / (dom_ms / dom_n / 1e3) / 1e9
        # the recorded step traffic was captured at context 8,196 on the 52-layer shape
        captured = dom_name != "decode_step_persistent" or (args.layers == SHAPE.layers and ctx == 8192)
        roof = {"bound": "hbm", "kernel": dom_name, "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
                "frac": round(ach / peak, 4), "traffic": ncu_traffic(dom_name) if captured else None,
                "peak_kind": peak_kind,
                "bytes_per_launch": dom_bytes, "us_per_launch": round(dom_ms / dom_n * 1e3, 2)}

    drafted = None
    if args.kv == "prefill" and args.drafted_tokens > 0:
        drafted = drafted_figures(model, kv, ids, first_id, ctx, args.drafted_tokens, dev)

    conc = None
    if args.concurrent_streams > 0 and args.kv == "prefill":
        conc = default_concurrent(model, shape, args.concurrent_streams, ctx, dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        per_tok, cores, desc, _, _ = oracle_sample(ctx, min_seconds=10.0)
        cpu = {"value": 1.0 / per_tok, "unit": "tok/s", "cores": cores, "kind": "oracle", "sample": desc}

    value = world * 1e3 / ms
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (random-init weights, uniform-random ids)",
        "config": decode_config(args, world),
        "step_hbm": {"bytes": step_b, "achieved_gbs": round(step_gbs, 1), "peak_gbs": peak,
                     "frac": round(step_gbs / peak, 4), "peak_kind": peak_kind},
        "roofline": roof,
        "prefill": ({"tokens": ctx, "seconds": round(prefill_s, 4), "tok_s": round(ctx / prefill_s, 1),
                     "path": "prompt chunks of 2,048 rows",
                     "roofline": prefill_roofline(shape, ctx, prefill_prof),
                     "kernels": {k: {"ms": round(v[0], 3), "launches": v[1]}
                                 for k, v in prefill_prof.items() if v[1]}} if prefill_s else None),
        "kv": args.kv,
        "kernels": {k: {"ms_per_step": round(v[0] / prof_steps, 4), "launches_per_step": v[1] / prof_steps}
                    for k, v in prof.items() if v[1]},
        "per_launch_path_ms_per_step": round(per_launch_ms, 4),
        "step_phases_us": phases,
        "gpu_launches": int(round(launches_per_step * args.steps)),
        "e2e": {"value": round(world / e2e_s, 3), "unit": "tok/s", "h2d_bytes_per_step": 4,
                "d2h_bytes_per_step": 4},
        "clocks": clk.summary(),
        "status": status,
        "drafted": drafted,
        "concurrent": conc,
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def default_concurrent(model, shape, S, ctx, dev):
    """The concurrent configuration of S streams at ctx tokens each: every stream
    prefills its own uniform-random prompt (seed 41 + s) in 2,048-row chunks,
    then decode steps of all S streams (one row each) are timed and checked
    equal to each stream alone."""
    cap = ctx + 3 + 16 + 1 + 4 + 4
    kvs = [model.kv(cap) for _ in range(S)]
    first = torch.empty(S, dtype=torch.int32, device=dev)
    last = torch.empty((1, shape.vocab), dtype=torch.bfloat16, device=dev)
    for s in range(S):
        p = synth.uniform_ids(41 + s, ctx, shape.vocab, dev)
        for c in range(0, ctx, 2048):
            model.prefill_chunk(kvs[s], p[c:c + 2048].contiguous(), last if c + 2048 >= ctx else None)
        model.argmax(last, first[s:s + 1])
    res = concurrent_figures(model, kvs, first, 16, 3)
    res["workload"] = f"{S} streams x 1 row, each after its own {ctx}-token uniform-random prompt (seeds 41..)"
    del kvs
    torch.cuda.empty_cache()
    return res


DRAFTER_LAYERS = 4


def drafted_figures(model, kv, ids, first_id, ctx, n, dev):
    """Drafted greedy decode of n tokens after the prompt (tfl_decode_drafted),
    with copy drafts and with a smaller random-init drafter of the same vocabulary
    (the 33B width, DRAFTER_LAYERS layers: about the bytes per step of a 3B
    model), against n plain one-row steps from the same prompt cache.  Wall-clock
    seconds around each host-synchronous call."""
    from gqa_decoder_forward_gb300 import tfl
    shape = model.shape
    prompt = [int(x) for x in ids.cpu()]
    context = prompt + [first_id]
    cap = ctx + max(n, 16) + 1

    def cache_from_prompt():
        c = model.kv(cap)
        tfl.tfl_kv_copy_prefix(model, kv, c, ctx)
        return c

    V = shape.vocab
    kvp = cache_from_prompt()
    pin = torch.tensor([first_id], dtype=torch.int32, device=dev)
    lg = torch.empty((1, V), dtype=torch.bfloat16, device=dev)
    out = torch.empty(n, dtype=torch.int32, device=dev)
    torch.cuda.synchronize()
    w0 = time.perf_counter()
    for t in range(n):
        model.decode_step([kvp], pin if t == 0 else out[t - 1:t], [1], lg)
        model.argmax(lg, out[t:t + 1])
    ref = out.cpu().numpy()
    plain_s = time.perf_counter() - w0
    del kvp
    res = {"tokens": n, "plain_tok_s": round(n / plain_s, 2),
           "reply_distinct_ids": int(len(set(ref.tolist())))}

    # the served model's cost of one verification window of R rows (pending token
    # + R - 1 guesses) at this context: device time of decode step + argmax
    st = torch.cuda.current_stream()
    win = {}
    wc = cache_from_prompt()
    wid = torch.tensor(context[-16:], dtype=torch.int32, device=dev)
    wlg = torch.empty((16, V), dtype=torch.bfloat16, device=dev)
    wout = torch.empty(16, dtype=torch.int32, device=dev)
    for R in (1, 2, 4, 8, 16):
        times = []
        for rep in range(4):
            wc.reset(ctx)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            model.decode_step([wc], wid[:R].contiguous(), [R], wlg[:R])
            model.argmax(wlg[:R], wout[:R])
            e1.record(st)
            torch.cuda.synchronize()
            if rep:
                times.append(e0.elapsed_time(e1))
        win[R] = round(min(times), 4)
    del wc
    res["window_ms"] = win
    # derived, not measured: tok/s if every guess of a k-guess window were kept
    res["tok_s_if_all_kept"] = {k: round((k + 1) / win[k + 1] * 1e3, 1) for k in (1, 3, 7, 15)}

    dshape = shape.with_layers(DRAFTER_LAYERS)
    dw = synth.model_weights(dshape, 23, dev)
    drafter = tfl.Model(dshape, dw, max_rows=2048, max_decode_rows=16, max_context=cap)
    for name, k, use in (("copy", 7, False), ("drafter", 3, True)):
        c = cache_from_prompt()
        d = dkv = None
        if use:
            d, dkv = drafter, drafter.kv(cap)
            for s0 in range(0, ctx, 2048):
                drafter.prefill_chunk(dkv, ids[s0:s0 + 2048].contiguous())
        torch.cuda.synchronize()
        w0 = time.perf_counter()
        got, st = model.decode_drafted(c, context, n, k, d, dkv)
        secs = time.perf_counter() - w0
        res[name] = {"draft_len": k, "tok_s": round(n / secs, 2), "equal_plain": bool((got == ref).all()),
                     "accept_rate": round(st["accepted"] / max(1, st["drafted"]), 4), **st}
        if use:
            res[name]["drafter"] = f"{DRAFTER_LAYERS}-layer 33B-width random-init model, seed 23"
        del c, dkv
    del drafter, dw
    torch.cuda.empty_cache()
    return res


def concurrent_figures(model, kvs, ids, steps, warmup, check_steps=4, clocks_index=None):
    """Decode steps of S streams x 1 row (the concurrent configurations), timed
    with CUDA events; then every stream's greedy ids (and logits) over
    check_steps steps together are compared with the same stream run alone from
    the same state ("each reply equal to its run alone")."""
    from gqa_decoder_forward_gb300 import tfl
    S = len(kvs)
    V = model.shape.vocab
    dev = ids.device
    st = torch.cuda.current_stream()
    logits = torch.empty((S, V), dtype=torch.bfloat16, device=dev)
    cur = ids.clone()

    def step():
        model.decode_step(kvs, cur, [1] * S, logits)
        model.argmax(logits, cur)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    start = [kv.length for kv in kvs]
    clk = ClockSampler(clocks_index) if clocks_index is not None else None
    if clk:
        clk.__enter__()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(st)
    for _ in range(steps):
        step()
    t1.record(st)
    torch.cuda.synchronize()
    if clk:
        clk.__exit__(None, None, None)
    ms = t0.elapsed_time(t1) / steps
    tfl.tfl_profile(model, True)
    step()
    prof = tfl.tfl_profile_read(model)
    phases = tfl.tfl_step_phases(model) if S <= 2 else None
    tfl.tfl_profile(model, False)
    # equal to solo, from the state after the timed steps
    base = [kv.length for kv in kvs]
    first = cur.clone()
    together = []
    for _ in range(check_steps):
        step()
        together.append((logits.clone(), cur.clone()))
    equal = True
    for s in range(S):
        kvs[s].reset(base[s])
        c = first[s:s + 1].clone()
        lg = torch.empty((1, V), dtype=torch.bfloat16, device=dev)
        for t in range(check_steps):
            model.decode_step([kvs[s]], c, [1], lg)
            model.argmax(lg, c)
            equal = equal and torch.equal(lg.view(torch.int16), together[t][0][s:s + 1].view(torch.int16)) \
                and int(c.item()) == int(together[t][1][s].item())
    shape = model.shape
    mean_ctx = sum(start) / S + (steps - 1) / 2.0
    w = step_bytes(shape, 0)
    kvb = shape.layers * 2 * shape.n_kv * shape.head_dim * 2 * mean_ctx * S
    peak, peak_kind = measured_peaks()
    gbs = (w + kvb) / (ms / 1e3) / 1e9
    out = {"streams": S, "context_start": start, "steps": steps, "warmup": warmup,
           "path": "persistent" if S <= 2 else "launch per operation",
           "tok_s": round(S * 1e3 / ms, 2), "ms_per_step": round(ms, 4), "bytes_per_step": int(w + kvb),
           "achieved_gbs": round(gbs, 1), "hbm_frac": round(gbs / peak, 4), "peak_kind": peak_kind,
           "equal_solo": bool(equal), "equal_solo_steps": check_steps, "status": model.status(),
           "step_phases_us": phases,
           "kernels_one_step": {k: {"ms": round(v[0], 4), "launches": v[1]} for k, v in prof.items() if v[1]}}
    if clk:
        out["clocks"] = clk.summary()
    return out


def run_concurrent(args):
    """Decode steps of S streams x 1 row over seeded caches of --context positions each
    (the concurrent configurations: 2 x 131,072 and 16 x 8,192), with the
    equal-to-solo check."""
    from gqa_decoder_forward_gb300 import build, tfl
    build.build()
    S, ctx = args.concurrent, args.context
    shape = SHAPE.with_layers(args.layers)
    dev = torch.device("cuda", torch.cuda.current_device())
    weights = synth.model_weights(shape, 21, dev)
    extra = args.warmup + args.steps + 16
    model = tfl.Model(shape, weights, max_rows=64, max_decode_rows=64, max_context=ctx + extra)
    kvs = [model.kv(ctx + extra) for _ in range(S)]
    for l in range(shape.layers):
        K, V = synth.kv_contents(shape, 22, l, ctx, dev)
        for kv in kvs:
            kv.write(l, 0, K, V)
        del K, V
    for kv in kvs:
        kv.reset(ctx)
    ids = synth.uniform_ids(41, S, shape.vocab, dev)
    res = concurrent_figures(model, kvs, ids, args.steps, args.warmup, clocks_index=0)
    print(json.dumps({"mode": "concurrent", "context": ctx, "layers": args.layers, "kv": "seeded", **res}),
          flush=True)


def run_op(args):
    """Times one decode op on a one-layer 33B-shaped model (a few GB on the device):
    the small case the kernel profiles are taken on."""
    from gqa_decoder_forward_gb300 import build, tfl
    build.build()
    one = SHAPE.with_layers(1)
    dev = torch.device("cuda", torch.cuda.current_device())
    w = {k: [synth.layer_weight(one, 21, 0, k, dev)] for k in synth.LAYER_KEYS}
    # the op entry points never read the embedding table or lm_head: small stand-ins
    w["embed"] = torch.zeros(64, dtype=torch.bfloat16, device=dev)
    w["final_norm"] = torch.ones(one.hidden, dtype=torch.bfloat16, device=dev)
    w["lm_head"] = torch.zeros(64, dtype=torch.bfloat16, device=dev)
    R, ctx = args.rows, args.context
    m = tfl.Model(one, w, max_rows=max(64, R), max_decode_rows=64, max_context=ctx + R)
    if args.op == "sample":
        # seeded draw at temperature 0.6, top-k 20, top-p 0.95 over the 166,912-id vocabulary
        lg = synth.normal_bf16(5, 5, (R, one.vocab), 2.0, dev)
        u = torch.rand(R, generator=torch.Generator().manual_seed(7)).to(dev)
        ids = torch.empty(R, dtype=torch.int32, device=dev)
        for _ in range(args.warmup):
            m.sample(lg, 0.6, 20, 0.95, u, ids)
        torch.cuda.synchronize()
        st = torch.cuda.current_stream()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(st)
        for _ in range(args.steps):
            m.sample(lg, 0.6, 20, 0.95, u, ids)
        t1.record(st)
        torch.cuda.synchronize()
        print(json.dumps({"op": "sample", "rows": R, "vocab": one.vocab, "us_per_launch":
                          round(t0.elapsed_time(t1) / args.steps * 1e3, 2), "status": m.status()}), flush=True)
        return
    kv = m.kv(ctx + R)
    K, V = synth.kv_contents(one, 22, 0, ctx + R, dev)
    kv.write(0, 0, K, V)
    H, QD, F = one.hidden, one.n_q * 128, one.ffn
    x = {"attn_norm": (H, H), "qkv_rope": (H, QD), "attention": (QD, QD), "o_residual": (QD, H),
         "gate_up": (H, F), "down_residual": (F, H), "norm_qkv_rope": (H, QD), "norm_gate_up": (H, F)}[args.op]
    inp = synth.normal_bf16(5, 5, (R, x[0]), 1.0, dev)
    out = synth.normal_bf16(6, 6, (R, x[1]), 1.0, dev)
    for _ in range(args.warmup):
        tfl.tfl_layer_op(m, args.op, 0, inp, out, kv, ctx, prompt=args.prompt)
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(st)
    for _ in range(args.steps):
        tfl.tfl_layer_op(m, args.op, 0, inp, out, kv, ctx, prompt=args.prompt)
    t1.record(st)
    torch.cuda.synchronize()
    us = t0.elapsed_time(t1) / args.steps * 1e3
    wbytes = {"attn_norm": 2 * H, "qkv_rope": (QD + 2 * 1024) * H * 2, "attention": 2 * 1024 * 2 * (ctx + R),
              "o_residual": H * QD * 2, "gate_up": 2 * F * H * 2, "down_residual": H * F * 2,
              "norm_qkv_rope": (QD + 2 * 1024) * H * 2, "norm_gate_up": 2 * F * H * 2}[args.op]
    flops = 2.0 * R * {"attn_norm": 0, "qkv_rope": (QD + 2 * 1024) * H, "o_residual": H * QD,
                       "norm_qkv_rope": (QD + 2 * 1024) * H, "norm_gate_up": 2 * F * H,
                       "gate_up": 2 * F * H, "down_residual": H * F,
                       "attention": one.n_q * 128 * 2 * (ctx + (R + 1) / 2)}[args.op]
    print(json.dumps({"op": args.op, "prompt": args.prompt, "rows": R, "context": ctx, "us_per_launch": round(us, 2),
                      "bytes": wbytes, "gbs": round(wbytes / us / 1e3, 1),
                      "tflops": round(flops / us / 1e6, 1)}), flush=True)


def main():
    args = parse()
    if args.op:
        run_op(args)
        return
    if args.concurrent:
        run_concurrent(args)
        return
    world, rank, local = dist_init(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_tfl(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
