"""Benchmark of the LongFlow fused decode step (attention + score + eviction).

One *step* = one decode token for every layer and sequence of the workload
(layers x batch "units", one lf_decode_step launch per layer).  The metric is
units per second ("fused decode steps/s (batch x layers)") and the achieved
HBM bandwidth of the decode kernel against the measured copy peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl ours|reference]

--impl reference times the fp64 CPU oracle on the host cores (the reference
arm: a deliberately slow, plain implementation of the same step).

Multi-GPU: every rank runs an independent replica (the path has no exchange
step); the time is the max over ranks and the value the units of all ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused decode steps/s (batch·layers) and achieved HBM GB/s vs ~8 TB/s peak"
UNIT = "units/s (unit = one (layer, sequence) decode step)"
NOMINAL_HBM_GBS = 8000.0


# ---------------------------------------------------------------------------
# byte model (algorithmic bytes of one (layer, sequence) unit)
# ---------------------------------------------------------------------------

def unit_bytes(wl, n_slots: int, evict: bool = True, writes_slot: bool = True,
               h2o: bool = False) -> int:
    """K and V of the n occupied slots, their ||v||_1 and positions, q read,
    out written, k_new / v_new read, and (when a slot is written) the new
    token's K, V, ||v||_1, position plus the evicted index.  The H2O score
    reads each slot's accumulator instead of its ||v|| and writes it back."""
    e = wl.elem_bytes
    hkv, hq, d = wl.kv_heads, wl.q_heads, wl.head_dim
    b = 2 * hkv * n_slots * d * e + 8 * hkv * n_slots
    b += 2 * hq * d * e + 2 * hkv * d * e
    b += 4 * hkv  # evicted slot index
    if writes_slot:
        b += 2 * hkv * d * e + 8 * hkv
    if h2o:
        b += 4 * hkv * n_slots + (4 * hkv if writes_slot else 0)
    return b


# Policy variants timed beside the default method (name -> LFCache keywords).
POLICY_VARIANTS = {
    "l2_sinks4": dict(norm=2, sinks=4),
    "deferred": dict(deferred=True),
    "layer_scope": dict(scope="layer"),
    "h2o": dict(score="h2o"),
    # the guide listing's choices together (window 1: only the new token protected)
    "listing": dict(sinks=4, deferred=True, scope="layer"),
}


KERNEL_SOURCES = ["lf_decode_tc.cuh", "lf_decode.cuh", "lf_device.cuh"]
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "decode_step_tc_qwen3-8b-steady.md")


def kernel_source_hash() -> str:
    """sha256 over the decode kernels' sources: ties a stored ncu traffic figure
    to the exact code it was measured on."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "decode_kv_cache_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def stored_traffic(workload: str, batch: int):
    """DRAM bytes (read + write) per decode launch from the committed ncu
    summary, if it was taken on this workload and on the current kernel source;
    else None."""
    try:
        text = open(PROFILE_SUMMARY).read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- `"):
            key, _, val = line.strip()[3:].partition("`:")
            vals[key.strip()] = val.strip().strip("`")
    try:
        if (vals.get("kernel_source_sha256") != kernel_source_hash() or
                vals.get("workload") != workload or int(vals.get("batch", -1)) != batch):
            return None
        return int(vals["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def aggregate(ms_local: float, units_local: int, dist=None):
    """Whole-job throughput of independent replicas: the slowest rank's time
    and the units of all ranks (max / sum over the process group)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return ms_local, units_local
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([ms_local], dtype=torch.float64, device=dev)
    u = torch.tensor([units_local], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), int(u.item())


def load_tensor_peak():
    """Measured dense bf16 TFLOP/s (burst: the compression is timed on its own)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline and reference arm)
# ---------------------------------------------------------------------------

def _oracle_worker(args):
    """Run OracleSequence steps of one (layer, sequence) for `seconds` (or `steps`)."""
    wl_name, overrides, seed, seconds, steps = args
    import numpy as np
    sys.path.insert(0, ROOT)
    import oracle
    from synth.workloads import get_workload
    wl = get_workload(wl_name).scaled(**overrides)
    rng = np.random.default_rng(seed)
    seq = oracle.OracleSequence(wl.kv_heads, wl.q_heads, wl.budget, wl.head_dim, wl.budget,
                                wl.window, evict=True)
    P = wl.budget  # steady state: the buffer is full, every step evicts
    k = rng.standard_normal((wl.kv_heads, P, wl.head_dim))
    v = rng.standard_normal((wl.kv_heads, P, wl.head_dim))
    seq.prefill(k, v)
    q = rng.standard_normal((wl.q_heads, wl.head_dim))
    done = 0
    t0 = time.perf_counter()
    while True:
        q = wl.rho * q + 0.44 * rng.standard_normal(q.shape)
        seq.step(q, rng.standard_normal((wl.kv_heads, wl.head_dim)),
                 rng.standard_normal((wl.kv_heads, wl.head_dim)))
        done += 1
        el = time.perf_counter() - t0
        if (steps and done >= steps) or (not steps and el >= seconds):
            return done, el


def run_oracle(wl_name: str, workers: int, seconds: float = 0.0, steps: int = 0):
    import multiprocessing as mp
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"  # one core per worker process: `cores` is exact
    ctx = mp.get_context("spawn")
    with ctx.Pool(workers) as pool:
        res = pool.map(_oracle_worker, [(wl_name, {}, 1000 + i, seconds, steps)
                                        for i in range(workers)])
    units = sum(r[0] for r in res)
    wall = max(r[1] for r in res)
    return units, wall


def cpu_baseline(wl_name: str, seconds: float):
    """The oracle on every host core (the reported value) and on one core."""
    cores = os.cpu_count() or 1
    units, wall = run_oracle(wl_name, cores, seconds=seconds)
    one_units, one_wall = run_oracle(wl_name, 1, seconds=max(1.0, seconds / 3))
    return {"value": units / wall, "unit": UNIT, "cores": cores, "kind": "oracle",
            "single_core_value": one_units / one_wall,
            "sample": f"{cores} spawn workers x ~{seconds:.0f} s each of fp64 oracle steps of one "
                      f"{wl_name}-shaped (layer, sequence) at steady state (full buffer, every "
                      f"step evicts); {units} units total. single_core_value: one worker, "
                      f"~{max(1.0, seconds / 3):.0f} s, {one_units} units"}


def workload_config(wl, layers: int) -> dict:
    """The workload keys of `config`, the same in both arms."""
    return {"workload": wl.name, "layers": layers, "batch": wl.batch, "q_heads": wl.q_heads,
            "kv_heads": wl.kv_heads, "head_dim": wl.head_dim, "budget": wl.budget,
            "window": wl.window,
            "state": ("steady (pre-filled to the budget, every step evicts)"
                      if wl.prefill >= wl.budget else
                      f"prompt {wl.prefill}, timed from the start of generation")}


def bench_reference(args):
    """--impl reference: the oracle as the reference arm on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    cores = os.cpu_count() or 1
    t_all = time.perf_counter()
    # warm-up: W oracle steps per worker, untimed
    if args.warmup:
        run_oracle(args.workload, cores, steps=args.warmup)
    units, wall = run_oracle(args.workload, cores, steps=args.steps)
    value = units / wall
    from synth import workloads as stream_mod
    wl = stream_mod.get_workload(args.workload)
    config = workload_config(wl, args.layers or wl.layers)
    config["sample"] = "one (layer, sequence) unit per worker per step, at steady state"
    line = {"metric": METRIC, "value": value, "unit": UNIT, "impl": "reference",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * wall / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config,
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"each of {cores} spawn workers runs {args.steps} fp64 "
                                       f"oracle steps of one {args.workload}-shaped (layer, "
                                       f"sequence) at steady state"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "wall_s": time.perf_counter() - t_all}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

def build_cache(wl, torch, lf, stream_mod, seed, evict=True, capacity=None, layers=None,
                cluster=0, stages=0, policy=None, kernel="auto"):
    L = wl.layers if layers is None else layers
    cap = capacity or wl.budget
    policy = policy or {}
    gen = stream_mod.InputStream(wl, seed=seed, device="cuda", layers=list(range(L)))
    budgets = gen.budgets if (evict and wl.ragged) else None
    cache = lf.LFCache(L, wl.batch, wl.kv_heads, wl.q_heads, wl.head_dim, cap, wl.window,
                       dtype=wl.dtype, evict=evict, budgets=budgets, cluster=cluster,
                       stages=stages, kernel=kernel, **policy)
    # deferred eviction keeps one slot free in the prompt (the step that fills
    # the buffer chooses the first victim)
    spare = 1 if (evict and policy.get("deferred")) else 0
    limits = [(budgets[b] if budgets else cap) - spare for b in range(wl.batch)]
    for l in range(L):
        # prompt tokens past a sequence's budget come out of the stream as its
        # first decode tokens (the batch advances in lock-step)
        k, v, lens = gen.prompt_split(l, limits)
        cache.prefill(l, k, v, lens)
        del k, v
    torch.cuda.synchronize()
    return cache, gen


def pregenerate(gen, steps, torch):
    """Inputs of `steps` decode steps, resident in HBM: list of (q, k, v) per layer."""
    out = []
    for _ in range(steps):
        qs, ks, vs = gen.next_step()
        out.append((qs, ks, vs))
    torch.cuda.synchronize()
    return out


def time_steps(cache, inputs, outs, evs, torch, graph: bool):
    """Run len(inputs) steps; return elapsed ms measured with CUDA events."""
    L = len(outs)
    stream = torch.cuda.current_stream()

    def launch_all():
        for (qs, ks, vs) in inputs:
            for l in range(L):
                cache.decode_step(l, qs[l], ks[l], vs[l], outs[l], evs[l])

    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            launch_all()
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(torch.cuda.current_stream())
        g.replay()
        end.record(torch.cuda.current_stream())
        end.synchronize()
        ms = start.elapsed_time(end)
        del g
        return ms
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    launch_all()
    end.record(stream)
    end.synchronize()
    return start.elapsed_time(end)


def bench_workload(args, torch, lf, stream_mod, peak, name, layers, steady, dist=None):
    """One more workload timed like the headline: its own cache, W untimed
    steps, then `args.steps` steps in one CUDA graph, from the start of
    generation (or at steady state with `steady`).  Returns units/s, the
    algorithmic GB/s of the decode launches, their fraction of the measured
    copy peak, the launch shape and the occupancy the steps ran at."""
    wl = stream_mod.get_workload(name)
    wl = wl.scaled(layers=min(wl.layers, layers))
    if steady:
        wl = wl.scaled(prefill=wl.budget)
    cache, gen = build_cache(wl, torch, lf, stream_mod, seed=400)
    L = wl.layers
    outs = [torch.empty(wl.batch, wl.q_heads, wl.head_dim, dtype=cache.dtype, device="cuda")
            for _ in range(L)]
    evs = [torch.empty(wl.batch, wl.kv_heads, dtype=torch.int32, device="cuda") for _ in range(L)]
    overflow = gen.overflow_lengths(0)
    warm = pregenerate(gen, args.warmup, torch)
    timed = pregenerate(gen, args.steps, torch)
    time_steps(cache, warm, outs, evs, torch, graph=False)
    del warm
    occ_start = cache.views()["count"][0, :, 0].cpu().tolist()
    planned = cache.plan(0) is not None
    torch.cuda.synchronize()
    ms = time_steps(cache, timed, outs, evs, torch, graph=not args.eager)
    ms = aggregate(ms, 0, dist)[0]
    bits = cache.check()
    if bits:
        raise RuntimeError(f"device error word {bits} in the {name} leg")
    occ_end = cache.views()["count"][0, :, 0].cpu().tolist()
    lay = cache.layout
    launches = L * args.steps
    bytes_per_launch = sum((unit_bytes(wl, int(a)) + unit_bytes(wl, int(e))) // 2
                           for a, e in zip(occ_start, occ_end))
    achieved = bytes_per_launch / (ms / 1000.0 / launches) / 1e9
    world = dist.get_world_size() if (dist is not None and dist.is_initialized()) else 1
    cache.close()
    del cache, gen, timed
    torch.cuda.empty_cache()
    return {
        "workload": name, "layers": L, "batch": wl.batch, "steps": args.steps,
        "state": ("steady (pre-filled to the budget, every step evicts)" if steady else
                  f"from the start of generation after step {args.warmup}"),
        "value": world * wl.batch * L * args.steps / (ms / 1000.0), "unit": UNIT,
        "ms_per_layer_step": ms / launches,
        "achieved_gbs": achieved, "frac_of_peak": achieved / peak,
        "frac_of_nominal_8000": achieved / NOMINAL_HBM_GBS,
        "bytes_per_launch": bytes_per_launch,
        "occupied_slots": {"start_mean": sum(occ_start) / len(occ_start),
                           "end_mean": sum(occ_end) / len(occ_end)},
        "prompt_remainder_steps": ({"sequences": sum(1 for x in overflow if x > 0),
                                    "max": max(overflow)} if max(overflow) > 0 else None),
        "launch_shape": {"cluster": lay.cluster, "stages": lay.stages,
                         "planned_at_start": planned},
    }


def bench_rkv(args, torch, lf, stream_mod, peak):
    """R-KV's cycle on rkv-r1-llama-8b: `buffer` decode steps that append into
    the staging buffer, then one compression per layer (lf_rkv_compress).
    Returns amortised units/s, the decode and compression rates, and the ratio
    to LongFlow measured on the same geometry (layers, batch, heads, budget,
    steady state, the window of the r1-llama-8b configuration)."""
    wl = stream_mod.get_workload("rkv-r1-llama-8b")
    L = min(wl.layers, args.rkv_layers)
    wl = wl.scaled(layers=L)
    B, buf, alpha = wl.budget, wl.rkv_buffer, wl.rkv_alpha
    cap = B + buf
    gen = stream_mod.InputStream(wl, seed=300, device="cuda", layers=list(range(L)))
    cache = lf.LFCache(L, wl.batch, wl.kv_heads, wl.q_heads, wl.head_dim, cap, 0, dtype=wl.dtype,
                       evict="rkv", rkv_buffer=buf, rkv_alpha=alpha, rkv_beta=wl.rkv_beta,
                       rkv_lambda=wl.rkv_lambda, rkv_tau=wl.rkv_tau)
    for l in range(L):
        k, v, lens = gen.prompt(l)
        cache.prefill(l, k, v, [min(P, cap) for P in lens])
        del k, v
    outs = [torch.empty(wl.batch, wl.q_heads, wl.head_dim, dtype=cache.dtype, device="cuda")
            for _ in range(L)]
    evs = [torch.empty(wl.batch, wl.kv_heads, dtype=torch.int32, device="cuda") for _ in range(L)]

    def cycle_inputs():
        steps = pregenerate(gen, buf, torch)
        # observation queries of the last alpha steps, per layer: [b][alpha][H_q][d]
        qobs = [torch.stack([steps[t][0][l] for t in range(buf - alpha, buf)], dim=1).contiguous()
                for l in range(L)]
        return steps, qobs

    st = torch.cuda.current_stream()
    # one untimed cycle (the first compression after the prompt), then a timed one
    steps, qobs = cycle_inputs()
    time_steps(cache, steps, outs, evs, torch, graph=False)
    for l in range(L):
        cache.rkv_compress(l, qobs[l])
    if cache.check() != 0:
        raise RuntimeError("device error in the R-KV warm-up cycle")
    steps, qobs = cycle_inputs()
    torch.cuda.synchronize()
    dec_ms = time_steps(cache, steps, outs, evs, torch, graph=not args.eager)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for l in range(L):
        cache.rkv_compress(l, qobs[l])
    e1.record(st)
    e1.synchronize()
    comp_ms = e0.elapsed_time(e1)
    bits = cache.check()
    if bits:
        raise RuntimeError(f"device error word {bits} in the R-KV cycle")
    counts = cache.views()["count"].cpu()
    rlay = cache.layout
    rkv_shape = {"cluster": rlay.cluster, "stages": rlay.stages}
    cache.close()
    del cache, gen, steps, qobs
    torch.cuda.empty_cache()
    units = wl.batch * L * buf
    # LongFlow on the same geometry: a cache at the same budget, filled to it, timed
    # over the same number of decode steps (every step evicts)
    lwl = wl.scaled(window=stream_mod.get_workload("r1-llama-8b").window, prefill=B)
    lcache, lgen = build_cache(lwl, torch, lf, stream_mod, seed=301)
    llay = lcache.layout
    lf_shape = {"cluster": llay.cluster, "stages": llay.stages,
                "planned_at_start": lcache.plan(0) is not None}
    lwarm = pregenerate(lgen, 3, torch)
    time_steps(lcache, lwarm, outs, evs, torch, graph=False)
    del lwarm
    lsteps = pregenerate(lgen, buf, torch)
    lf_ms = time_steps(lcache, lsteps, outs, evs, torch, graph=not args.eager)
    if lcache.check() != 0:
        raise RuntimeError("device error in the LongFlow run on the R-KV geometry")
    lcache.close()
    del lcache, lgen, lsteps
    torch.cuda.empty_cache()
    longflow_units_per_s = units / (lf_ms / 1000.0)
    # decode bytes: occupancy grows from B to B + buf - 1 over the cycle
    dec_bytes = sum(unit_bytes(wl, B + t) for t in range(buf)) * wl.batch * L
    # compression: the key dot products of the blocks J >= I plus two importance passes
    n = cap
    nb = (n + 127) // 128
    qn = (alpha * wl.group + 15) // 16 * 16
    flops_unit = nb * (nb + 1) // 2 * 2 * 128 * 128 * 128 + 2 * nb * 2 * 128 * qn * 128
    comp_units = wl.batch * wl.kv_heads * L
    value = units / ((dec_ms + comp_ms) / 1000.0)
    return {
        "workload": wl.name, "layers": L, "batch": wl.batch, "budget": B, "buffer": buf,
        "alpha": alpha, "lambda": wl.rkv_lambda, "tau": wl.rkv_tau, "beta": wl.rkv_beta,
        "value": value, "unit": UNIT,
        "cycle": f"{buf} decode steps + 1 compression per layer",
        "decode_units_per_s": units / (dec_ms / 1000.0),
        "decode_achieved_gbs": dec_bytes / (dec_ms / 1000.0) / 1e9,
        "decode_frac_of_peak": dec_bytes / (dec_ms / 1000.0) / 1e9 / peak,
        "compress_ms_per_layer": comp_ms / L,
        "compress_share_of_cycle": comp_ms / (dec_ms + comp_ms),
        "compress_tensor_tflops": flops_unit * comp_units / (comp_ms / 1000.0) / 1e12,
        "compress_frac_of_tensor_peak": (flops_unit * comp_units / (comp_ms / 1000.0) / 1e12
                                         / load_tensor_peak()[0]),
        "tensor_peak_kind": load_tensor_peak()[1],
        "counts_after": [int(counts.min()), int(counts.max())],
        "longflow_units_per_s_same_geometry": longflow_units_per_s,
        "launch_shapes": {"rkv_decode": rkv_shape, "longflow": lf_shape},
        "longflow_geometry": f"{L} layers, batch {wl.batch}, budget {B}, window {lwl.window}, "
                             f"steady, {buf} steps",
        "longflow_over_rkv": longflow_units_per_s / value,
    }


def bench_ours(args):
    import torch
    import torch.distributed as dist

    from decode_kv_cache_gb300 import longflow as lf
    from synth import workloads as stream_mod

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    from decode_kv_cache_gb300 import build as _b
    if rank == 0 or world == 1:
        _b.build()
    if world > 1:
        dist.barrier()
    lf.load_library()

    wl = stream_mod.get_workload(args.workload)
    if args.layers:
        wl = wl.scaled(layers=args.layers)
    if args.batch:
        wl = wl.scaled(batch=args.batch)
    if args.steady and not wl.ragged:
        wl = wl.scaled(prefill=wl.budget)
    peak, peak_kind = load_peaks()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def max_over_ranks(x: float) -> float:
        return aggregate(x, 0, dist)[0]

    # ---- eviction on, steady state (cache pre-filled to the budget) ----
    cache, gen = build_cache(wl, torch, lf, stream_mod, seed=rank, cluster=args.cluster,
                             stages=args.stages, kernel=args.kernel)
    L = wl.layers
    outs = [torch.empty(wl.batch, wl.q_heads, wl.head_dim, dtype=cache.dtype, device="cuda")
            for _ in range(L)]
    evs = [torch.empty(wl.batch, wl.kv_heads, dtype=torch.int32, device="cuda") for _ in range(L)]
    warm = pregenerate(gen, args.warmup, torch)
    timed = pregenerate(gen, args.steps, torch)
    time_steps(cache, warm, outs, evs, torch, graph=False)  # W untimed warm-up steps
    del warm
    if cache.check() != 0:
        raise RuntimeError("device error during warm-up")
    occ_start = cache.views()["count"][0, :, 0].cpu().tolist()  # occupied slots per sequence
    planned = cache.plan(0) is not None
    clocks = ClockSampler(local)
    barrier()
    clocks.start()
    ms = time_steps(cache, timed, outs, evs, torch, graph=not args.eager)
    barrier()
    clk = clocks.stop()
    bits = cache.check()
    if bits:
        raise RuntimeError(f"device error word {bits} after the timed region")
    ms, all_units = aggregate(ms, wl.batch * L * args.steps, dist)
    value = all_units / (ms / 1000.0)
    launches = L * args.steps
    # algorithmic bytes per launch: the mean occupancy over the timed steps (the
    # start and end counts; steady workloads stay at the budget throughout)
    occ_end = cache.views()["count"][0, :, 0].cpu().tolist()
    bytes_per_launch = sum((unit_bytes(wl, int(a)) + unit_bytes(wl, int(e))) // 2
                           for a, e in zip(occ_start, occ_end))
    achieved = bytes_per_launch / (ms / 1000.0 / launches) / 1e9
    lay = cache.layout

    # ---- e2e: host buffers, copies inside the timed region ----
    # Each step's inputs (every layer's q, k_new, v_new) sit in one pinned host
    # buffer and go up in one copy; each step's results (out, evicted) come back
    # in one copy.  Copies run on their own streams, two steps in flight: the
    # upload of step s+1 and the download of step s-1 overlap step s's kernels.
    e2e_steps = min(args.steps, args.e2e_steps)
    shapes_in = [(t.shape, t.dtype) for grp in timed[0] for t in grp]
    shapes_out = [(o.shape, o.dtype) for o in outs] + [(e.shape, e.dtype) for e in evs]

    def nbytes(shape, dtype):
        return math.prod(shape) * torch.empty((), dtype=dtype).element_size()

    h2d = sum(nbytes(*sd) for sd in shapes_in)
    d2h = sum(nbytes(*sd) for sd in shapes_out)

    def carve(flat, shapes):
        views, off = [], 0
        for shape, dtype in shapes:
            nb = nbytes(shape, dtype)
            views.append(flat[off:off + nb].view(dtype).view(shape))
            off += (nb + 255) // 256 * 256
        return views

    def padded(shapes):
        return sum((nbytes(*sd) + 255) // 256 * 256 for sd in shapes)

    host_in = []
    for (qs, ks, vs) in timed[:e2e_steps]:
        flat = torch.empty(padded(shapes_in), dtype=torch.uint8).pin_memory()
        for dst, src in zip(carve(flat, shapes_in), list(qs) + list(ks) + list(vs)):
            dst.copy_(src.cpu())
        host_in.append(flat)
    del timed
    dev_in = [torch.empty(padded(shapes_in), dtype=torch.uint8, device="cuda") for _ in range(2)]
    dev_out = [torch.empty(padded(shapes_out), dtype=torch.uint8, device="cuda") for _ in range(2)]
    host_out = [torch.empty(padded(shapes_out), dtype=torch.uint8).pin_memory() for _ in range(2)]
    in_views = [carve(b, shapes_in) for b in dev_in]
    out_views = [carve(b, shapes_out) for b in dev_out]
    barrier()
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()

    def ev():
        return torch.cuda.Event()

    uploaded = [ev() for _ in range(e2e_steps)]
    computed = [ev() for _ in range(e2e_steps)]
    downloaded = [ev() for _ in range(e2e_steps)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)

    def upload(s):
        up.wait_event(e0)
        if s >= 2:
            up.wait_event(computed[s - 2])        # the kernels of step s-2 read this buffer
        with torch.cuda.stream(up):
            dev_in[s % 2].copy_(host_in[s], non_blocking=True)
        uploaded[s].record(up)

    upload(0)
    for s in range(e2e_steps):
        if s + 1 < e2e_steps:
            upload(s + 1)
        comp.wait_event(uploaded[s])
        if s >= 2:
            comp.wait_event(downloaded[s - 2])    # step s-2's results have left this buffer
        v = in_views[s % 2]
        o = out_views[s % 2]
        for l in range(L):
            cache.decode_step(l, v[l], v[L + l], v[2 * L + l], o[l], o[L + l])
        computed[s].record(comp)
        down.wait_event(computed[s])
        with torch.cuda.stream(down):
            host_out[s % 2].copy_(dev_out[s % 2], non_blocking=True)
        downloaded[s].record(down)
    comp.wait_event(downloaded[e2e_steps - 1])
    e1.record(comp)
    e1.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1))
    e2e_value = world * wl.batch * L * e2e_steps / (e2e_ms / 1000.0)
    cache.close()
    del cache, gen, host_in, dev_in, dev_out, host_out, in_views, out_views
    torch.cuda.empty_cache()

    # ---- eviction off: the same kernel over the full-length KV (read only) ----
    full = None
    if args.full_kv and wl.full_kv_capacity:
        cap = wl.full_kv_capacity
        fl = min(L, args.full_kv_layers)
        wl_full = wl.scaled(prefill=cap, layers=fl)
        need = 2 * fl * wl.batch * wl.kv_heads * cap * wl.head_dim * wl.elem_bytes
        free = torch.cuda.mem_get_info()[0]
        if need * 1.3 < free:
            cfull, gfull = build_cache(wl_full, torch, lf, stream_mod, seed=rank + 100, evict=False,
                                       capacity=cap, layers=fl)
            outs_f = outs[:fl]
            evs_f = evs[:fl]
            fsteps = max(4, args.steps // 4)
            warm = pregenerate(gfull, args.warmup, torch)
            time_steps(cfull, warm, outs_f, evs_f, torch, graph=False)
            del warm
            tin = pregenerate(gfull, fsteps, torch)
            barrier()
            fms = max_over_ranks(time_steps(cfull, tin, outs_f, evs_f, torch,
                                            graph=not args.eager))
            fb = unit_bytes(wl_full, cap, writes_slot=False) * wl.batch
            full = {"value": world * wl.batch * fl * fsteps / (fms / 1000.0), "unit": UNIT,
                    "layers": fl, "steps": fsteps, "capacity": cap,
                    "ms_per_layer_step": fms / (fl * fsteps),
                    "achieved_gbs": fb / (fms / 1000.0 / (fl * fsteps)) / 1e9}
            cfull.close()
            del tin
        else:
            full = {"skipped": f"needs {need / 1e9:.1f} GB, {free / 1e9:.1f} GB free"}

    # ---- policy variants on the same workload (fewer layers) ----
    policies = None
    if args.policies and wl.prefill >= wl.budget and not wl.ragged:
        policies = {}
        pl = min(L, args.policy_layers)
        psteps = max(8, args.steps // 4)
        for name, kw in POLICY_VARIANTS.items():
            wl_p = wl.scaled(layers=pl, window=1) if name == "listing" else wl.scaled(layers=pl)
            cp, gp = build_cache(wl_p, torch, lf, stream_mod, seed=rank + 200, layers=pl,
                                 cluster=args.cluster, stages=args.stages, policy=kw)
            warm = pregenerate(gp, args.warmup, torch)
            time_steps(cp, warm, outs[:pl], evs[:pl], torch, graph=False)
            del warm
            tin = pregenerate(gp, psteps, torch)
            barrier()
            pms = max_over_ranks(time_steps(cp, tin, outs[:pl], evs[:pl], torch,
                                            graph=not args.eager))
            if cp.check() != 0:
                raise RuntimeError(f"device error in the {name} variant")
            pb = unit_bytes(wl_p, wl_p.budget, h2o=(kw.get("score") == "h2o")) * wl.batch
            per_launch = pms / 1000.0 / (pl * psteps)
            policies[name] = {
                "policy": kw, "value": world * wl.batch * pl * psteps / (pms / 1000.0),
                "unit": UNIT, "layers": pl, "steps": psteps,
                "launches_per_layer_step": 2 if kw.get("scope") == "layer" else 1,
                "bytes_per_layer_step": pb, "achieved_gbs": pb / per_launch / 1e9,
                "frac_of_peak": pb / per_launch / 1e9 / peak}
            cp.close()
            del cp, gp, tin
            torch.cuda.empty_cache()

    # ---- the other two timed workloads: batch 32 at budget 3276 (steady) and
    # the ragged serving batch (from its prompts, remainders fed as steps) ----
    others = {}
    if args.other_workloads and not (args.layers or args.batch):
        others["r1_llama_steady"] = bench_workload(args, torch, lf, stream_mod, peak,
                                                   "r1-llama-8b", args.r1_layers, True, dist)
        others["ragged"] = bench_workload(args, torch, lf, stream_mod, peak, "ragged-serving",
                                          args.ragged_layers, False, dist)

    # ---- R-KV, the pages' baseline, on its own workload (fewer layers) ----
    rkv = None
    if args.rkv and rank == 0:
        rkv = bench_rkv(args, torch, lf, stream_mod, peak)

    if rank != 0:
        return 0
    cpu = None
    if not args.no_cpu_baseline:
        cpu = cpu_baseline(args.workload, args.cpu_seconds)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if
        wl.dtype == "bf16" else "f32", "data": "synthetic",
        "config": {**workload_config(wl, L),
                   "l2": "inputs larger than L2: each layer's slab is "
                   f"{wl.batch * wl.kv_heads * lay.slot_stride * wl.head_dim * 2 * wl.elem_bytes / 1e6:.0f} MB",
                   "cluster": lay.cluster, "stages": lay.stages,
                   "launch": "eager" if args.eager else "CUDA graph of all timed steps",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "frac_of_nominal_8000": achieved / NOMINAL_HBM_GBS,
                     "traffic": stored_traffic(wl.name, wl.batch),
                     "kernel": (f"decode_step_tc_kernel<{wl.group}, "
                                f"{'true' if planned else 'false'}>" if lay.kernel == 2 else
                                f"decode_step_simt_kernel<{wl.dtype},{wl.head_dim},{wl.group}>"),
                     "bytes_per_launch": bytes_per_launch,
                     "timing": "timed region / launches (includes launch gaps)"},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": launches,
        "clocks": clk,
        "full_kv": full,
        "policy_variants": policies,
        "rkv": rkv,
        **others,
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=128)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="qwen3-8b-steady")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=0, help="override the layer count")
    ap.add_argument("--batch", type=int, default=0, help="override the batch (sequences)")
    ap.add_argument("--kernel", default="auto", choices=["auto", "simt", "tc"],
                    help="decode kernel of the timed workload (auto: tensor cores where built)")
    ap.add_argument("--steady", action="store_true",
                    help="start with the cache filled to the budget (every step evicts) "
                         "instead of from the workload's prompt")
    ap.add_argument("--cluster", type=int, default=0)
    ap.add_argument("--stages", type=int, default=0)
    ap.add_argument("--eager", action="store_true", help="launch eagerly instead of a CUDA graph")
    ap.add_argument("--e2e-steps", type=int, default=32)
    ap.add_argument("--full-kv", dest="full_kv", action="store_true", default=True)
    ap.add_argument("--no-full-kv", dest="full_kv", action="store_false")
    ap.add_argument("--full-kv-layers", type=int, default=8)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-policies", dest="policies", action="store_false", default=True,
                    help="skip timing the policy variants")
    ap.add_argument("--policy-layers", type=int, default=8)
    ap.add_argument("--no-rkv", dest="rkv", action="store_false", default=True,
                    help="skip the R-KV baseline leg")
    ap.add_argument("--rkv-layers", type=int, default=4)
    ap.add_argument("--no-other-workloads", dest="other_workloads", action="store_false",
                    default=True, help="skip the r1-llama-8b steady and ragged legs")
    ap.add_argument("--r1-layers", type=int, default=32)
    ap.add_argument("--ragged-layers", type=int, default=8)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return bench_reference(args)
    return bench_ours(args)


if __name__ == "__main__":
    sys.exit(main())
