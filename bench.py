#!/usr/bin/env python
"""Throughput of one Mixture-of-Experts layer forward on GB300.

A step is one pass of the whole layer (router, softmax/top-8/renormalise,
permutation, expert SwiGLU FFNs, weighted combine) over one batch of
synthetic tokens, with the weights resident in HBM. The default run measures
all six workloads of the layer (d=4096, E=256 experts, top-8, I=1536):

  decode_t1        T=1 single-request decode, bf16 experts      (the headline)
  decode_t4/_t16   T=4 / 16 batched decode / speculative verify, bf16 experts
  prefill_t4096    T=4096 prefill, bf16 experts, Zipf-skewed router bias
  nvfp4_prefill_t4096  the same prefill layer with NVFP4 experts
  nvfp4_stack_t4   8 stacked layers (RMSNorm, MoE, residual), T=4, NVFP4 experts

and prints ONE JSON line: the headline's fields at the top level and every
workload's measurement under "workloads". Tokens rotate through a pool of 64
seeded N(0,1) batches and L2 is flushed (256 MiB write) before every step,
outside the step's CUDA events, so every step streams its weights from HBM.

    python bench.py [--gpus N --steps K --warmup W] [--impl reference] [--workload NAME|all]

Under torchrun (N > 1) every rank holds full layer replicas and processes its
own tokens (no data-path collective); rank 0 prints the line, with each
workload's time taken as the max over ranks.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import datagen  # noqa: E402

METRIC = "MoE-layer tok/s; decode HBM GB/s vs ~8 TB/s; prefill TFLOP/s vs bf16 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FLUSH_BYTES = 256 << 20
POOL = 64
HEAD_START_GROUP = 16      # steps enqueued behind one device-side spin
HEAD_START_HZ = 2.1e9      # spin length in SM cycles per second (at most the maximum SM clock)
HEADLINE = "decode_t1"
DECODE_PATHS = {"auto": 0, "cuda_cores": 1, "tensor_cores": 2}
ORDER = ["decode_t1", "decode_t4", "decode_t16", "prefill_t4096", "nvfp4_prefill_t4096", "nvfp4_stack_t4"]


# ---------------------------------------------------------------------------
# helpers shared by both arms
# ---------------------------------------------------------------------------

def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="all", choices=["all"] + sorted(datagen.WORKLOADS))
    p.add_argument("--gate-up-layout", choices=["separate", "interleaved"], default="separate",
                   help="bf16 gate/up weights as two [E, I, d] tensors, or one [E, I, 2, d] interleaved by row")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=200)
    p.add_argument("--decode-path", choices=["auto", "cuda_cores", "tensor_cores"], default="auto",
                   help="small-batch kernel (T <= 16): the library's choice, or one forced")
    p.add_argument("--experts", type=int, default=0,
                   help="override E (a smaller layer of the same kernels, for profiler captures)")
    return p.parse_args(argv)


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def init_dist(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def reduce_max(value: float, dist, device=None) -> float:
    """Max of a float over ranks (identity without a process group)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(units_per_rank: float, seconds_per_rank: float, dist, device=None):
    """Whole-job throughput: all ranks' units over the slowest rank's time."""
    world = 1 if dist is None else dist.get_world_size()
    t = reduce_max(seconds_per_rank, dist, device)
    return units_per_rank * world / t, t


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch of the
# dominant kernel, from one ncu capture: a 32-expert layer of the same kernel
# (T=1 streams the same 8 experts), plus the 256-expert router's extra 1.84 MB.
# Valid only for the kernel source it was taken on: the sha256 of the kernel's
# source files must match, else the bench reports traffic as null.
TRAFFIC = {
    "decode_t1": {"bytes": 304.23e6 + 3.32e6,
                  "sources": ("top_moe_expert_router_gb300/csrc/decode_fused.cuh",
                              "top_moe_expert_router_gb300/csrc/decode_fused.cu",
                              "top_moe_expert_router_gb300/csrc/common.cuh",
                              "top_moe_expert_router_gb300/csrc/decode_common.cuh"),
                  "sha256": ("dda2ca4a74c5a09ac6a1f90d0e72915d5cde06064ac2b6ae3d82ded3d5d41ef9",
                             "1d39e048978fb78a6191116a4ce545b150e1efd7577999126a1f97db51c5e355",
                             "1e4bae8433f4bd55832d6ff4c6cc33eb01e10da95441e7ecae209f1d2717eec4",
                             "dac14814856e90a1fc7b34e6b39a4cafaec2db008a714d6fe2cf1818f341f284")},
}


def measured_traffic(workload: str):
    """Per-launch DRAM bytes of the captured kernel, or None if it changed since."""
    import hashlib
    t = TRAFFIC.get(workload)
    if t is None:
        return None
    for src, want in zip(t["sources"], t["sha256"]):
        with open(os.path.join(ROOT, src), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != want:
                return None
    return t["bytes"]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            raw = json.load(f)
        out = {}
        for key in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
            v = raw.get(key)
            if isinstance(v, dict):
                v = v.get("value")
            if isinstance(v, (int, float)):
                out[key] = float(v)
        if "hbm_gbs" in out:
            return out, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
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
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.15)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        self.proc.wait(timeout=5)
        rows = [ln.split(",") for ln in open(self.path).read().strip().splitlines() if ln.strip()]
        os.unlink(self.path)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [c.strip() for c in r]
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def workload_config(w: datagen.Workload, **extra):
    desc = (f"{w.name}: T={w.T}, d={w.d}, E={w.E}, top-{w.k}, I={w.I}, {w.fmt} experts"
            + (f", {w.layers} stacked layers" if w.layers > 1 else "")
            + (", Zipf-skewed router bias" if w.zipf_alpha else ""))
    cfg = {"workload": desc, "T": w.T, "d": w.d, "E": w.E, "top_k": w.k, "I": w.I, "expert_format": w.fmt,
           "layers": w.layers, "router_scale": w.router_scale, "tokens": f"pool of {POOL} seeded N(0,1) batches"}
    cfg.update(extra)
    return cfg


def token_pool(w: datagen.Workload, rank: int):
    """Each rank's POOL batches of w.T tokens (distinct rows of the token stream)."""
    return [datagen.tokens(w, w.T, start_row=(rank * POOL + i) * w.T) for i in range(POOL)]


# ---------------------------------------------------------------------------
# CPU oracle: the reference arm and the cpu_baseline legs
# ---------------------------------------------------------------------------

def _timed(fn, budget_s: float, max_calls: int):
    """Calls fn(i) for i = 0, 1, ... until budget_s has passed (at least once,
    at most max_calls). Returns (calls, seconds)."""
    t0 = time.perf_counter()
    n = 0
    while n < max_calls:
        fn(n)
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    return n, time.perf_counter() - t0


def oracle_decode_rates(w, wr, bias, pool_np, budget_s=4.0):
    """Oracle tok/s on the workload's own steps (one batch of w.T pool tokens
    per oracle forward), all host threads and one thread."""
    import oracle
    xs = np.concatenate(pool_np)
    lg = oracle.router_logits(xs, wr, bias)
    ids, _, _ = oracle.select_topk(lg, w.k)
    g, u, d = datagen.expert_weights(w, experts=np.unique(ids))
    L = oracle.Layer(wr, g, u, d, router_bias=bias, k=w.k)
    out = {}
    cores = oracle.max_threads()
    for threads, budget in ((cores, budget_s), (1, budget_s)):
        oracle.set_threads(threads)
        L.forward(pool_np[0])                     # warm
        n, dt = _timed(lambda i: L.forward(pool_np[i % POOL]), budget, POOL)
        out[threads] = {"value": n * w.T / dt, "unit": "tok/s", "cores": threads, "kind": "oracle",
                        "sample": f"{n} steps of the workload ({w.T} pool token(s) per oracle call), {dt:.1f} s"}
    oracle.set_threads(cores)
    line = dict(out[cores])
    line["single_thread"] = out[1]
    return line


def oracle_nvfp4_packs(w, layer, need):
    """The oracle's own NVFP4 quantisation of the listed experts of one layer
    (full-shape arrays, other experts left zero)."""
    import oracle
    g, u, d = datagen.expert_weights(w, layer, experts=need)
    host = {}
    for name, arr in (("gate", g), ("up", u), ("down", d)):
        E, rows, K = arr.shape
        q = np.zeros((E, rows, K // 2), np.uint8)
        s = np.zeros((E, rows, K // 16), np.uint8)
        gs = np.ones(E, np.float32)
        for e in need:
            q[e], s[e], gs[e] = oracle.quantize_nvfp4(arr[e])
        host["q_" + name], host["s_" + name], host["g_" + name] = q, s, gs
    return host


def oracle_prefill_rates(w, wr, bias, x, sample_all=256, sample_one=8):
    """Prefill: routing of all T tokens plus the expert FFNs of a seeded token
    sample, extrapolated per token to T (all threads: sample_all tokens; one
    thread: sample_one tokens). NVFP4 experts: the oracle quantises the
    sample's experts itself, untimed."""
    import oracle
    cores = oracle.max_threads()
    lg = oracle.router_logits(x, wr, bias)
    ids, _, _ = oracle.select_topk(lg, w.k)
    rng = np.random.default_rng(1)
    sample = np.sort(rng.choice(w.T, sample_all, replace=False))
    need = np.unique(ids[sample])
    if w.fmt == "nvfp4":
        L = oracle.Layer(wr, k=w.k, nvfp4=oracle_nvfp4_packs(w, 0, need), router_bias=bias)
    else:
        g, u, d = datagen.expert_weights(w, experts=need)
        L = oracle.Layer(wr, g, u, d, router_bias=bias, k=w.k)
    out = {}
    for threads, n_s in ((cores, sample_all), (1, sample_one)):
        oracle.set_threads(threads)
        t0 = time.perf_counter()
        lg = oracle.router_logits(x, wr, bias)
        oracle.select_topk(lg, w.k)
        t_route = time.perf_counter() - t0
        t0 = time.perf_counter()
        L.forward(x, tokens=sample[:n_s])
        t_ffn = time.perf_counter() - t0
        t_tot = t_route + t_ffn * w.T / n_s
        out[threads] = {"value": w.T / t_tot, "unit": "tok/s", "cores": threads, "kind": "oracle",
                        "sample": (f"routing of all {w.T} tokens ({t_route:.1f} s) + expert FFNs of {n_s} seeded "
                                   f"tokens ({t_ffn:.1f} s), extrapolated per token to {w.T}")}
    oracle.set_threads(cores)
    line = dict(out[cores])
    line["single_thread"] = out[1]
    return line


def oracle_stack_rates(w, x_batch, n_one=1):
    """Stacked NVFP4 layers: the oracle's own quantisation of each layer's
    bf16 weights (the experts its own routing picks; untimed), then the timed
    forward of the step: per layer RMSNorm, layer, residual add."""
    import oracle
    cores = oracle.max_threads()
    packs, routers = [], []
    cur = x_batch
    for li in range(w.layers):        # untimed preparation, following the oracle's own routing
        wr = datagen.router_weights(w, li)
        u_in = oracle.rmsnorm(cur, 1e-6)
        ids, _, _ = oracle.select_topk(oracle.router_logits(u_in, wr), w.k)
        L = oracle.Layer(wr, k=w.k, nvfp4=oracle_nvfp4_packs(w, li, np.unique(ids)))
        cur = oracle.residual_add(cur, L.forward(u_in)["y"])
        packs.append(L)
        routers.append(wr)

    def step(xb):
        c = xb
        for L in packs:
            u_in = oracle.rmsnorm(c, 1e-6)
            c = oracle.residual_add(c, L.forward(u_in)["y"])
        return c

    out = {}
    for threads, n_tok in ((cores, w.T), (1, n_one)):
        oracle.set_threads(threads)
        t0 = time.perf_counter()
        step(x_batch[:n_tok])
        dt = time.perf_counter() - t0
        out[threads] = {"value": n_tok / dt, "unit": "tok/s", "cores": threads, "kind": "oracle",
                        "sample": (f"one step: {n_tok} token(s) through all {w.layers} layers ({dt:.1f} s); the "
                                   "oracle quantises the experts its own routing picks, untimed")}
    oracle.set_threads(cores)
    line = dict(out[cores])
    line["single_thread"] = out[1]
    return line


def run_reference(args):
    """The reference arm: the CPU oracle timed on the host cores, on the
    headline workload's steps (one pool batch per oracle forward)."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    name = HEADLINE if args.workload == "all" else args.workload
    w = datagen.WORKLOADS[name]
    if w.fmt != "bf16" or w.layers != 1 or w.T > 16:
        print(json.dumps({"impl": "reference", "unavailable": "reference arm runs the bf16 decode workloads"}))
        return 0
    pool = token_pool(w, 0)
    wr = datagen.router_weights(w)
    bias = datagen.router_bias(w)
    lg = oracle.router_logits(np.concatenate(pool), wr, bias)
    ids, _, _ = oracle.select_topk(lg, w.k)
    g, u, d = datagen.expert_weights(w, experts=np.unique(ids))
    L = oracle.Layer(wr, g, u, d, router_bias=bias, k=w.k)
    for s in range(args.warmup):
        L.forward(pool[s % POOL])
    t0 = time.perf_counter()
    for s in range(args.steps):
        L.forward(pool[s % POOL])
    total = time.perf_counter() - t0
    value = w.T * args.steps / total
    sample = f"{args.steps} steps of the workload ({w.T} pool token(s) per oracle call)"
    line = {"metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": workload_config(w, parallelism="host cores, OpenMP over (token, expert) pairs"),
            "cpu_baseline": {"value": value, "unit": "tok/s", "cores": oracle.max_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------------------
# the CUDA arm
# ---------------------------------------------------------------------------

class Ctx:
    """Per-process state of the CUDA arm."""

    def __init__(self, args, moe, device, dist, rank, world, local_rank):
        import torch
        self.args, self.moe, self.device, self.dist = args, moe, device, dist
        self.rank, self.world, self.local_rank = rank, world, local_rank
        self.flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.peaks, self.peak_src = load_peaks()

    def bf(self, a):
        import torch
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(self.device)


def timed_steps(ctx, run_step, steps, warmup, per_step_launches, before_timed=None):
    """Warm-up, then `steps` steps each preceded by an L2 flush (outside the
    step's events). before_timed() runs between the two (e.g. to start the
    library's per-kernel event recording). Returns (per-step ms array,
    clocks, launches)."""
    import torch
    stream = torch.cuda.current_stream()
    t_host = time.perf_counter()
    for s in range(warmup):
        ctx.flush.zero_()
        run_step(s)
    t_host = (time.perf_counter() - t_host) / max(warmup, 1)   # host seconds to enqueue one step
    torch.cuda.synchronize()
    if before_timed is not None:
        before_timed()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    if ctx.dist is not None:
        ctx.dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(ctx.local_rank)
    clocks.start()
    launches = 0
    for s in range(steps):
        if s % HEAD_START_GROUP == 0:
            # a device-side spin outside the step events, long enough for the
            # host to enqueue the next group of steps: the events then time
            # the device work, not a GPU waiting on the Python loop (the e2e
            # figure keeps the host path)
            n = min(HEAD_START_GROUP, steps - s)
            torch.cuda._sleep(int(min(2.0 * n * t_host + 2e-4, 0.05) * HEAD_START_HZ))
        ctx.flush.zero_()
        evs[s][0].record(stream)
        run_step(s)
        evs[s][1].record(stream)
        launches += per_step_launches()
    torch.cuda.synchronize()
    if ctx.dist is not None:
        ctx.dist.barrier()
    clk = clocks.stop()
    return np.array([a.elapsed_time(b) for a, b in evs], np.float64), clk, launches


def e2e_host(ctx, w, pool_np, call, n_steps):
    """End to end through the C ABI from pinned host memory: every step copies
    its tokens in, runs the layer(s), copies the result out and waits."""
    import torch
    xh = [torch.from_numpy(p.view(np.int16)).view(torch.bfloat16).pin_memory() for p in pool_np]
    oh = torch.empty((w.T, w.d), dtype=torch.bfloat16).pin_memory()
    n = len(xh)
    for s in range(3):
        call(xh[s % n], oh)
    t0 = time.perf_counter()
    for s in range(n_steps):
        call(xh[s % n], oh)
    dt = time.perf_counter() - t0
    v, _ = aggregate(w.T * n_steps, dt, ctx.dist, ctx.device)
    return {"value": v, "unit": "tok/s", "h2d_bytes_per_step": w.T * w.d * 2, "d2h_bytes_per_step": w.T * w.d * 2,
            "steps": n_steps, "note": "pinned host tokens -> device, the step, result -> pinned host, stream sync; "
                                      "no L2 flush"}


def unique_experts(gl, pool):
    return np.array([int((gl.route(p)["counts"] > 0).sum().item()) for p in pool], np.float64)


def measure_decode(ctx, w, gl, host):
    """bf16 decode (T <= 16): one persistent launch per step."""
    import torch
    args = ctx.args
    pool_np = token_pool(w, ctx.rank)
    pool = [ctx.bf(p) for p in pool_np]
    out = torch.empty((w.T, w.d), dtype=torch.bfloat16, device=ctx.device)
    # One launch of ours per step (the launch list in profiles/ shows nothing
    # else between the step events): the step's own events then time that
    # kernel, and the library records no second pair of events inside the
    # step (measured: that pair adds ~4 us to a 67 us step). With more
    # launches per step the library's events time the layer kernel.
    gl.forward(pool[0], out)
    torch.cuda.synchronize()
    single = gl.last_launch_count() == 1
    step_ms, clk, launches = timed_steps(ctx, lambda s: gl.forward(pool[s % POOL], out), args.steps, args.warmup,
                                         gl.last_launch_count,
                                         None if single else (lambda: gl.profile_begin(args.steps)))
    prof = step_ms.reshape(-1, 1) if single else gl.profile_end()
    assert gl.device_status() == 0, "device error"
    total_s = float(step_ms.sum()) / 1e3
    value, t_max = aggregate(w.T * args.steps, total_s, ctx.dist, ctx.device)
    U = unique_experts(gl, pool)[np.arange(args.steps) % POOL]
    layer_bytes = U * w.expert_bytes_bf16 + w.E * w.d * 2          # active experts + router
    hbm = ctx.peaks["hbm_gbs"]
    k_ms = prof[:, 0].astype(np.float64)
    ach = float(layer_bytes.mean() / (k_ms.mean() / 1e3) / 1e9)
    mma = args.decode_path == "tensor_cores" or (args.decode_path == "auto" and w.T >= 8)
    roof = {"kernel": "decode_mma_kernel" if mma else "decode_layer_kernel", "bound": "hbm", "achieved": ach,
            "peak": hbm, "unit": "GB/s", "timed_by": "step events (one launch per step)" if single else
            "the library's events around the layer kernel",
            "frac": ach / hbm, "traffic": measured_traffic(w.name) if not args.experts else None,
            "peak_source": ctx.peak_src, "bytes_per_launch": float(layer_bytes.mean()),
            "bytes_rule": "unique active experts x 3*d*I*2 B + router E*d*2 B",
            "unique_experts_per_step": float(U.mean()), "ms_per_launch": float(k_ms.mean())}
    res = {"value": value, "unit": "tok/s", "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": t_max * 1e3 / args.steps, "roofline": roof, "gpu_launches": launches, "clocks": clk,
           "config": workload_config(w, l2="flushed before every step (256 MiB write), outside the step events")}
    res["e2e"] = e2e_host(ctx, w, pool_np, gl.forward_host, min(args.e2e_steps, args.steps))
    if ctx.rank == 0 and not args.no_cpu_baseline:
        wr, bias = host
        res["cpu_baseline"] = oracle_decode_rates(w, wr, bias, pool_np)
    return res


def measure_prefill(ctx, w, gl, host):
    """bf16 prefill (T = 4096): routing, gather, two grouped tcgen05 GEMMs, combine."""
    import torch
    args = ctx.args
    n_pool = 4                                   # 4 distinct 4096-token batches
    pool_np = [datagen.tokens(w, w.T, start_row=(ctx.rank * n_pool + i) * w.T) for i in range(n_pool)]
    pool = [ctx.bf(p) for p in pool_np]
    out = torch.empty((w.T, w.d), dtype=torch.bfloat16, device=ctx.device)
    step_ms, clk, launches = timed_steps(ctx, lambda s: gl.forward(pool[s % n_pool], out), args.steps, args.warmup,
                                         gl.last_launch_count, lambda: gl.profile_begin(args.steps))
    prof = gl.profile_end()                      # [steps, 3] = route + gather, expert GEMMs, combine
    assert gl.device_status() == 0, "device error"
    total_s = float(step_ms.sum()) / 1e3
    value, t_max = aggregate(w.T * args.steps, total_s, ctx.dist, ctx.device)
    U = np.array([int((gl.route(p)["counts"] > 0).sum().item()) for p in pool], np.float64)
    flops = 2.0 * w.T * w.k * 3 * w.d * w.I
    ex_ms = prof[:, 1].astype(np.float64)
    tf = flops / (ex_ms.mean() / 1e3) / 1e12
    peak_tf = ctx.peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    fp4 = w.fmt == "nvfp4"
    wbytes = float(U.mean()) * (w.expert_bytes_nvfp4 if fp4 else w.expert_bytes_bf16)
    gbs = wbytes / (ex_ms.mean() / 1e3) / 1e9
    hbm = ctx.peaks["hbm_gbs"]
    t_flop, t_byte = flops / peak_tf / 1e12, wbytes / hbm / 1e9
    tensor = {"achieved": tf, "peak": peak_tf, "unit": "TFLOP/s", "frac": tf / peak_tf, "flops_per_launch": flops,
              "peak_note": "16-bit dense tensor peak (f16 and bf16 run at the same rate)",
              "ceiling_frac": t_flop / max(t_flop, t_byte)}
    hbm_obj = {"achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm, "bytes_per_launch": wbytes,
               "bytes_rule": ("unique active experts x " + ("10,616,832 B (NVFP4 codes + block scales)" if fp4
                                                           else "3*d*I*2 B") + " (weights read once)")}
    kname = ("grouped_gemm_fp4_kernel (gate/up + down, NVFP4 tiles widened in shared memory)" if fp4
             else "grouped_gemm_kernel (gate/up + down)")
    if t_byte > t_flop:
        # bf16 at T = 4096: the weight stream outlasts the arithmetic (128
        # FLOP/B < the ridge point), so HBM is the binding ceiling
        roof = dict(hbm_obj, kernel=kname, bound="hbm", traffic=None, peak_source=ctx.peak_src,
                    ms_per_launch=float(ex_ms.mean()), tensor=tensor)
    else:
        # NVFP4 weights are 3.55x fewer bytes: the tensor pipe is the ceiling
        roof = dict(tensor, kernel=kname, bound="tensor", traffic=None, peak_source=ctx.peak_src,
                    ms_per_launch=float(ex_ms.mean()), hbm=hbm_obj)
    kernel_ms = {"route_gather": float(prof[:, 0].mean()), "expert_gemms": float(ex_ms.mean()),
                 "combine": float(prof[:, 2].mean())}
    res = {"value": value, "unit": "tok/s", "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": t_max * 1e3 / args.steps, "roofline": roof, "kernel_ms": kernel_ms,
           "gpu_launches": launches, "clocks": clk,
           "config": workload_config(w, tokens=f"pool of {n_pool} seeded 4096-token batches",
                                     l2="flushed before every step (256 MiB write), outside the step events")}
    if fp4:
        res["dtype"] = "nvfp4 experts widened to f16/bf16 in shared memory, fp32 accumulate"
    res["e2e"] = e2e_host(ctx, w, pool_np, gl.forward_host, min(args.e2e_steps, args.steps, 20))
    if ctx.rank == 0 and not args.no_cpu_baseline:
        wr, bias = host
        res["cpu_baseline"] = (oracle_prefill_rates(w, wr, bias, pool_np[0], 64, 4) if fp4
                               else oracle_prefill_rates(w, wr, bias, pool_np[0]))
    return res


def build_stack(ctx, w):
    """The stacked workload's NVFP4 layers, quantised on the GPU from the
    seeded bf16 weights (quantisation is set-up, not part of a step)."""
    import torch
    moe = ctx.moe
    layers = []
    for li in range(w.layers):
        wr = datagen.router_weights(w, li)
        g, u, d = datagen.expert_weights(w, li)
        packs = {}
        for name, arr in (("gate", g), ("up", u), ("down", d)):
            dev = ctx.bf(arr)
            packs["q_" + name], packs["s_" + name], packs["g_" + name] = moe.quantize_nvfp4(dev)
            del dev
        del g, u, d
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        layers.append(moe.MoeLayer(ctx.bf(wr), nvfp4=packs, top_k=w.k, max_tokens=max(w.T, 16)))
        layers[-1].set_decode_path(DECODE_PATHS[ctx.args.decode_path])
    return layers


def measure_stack(ctx, w, layers):
    """8 NVFP4 layers, each RMSNorm -> MoE -> residual, in one launch per step."""
    import torch
    args, moe = ctx.args, ctx.moe
    pool_np = token_pool(w, ctx.rank)
    pool = [ctx.bf(p) for p in pool_np]
    stack = moe.MoeStack(layers)
    xcur = torch.empty((w.T, w.d), dtype=torch.bfloat16, device=ctx.device)

    def step(s):
        xcur.copy_(pool[s % POOL])
        stack.forward(xcur, out=xcur, eps=1e-6)

    step_ms, clk, launches = timed_steps(ctx, step, args.steps, args.warmup, lambda: 1)
    assert layers[0].device_status() == 0, "device error"
    total_s = float(step_ms.sum()) / 1e3
    value, t_max = aggregate(w.T * args.steps, total_s, ctx.dist, ctx.device)
    # unique experts per layer per pool batch, from an untimed layer-by-layer replay
    U = np.zeros((POOL, w.layers))
    ubuf = torch.empty((w.T, w.d), dtype=torch.bfloat16, device=ctx.device)
    for i in range(POOL):
        xcur.copy_(pool[i])
        for li, gl in enumerate(layers):
            moe.rmsnorm(xcur, 1e-6, out=ubuf)
            U[i, li] = int((gl.route(ubuf)["counts"] > 0).sum().item())
            gl.forward(ubuf, out=xcur, res=xcur)
    torch.cuda.synchronize()
    Us = U[np.arange(args.steps) % POOL]                               # [steps, layers]
    layer_bytes = Us * w.expert_bytes_nvfp4 + w.E * w.d * 2           # [steps, layers]
    step_bytes = layer_bytes.sum(1)
    hbm = ctx.peaks["hbm_gbs"]
    # the stacked launch is the step (plus one 32 KB token copy)
    ach = float(step_bytes.mean() / (step_ms.mean() / 1e3) / 1e9)
    roof = {"kernel": f"decode_layer_kernel (NVFP4, {w.layers} layers in one launch)", "bound": "hbm",
            "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm, "traffic": None,
            "peak_source": ctx.peak_src, "bytes_per_launch": float(step_bytes.mean()),
            "bytes_rule": "sum over layers of unique active experts x 10,616,832 B (NVFP4 codes + block scales) "
                          "+ router E*d*2 B",
            "unique_experts_per_layer": float(Us.mean()), "ms_per_launch": float(step_ms.mean())}
    res = {"value": value, "unit": "tok/s", "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": t_max * 1e3 / args.steps, "roofline": roof, "gpu_launches": launches, "clocks": clk,
           "dtype": "nvfp4 experts, bf16 activations, fp32 accumulate",
           "config": workload_config(w, step=f"{w.layers} x (RMSNorm, MoE, residual), one launch",
                                     l2="flushed before every step (256 MiB write), outside the step events")}
    res["e2e"] = e2e_host(ctx, w, pool_np, lambda xh, oh: stack.forward_host(xh, oh, eps=1e-6),
                          min(args.e2e_steps, args.steps))
    if ctx.rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = oracle_stack_rates(w, pool_np[0])
    stack.close()
    return res


def run_ours(args):
    import torch
    rank, world, local_rank = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device; the CUDA arm needs a GB300")
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    dist = init_dist(world, "nccl")
    import top_moe_expert_router_gb300 as moe
    moe.load()
    ctx = Ctx(args, moe, device, dist, rank, world, local_rank)
    names = ORDER if args.workload == "all" else [args.workload]
    extra_cfg = {"gate_up_layout": args.gate_up_layout, "decode_path": args.decode_path}
    results = {}

    bf16_names = [n for n in names if datagen.WORKLOADS[n].fmt == "bf16"]
    fp4_prefill = [n for n in names if datagen.WORKLOADS[n].fmt == "nvfp4" and datagen.WORKLOADS[n].layers == 1]
    if bf16_names or fp4_prefill:
        # decode and prefill share the layer's weights (seed 0, layer 0);
        # prefill adds the skewed router bias
        w0 = datagen.WORKLOADS[(bf16_names + fp4_prefill)[0]]
        if args.experts:
            w0 = dataclasses.replace(w0, E=args.experts)
        wr = datagen.router_weights(w0)
        g, u, d = datagen.expert_weights(w0)
        dev = {"wr": ctx.bf(wr), "gate": ctx.bf(g), "up": ctx.bf(u), "down": ctx.bf(d)}
        del g, u, d
        if args.gate_up_layout == "interleaved":
            dev["gate_up"] = torch.stack((dev["gate"], dev["up"]), dim=2).contiguous()   # [E, I, 2, d]
        for n in bf16_names:
            w = datagen.WORKLOADS[n]
            if args.experts:
                w = dataclasses.replace(w, E=args.experts)
            bias = datagen.router_bias(w)
            wb = None if bias is None else torch.from_numpy(bias).to(device)
            if args.gate_up_layout == "interleaved":
                gl = moe.MoeLayer(dev["wr"], w_gate_up=dev["gate_up"], w_down=dev["down"], router_bias=wb,
                                  top_k=w.k, max_tokens=max(w.T, 16))
            else:
                gl = moe.MoeLayer(dev["wr"], w_gate=dev["gate"], w_up=dev["up"], w_down=dev["down"], router_bias=wb,
                                  top_k=w.k, max_tokens=max(w.T, 16))
            gl.set_decode_path(DECODE_PATHS[args.decode_path])
            fn = measure_prefill if w.T > 16 else measure_decode
            results[n] = fn(ctx, w, gl, (wr, bias))
            gl.close()
            torch.cuda.empty_cache()
        for n in fp4_prefill:
            # the same layer's experts quantised to NVFP4 on the GPU (set-up, not timed)
            w = datagen.WORKLOADS[n]
            if args.experts:
                w = dataclasses.replace(w, E=args.experts)
            packs = {}
            for name in ("gate", "up", "down"):
                packs["q_" + name], packs["s_" + name], packs["g_" + name] = moe.quantize_nvfp4(dev[name])
            bias = datagen.router_bias(w)
            gl = moe.MoeLayer(dev["wr"], nvfp4=packs, router_bias=torch.from_numpy(bias).to(device),
                              top_k=w.k, max_tokens=w.T)
            results[n] = measure_prefill(ctx, w, gl, (wr, bias))
            gl.close()
            del packs
            torch.cuda.empty_cache()
        del dev
        torch.cuda.empty_cache()
    for n in names:
        w = datagen.WORKLOADS[n]
        if w.fmt == "nvfp4" and w.layers > 1:
            if args.experts:
                w = dataclasses.replace(w, E=args.experts)
            layers = build_stack(ctx, w)
            results[n] = measure_stack(ctx, w, layers)
            for gl in layers:
                gl.close()
            del layers
            torch.cuda.empty_cache()

    if rank == 0:
        head_name = HEADLINE if HEADLINE in results else names[0]
        head = results[head_name]
        line = {
            "metric": METRIC, "value": head["value"], "unit": "tok/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": head.get("dtype", "bf16"), "data": "synthetic",
            "config": dict(head["config"], parallelism=f"replicas x{world}, tokens split by rank", **extra_cfg),
            "roofline": head["roofline"],
            "cpu_baseline": head.get("cpu_baseline"),
            "e2e": head["e2e"],
            "gpu_launches": head["gpu_launches"],
            "clocks": head["clocks"],
            "workloads": {n: results[n] for n in names},
        }
        print(json.dumps(line))
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
