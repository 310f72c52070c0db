#!/usr/bin/env python
"""Throughput of one Mixture-of-Experts layer forward on GB300.

A step is one pass of the whole layer (router, softmax/top-8/renormalise,
permutation, expert SwiGLU FFNs, weighted combine) over one batch of
synthetic tokens with the weights resident in HBM. The default workload is
single-request decode: T=1 token, d=4096, E=256 experts, top-8, I=1536, bf16
expert weights; tokens rotate through a pool of 64 seeded N(0,1) rows and L2
is flushed (256 MiB write) before every step, so every step streams its 8
experts' weights (302 MB) from HBM.

    python bench.py [--gpus N --steps K --warmup W] [--impl reference] [--workload NAME]

Prints one JSON line. Under torchrun (N > 1) every rank holds a full layer
replica and processes its own tokens (no data-path collective); rank 0
prints the line, with the time taken as the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import datagen  # noqa: E402

METRIC = "MoE-layer tok/s; decode HBM GB/s vs ~8 TB/s; prefill TFLOP/s vs bf16 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FLUSH_BYTES = 256 << 20
POOL = 64


# ---------------------------------------------------------------------------
# helpers shared by both arms
# ---------------------------------------------------------------------------

def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="decode_t1", choices=sorted(datagen.WORKLOADS))
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=500)
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
    "decode_t1": {"bytes": 304.22e6 + 3.52e6,
                  "sources": ("top_moe_expert_router_gb300/csrc/decode_fused.cuh",
                              "top_moe_expert_router_gb300/csrc/decode_fused.cu",
                              "top_moe_expert_router_gb300/csrc/common.cuh"),
                  "sha256": ("6d828c4220d259f61ae9b2d532b6178dadd6062a79eafbf6cc60c4a174d426cb",
                             "1d39e048978fb78a6191116a4ce545b150e1efd7577999126a1f97db51c5e355",
                             "7dd70629dc137bc914f03f15ee8566d22afb9a3e9583266dc02b5c21e57e759f")},
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


# ---------------------------------------------------------------------------
# CPU oracle: the reference arm and the cpu_baseline leg
# ---------------------------------------------------------------------------

def oracle_token_rate(host_layer, x_tokens: np.ndarray, budget_s: float = 20.0):
    """Oracle throughput (tok/s) on a bounded sample of tokens, all threads."""
    import oracle
    n = x_tokens.shape[0]
    t0 = time.perf_counter()
    host_layer.forward(x_tokens)
    dt = time.perf_counter() - t0
    return n / dt, dt, oracle.max_threads()


def run_reference(args):
    """The reference arm: the CPU oracle timed on the host cores."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    w = datagen.WORKLOADS[args.workload]
    if w.fmt != "bf16" or w.layers != 1:
        print(json.dumps({"impl": "reference", "unavailable": "reference arm runs the bf16 single-layer workloads"}))
        return 0
    pool = [datagen.tokens(w, w.T, start_row=i * w.T) for i in range(POOL)]
    wr = datagen.router_weights(w)
    bias = datagen.router_bias(w)
    lg = oracle.router_logits(np.concatenate(pool), wr, bias)
    ids, _, _ = oracle.select_topk(lg, w.k)
    g, u, d = datagen.expert_weights(w, experts=np.unique(ids))
    L = oracle.Layer(wr, g, u, d, router_bias=bias, k=w.k)
    # one step = the oracle forward of one batch; bound the whole run to ~150 s
    t0 = time.perf_counter()
    L.forward(pool[0])
    t_step = time.perf_counter() - t0
    tokens_per_step = w.T
    sample = "full batch per step"
    if t_step * (args.steps + args.warmup) > 150.0 and w.T > 1:
        tokens_per_step = max(1, int(w.T * 150.0 / (t_step * (args.steps + args.warmup))))
        sample = f"first {tokens_per_step} of {w.T} tokens per step"
    for s in range(args.warmup):
        L.forward(pool[s % POOL][:tokens_per_step])
    t0 = time.perf_counter()
    for s in range(args.steps):
        L.forward(pool[s % POOL][:tokens_per_step])
    total = time.perf_counter() - t0
    value = tokens_per_step * args.steps / total
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

def build_gpu_layer(moe, w: datagen.Workload, device, layer: int = 0):
    import torch
    wr = datagen.router_weights(w, layer)
    bias = datagen.router_bias(w, layer)
    g, u, d = datagen.expert_weights(w, layer)

    def bf(a):
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)

    gl = moe.MoeLayer(bf(wr), w_gate=bf(g), w_up=bf(u), w_down=bf(d),
                      router_bias=None if bias is None else torch.from_numpy(bias).to(device),
                      top_k=w.k, max_tokens=max(w.T, 16))
    return gl, (wr, bias, g, u, d)


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
    w = datagen.WORKLOADS[args.workload]
    if args.experts:
        import dataclasses
        w = dataclasses.replace(w, E=args.experts)
    if w.layers != 1 or w.fmt != "bf16":
        return run_stack(args, w, moe, device, dist, rank, world, local_rank)
    gl, host = build_gpu_layer(moe, w, device)
    # each rank draws its own token pool (distinct rows of the token stream)
    pool_np = [datagen.tokens(w, w.T, start_row=(rank * POOL + i) * w.T) for i in range(POOL)]
    pool = [torch.from_numpy(p.view(np.int16)).view(torch.bfloat16).to(device) for p in pool_np]
    out = torch.empty((w.T, w.d), dtype=torch.bfloat16, device=device)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()

    for s in range(args.warmup):
        flush.zero_()
        gl.forward(pool[s % POOL], out)
    torch.cuda.synchronize()
    assert gl.device_status() == 0, "device error during warm-up"

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    gl.profile_begin(args.steps)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank)
    clocks.start()
    launches = 0
    for s in range(args.steps):
        flush.zero_()
        evs[s][0].record(stream)
        gl.forward(pool[s % POOL], out)
        evs[s][1].record(stream)
        launches += gl.last_launch_count()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()
    step_ms = np.array([a.elapsed_time(b) for a, b in evs])
    # decode: [steps, 4] = route, gate/up, down, combine
    # prefill: [steps, 3] = route + gather, grouped GEMMs, combine
    prof = gl.profile_end()
    status = gl.device_status()
    assert status == 0, f"device error {status}"
    total_s = float(step_ms.sum()) / 1e3
    value, t_max = aggregate(w.T * args.steps, total_s, dist, device)

    # unique experts per step (for the bytes each step must stream)
    uniq = []
    for p in pool:
        r = gl.route(p)
        uniq.append(int((r["counts"] > 0).sum().item()))
    U = np.array([uniq[s % POOL] for s in range(args.steps)], np.float64)
    eb = w.expert_bytes_bf16
    gateup_bytes = U * 2 * w.I * w.d * 2                # W_gate + W_up rows of the active experts
    layer_bytes = U * eb + w.E * w.d * 2                # all active expert weights + router
    peaks, peak_src = load_peaks()
    hbm = peaks["hbm_gbs"]
    step_gbs = float(layer_bytes.sum() / total_s / 1e9)
    if prof.shape[1] == 1:
        # the whole layer is one persistent kernel: router, routing, expert stream, combine
        ly_ms = prof[:, 0].astype(np.float64)
        ly_gbs = float(layer_bytes.mean() / (ly_ms.mean() / 1e3) / 1e9)
        roofline = {"kernel": "decode_layer_kernel", "bound": "hbm", "achieved": ly_gbs, "peak": hbm,
                    "unit": "GB/s", "frac": ly_gbs / hbm,
                    "traffic": measured_traffic(args.workload) if not args.experts else None,
                    "peak_source": peak_src,
                    "bytes_per_launch": float(layer_bytes.mean()), "ms_per_launch": float(ly_ms.mean())}
        kernel_ms = {"layer": float(ly_ms.mean())}
    elif prof.shape[1] == 4:
        gu_ms = prof[:, 1].astype(np.float64)
        gu_gbs = float(gateup_bytes.mean() / (gu_ms.mean() / 1e3) / 1e9)
        roofline = {"kernel": "decode_gateup_kernel", "bound": "hbm", "achieved": gu_gbs, "peak": hbm,
                    "unit": "GB/s", "frac": gu_gbs / hbm, "traffic": None, "peak_source": peak_src,
                    "bytes_per_launch": float(gateup_bytes.mean()), "ms_per_launch": float(gu_ms.mean())}
        kernel_ms = {"route": float(prof[:, 0].mean()), "gateup": float(gu_ms.mean()),
                     "down": float(prof[:, 2].mean()), "combine": float(prof[:, 3].mean())}
    else:
        # expert GEMMs: 2 FLOP x rows (T*k) x (2*d*I gate/up + d*I down)
        flops = 2.0 * w.T * w.k * 3 * w.d * w.I
        ex_ms = prof[:, 1].astype(np.float64)
        tf = flops / (ex_ms.mean() / 1e3) / 1e12
        peak_tf = peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops"))
        roofline = {"kernel": "grouped_gemm_kernel (gate/up + down)", "bound": "tensor", "achieved": tf,
                    "peak": peak_tf, "unit": "TFLOP/s", "frac": tf / peak_tf, "traffic": None,
                    "peak_source": peak_src, "flops_per_launch": flops, "ms_per_launch": float(ex_ms.mean()),
                    "hbm_frac_of_expert_stage": float(U.mean() * eb / (ex_ms.mean() / 1e3) / 1e9 / hbm)}
        kernel_ms = {"route_gather": float(prof[:, 0].mean()), "expert_gemms": float(ex_ms.mean()),
                     "combine": float(prof[:, 2].mean())}

    # end to end through the C ABI from pinned host memory
    e2e = None
    if rank == 0 or True:
        xh = [torch.from_numpy(p.view(np.int16)).view(torch.bfloat16).pin_memory() for p in pool_np]
        oh = torch.empty((w.T, w.d), dtype=torch.bfloat16).pin_memory()
        for s in range(5):
            gl.forward_host(xh[s % POOL], oh)
        n_e2e = min(args.e2e_steps, args.steps)
        t0 = time.perf_counter()
        for s in range(n_e2e):
            gl.forward_host(xh[s % POOL], oh)
        e2e_s = time.perf_counter() - t0
        e2e_v, _ = aggregate(w.T * n_e2e, e2e_s, dist, device)
        e2e = {"value": e2e_v, "unit": "tok/s", "h2d_bytes_per_step": w.T * w.d * 2,
               "d2h_bytes_per_step": w.T * w.d * 2, "steps": n_e2e,
               "note": "moe_forward_host: H2D copy, layer, D2H copy, stream sync per step; no L2 flush"}

    cpu = None
    if rank == 0 and world >= 1 and not args.no_cpu_baseline:
        import oracle
        wr, bias, g, u, d = host
        L = oracle.Layer(wr, g, u, d, router_bias=bias, k=w.k)
        n_tok = 32
        xs = np.concatenate(pool_np)[:n_tok]
        rate, dt, cores = oracle_token_rate(L, xs)
        cpu = {"value": rate, "unit": "tok/s", "cores": cores, "kind": "oracle",
               "sample": f"{n_tok} tokens of the pool, full layer each, one oracle call ({dt:.1f} s)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t_max * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config(w, parallelism=f"replicas x{world}, tokens split by rank",
                                      l2="flushed before every step (256 MiB write), outside the step events"),
            "roofline": roofline,
            "step_roofline": {"bound": "hbm", "achieved": step_gbs, "peak": hbm, "unit": "GB/s",
                              "frac": step_gbs / hbm, "bytes_per_step": float(layer_bytes.mean()),
                              "unique_experts_per_step": float(U.mean()), "kernel_ms": kernel_ms},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clk,
        }
        print(json.dumps(line))
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def run_stack(args, w, moe, device, dist, rank, world, local_rank):
    """Stacked NVFP4 decode: every step runs the token batch through all
    layers, each RMSNorm -> MoE (NVFP4 experts) -> residual add."""
    import torch

    def bf(a):
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)

    layers, host_routers = [], []
    for li in range(w.layers):
        wr = datagen.router_weights(w, li)
        g, u, d = datagen.expert_weights(w, li)
        packs = {}
        for name, arr in (("gate", g), ("up", u), ("down", d)):
            dev = bf(arr)
            q, s, gs = moe.quantize_nvfp4(dev)
            packs["q_" + name], packs["s_" + name], packs["g_" + name] = q, s, gs
            del dev
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        layers.append(moe.MoeLayer(bf(wr), nvfp4=packs, top_k=w.k, max_tokens=max(w.T, 16)))
        host_routers.append(wr)
    pool_np = [datagen.tokens(w, w.T, start_row=(rank * POOL + i) * w.T) for i in range(POOL)]
    pool = [bf(p) for p in pool_np]
    xcur = torch.empty((w.T, w.d), dtype=torch.bfloat16, device=device)
    ubuf = torch.empty_like(xcur)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()

    # the whole stack in one launch when the batch fits (T <= 8)
    stack = moe.MoeStack(layers) if w.T <= 8 else None

    def step(x0, route_log=None):
        xcur.copy_(x0)
        if stack is not None and route_log is None:
            stack.forward(xcur, out=xcur, eps=1e-6)
            return
        for gl in layers:
            moe.rmsnorm(xcur, 1e-6, out=ubuf)
            if route_log is not None:
                route_log.append(int((gl.route(ubuf)["counts"] > 0).sum().item()))
            gl.forward(ubuf, out=xcur, res=xcur)

    for s in range(args.warmup):
        flush.zero_()
        step(pool[s % POOL])
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for gl in layers:
        gl.profile_begin(args.steps)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank)
    clocks.start()
    launches = 0
    for s in range(args.steps):
        flush.zero_()
        evs[s][0].record(stream)
        step(pool[s % POOL])
        evs[s][1].record(stream)
        launches += 1 if stack is not None else w.layers * (1 + layers[0].last_launch_count())
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()
    step_ms = np.array([a.elapsed_time(b) for a, b in evs])
    profs = [gl.profile_end() for gl in layers]             # each [steps, 4] (empty for the stacked launch)
    for gl in layers:
        assert gl.device_status() == 0
    total_s = float(step_ms.sum()) / 1e3
    value, t_max = aggregate(w.T * args.steps, total_s, dist, device)
    # unique experts per layer per step, from an untimed replay of the pool
    U = np.zeros((POOL, w.layers))
    for i in range(POOL):
        log = []
        step(pool[i], route_log=log)
        U[i] = log
    torch.cuda.synchronize()
    Us = np.array([U[s % POOL] for s in range(args.steps)])      # [steps, layers]
    eb = w.expert_bytes_nvfp4
    peaks, peak_src = load_peaks()
    hbm = peaks["hbm_gbs"]
    layer_bytes = Us * eb + w.E * w.d * 2                           # [steps, layers]
    if stack is not None:
        # one stacked launch per step: its bytes are all layers' bytes, its
        # time the step's (the step adds one 32 KB token copy)
        kname = f"decode_layer_kernel (NVFP4, {w.layers} layers in one launch)"
        k_bytes = layer_bytes.sum(1, keepdims=True)
        k_ms = step_ms[:, None].astype(np.float64)
        kms = {"stack": float(k_ms.mean()), "per_layer": float(k_ms.mean() / w.layers)}
    elif profs[0].shape[1] == 1:
        kname = "decode_layer_kernel (NVFP4)"
        k_bytes = layer_bytes
        k_ms = np.stack([p[:, 0] for p in profs], axis=1).astype(np.float64)
        kms = {"layer": float(k_ms.mean())}
    else:
        kname = "decode_gateup_kernel (NVFP4)"
        k_bytes = Us * 2 * w.I * (w.d // 2 + w.d // 16)             # gate + up codes and scales
        k_ms = np.stack([p[:, 1] for p in profs], axis=1).astype(np.float64)
        kms = {name: float(np.mean([p[:, i].mean() for p in profs]))
               for i, name in enumerate(["route", "gateup", "down", "combine"])}
    gu_bytes, gu_ms = k_bytes, k_ms
    gu_gbs = float(gu_bytes.sum() / (gu_ms.sum() / 1e3) / 1e9)
    step_bytes = layer_bytes.sum(1)
    step_gbs = float(step_bytes.sum() / total_s / 1e9)
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t_max * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4 experts, bf16 activations, fp32 accumulate",
            "data": "synthetic",
            "config": workload_config(w, parallelism=f"replicas x{world}",
                                      l2="flushed before every step (256 MiB write), outside the step events",
                                      step="8 x (RMSNorm, MoE, residual)" + (", one launch" if stack is not None else "")),
            "roofline": {"kernel": kname, "bound": "hbm", "achieved": gu_gbs, "peak": hbm,
                         "unit": "GB/s", "frac": gu_gbs / hbm, "traffic": None, "peak_source": peak_src,
                         "bytes_per_launch": float(gu_bytes.mean()), "ms_per_launch": float(gu_ms.mean())},
            "step_roofline": {"bound": "hbm", "achieved": step_gbs, "peak": hbm, "unit": "GB/s",
                              "frac": step_gbs / hbm, "bytes_per_step": float(step_bytes.mean()),
                              "unique_experts_per_layer": float(Us.mean()), "kernel_ms_per_layer": kms},
            "cpu_baseline": None,
            "e2e": None,
            "gpu_launches": launches,
            "clocks": clk,
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
