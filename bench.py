#!/usr/bin/env python3
"""Benchmark of the sparse MoE FFN layer forward on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]

Default workload: the Mixtral-shaped top-2 layer (T=16384, d=4096, E=8, k=2,
SwiGLU d_ff=14336, renormalised gates, no capacity limit, bf16 experts, fp32
router), the largest of the layer configurations, on seeded synthetic inputs;
--config switch|deepseek|skewed|decode|decode_nocap|tiny selects another.
A step is one pass of the whole layer (router, dispatch, grouped GEMM,
combine) through the C ABI, timed with CUDA events on the launching stream;
L2 is flushed (a 2x-L2 buffer is written) between steps, outside the timed
events.  Prints one JSON line (rank 0).

--impl reference times the fp64 CPU oracle on the host cores instead: every
step routes all T tokens and runs the experts on a seeded sample of tokens,
the expert part extrapolated per kept slot to the whole batch.

Under torchrun (N > 1) every rank runs its own replica of the workload (the
layer shards over tokens with no data-path exchange); timings are reduced with
a max over ranks.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer fwd tokens/s on 1 B300; % of bf16 TC peak and HBM GB/s"
UNIT = "tokens/s"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="mixtral")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override T (a smaller case of the same layer shape, e.g. for ncu captures)")
    ap.add_argument("--d-ff", type=int, default=None,
                    help="override d_ff (router, dispatch and combine do not depend on it)")
    ap.add_argument("--profile-only", action="store_true",
                    help="only run warm-up + steps forwards through moe_forward (direct launches, no "
                         "timing, no e2e, no CPU baseline): the command ncu captures")
    ap.add_argument("--clocks-csv", default=None,
                    help="where the nvidia-smi clock samples of the timed region go (default: a temp file)")
    ap.add_argument("--impl", default="b300", choices=["b300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--noisy", action="store_true",
                    help="noisy top-k gating (training-mode router; noise floor 0.01)")
    ap.add_argument("--int8", action="store_true",
                    help="int8 expert weights with per-row scales (quantised by the library)")
    ap.add_argument("--int4", action="store_true",
                    help="4-bit expert weights with scales per group of 128 inputs (quantised by the library)")
    ap.add_argument("--ep", type=int, default=None,
                    help="run the layer expert-parallel over this many ranks emulated on the GPU")
    ap.add_argument("--backward", action="store_true",
                    help="time a training step instead: moe_forward + moe_backward")
    ap.add_argument("--split-router-per-call", action="store_true",
                    help="split the router weights on every call instead of once per weight update")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch each stage directly instead of replaying a captured CUDA graph")
    return ap.parse_args()


def workload_name(cfg) -> str:
    cap = "none" if cfg.cf is None else f"{cfg.cf:g}"
    shared = f"+{cfg.S}shared" if cfg.S else ""
    noisy = f", noisy top-k gating (noise floor {cfg.noise_min_std:g})" if cfg.noisy else ""
    wq = {"int8": " with int8 weights (per-row scales)",
          "int4": " with 4-bit weights (scales per group of 128 inputs)"}.get(cfg.weights, "")
    return (f"{cfg.name} MoE FFN layer: T={cfg.T} d_model={cfg.d} E={cfg.E}{shared} k={cfg.k} "
            f"d_ff={cfg.F} {cfg.act} capacity_factor={cap} {cfg.dtype} experts{wq}, fp32 router{noisy}")


def bench_config(args):
    from sparse_mixture_experts_scan_b300 import config
    kw = {}
    if args.noisy:
        kw.update(noisy=True, noise_min_std=0.01)
    if args.int8:
        kw.update(weights="int8")
    if args.int4:
        kw.update(weights="int4")
    if args.tokens is not None:
        kw.update(T=args.tokens)
    if args.d_ff is not None:
        kw.update(F=args.d_ff)
    return config(args.config, **kw)


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p["bf16_tflops_sustained"], "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
                "source": "fallback"}


def max_over_ranks(value: float, device=None) -> float:
    """The maximum of `value` over all ranks (the value itself without a process group).

    Works with any torch.distributed backend: NCCL on the GPU machine (device = the rank's
    GPU), gloo on CPU (device None)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world: int, tokens_per_rank: int, ms: float) -> float:
    """Whole-job tokens/s of `world` replicas that each process `tokens_per_rank` tokens in
    `ms` milliseconds (the max over ranks)."""
    return world * tokens_per_rank / (ms * 1e-3)


def clocks_path(args, rank: int) -> str:
    if args.clocks_csv:
        return args.clocks_csv if rank == 0 else f"{args.clocks_csv}.rank{rank}"
    import tempfile
    return os.path.join(tempfile.gettempdir(), f"moe_bench_clocks_rank{rank}.csv")


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, path: str):
        self.index, self.path, self.proc = index, path, None

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm, mx, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        top = max(power)
        loaded = [s for s, p in zip(sm, power) if p >= 0.5 * top] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm), "power_w_max": top}


class NvmlSampler:
    """SM clock and clock-event reasons from the driver's NVML library (the library
    nvidia-smi reads) every ~1 ms: a timed region of a few milliseconds is shorter
    than nvidia-smi's sampling interval.  Loaded with ctypes (no Python binding needed)."""

    CLOCK_SM = 1
    REASONS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
               "hw_thermal_slowdown": 0x40}

    def __init__(self, index: int):
        self.index, self.samples, self.ok, self.error = index, [], False, None

    def __enter__(self):
        import ctypes
        import threading
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                raise OSError("nvmlInit_v2 failed")
            h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)) != 0:
                raise OSError("nvmlDeviceGetHandleByIndex_v2 failed")
            self.get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint()
            lib.nvmlDeviceGetMaxClockInfo(h, ctypes.c_int(self.CLOCK_SM), ctypes.byref(mx))
            self.lib, self.h, self.max_mhz, self.ct = lib, h, mx.value, ctypes
            self.ok = True
        except (OSError, AttributeError) as exc:
            self.error = str(exc)
            return self
        self.stop = threading.Event()

        def loop():
            while not self.stop.is_set():
                self._sample()
                time.sleep(0.001)

        self._sample()  # at least one sample at the start of the region
        self.th = threading.Thread(target=loop, daemon=True)
        self.th.start()
        return self

    def _sample(self):
        ct = self.ct
        clk, rs = ct.c_uint(), ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, ct.c_int(self.CLOCK_SM), ct.byref(clk)) == 0 and \
                self.get_reasons(self.h, ct.byref(rs)) == 0:
            self.samples.append((clk.value, rs.value))

    def __exit__(self, *exc):
        if self.ok:
            self.stop.set()
            self.th.join()

    def summary(self):
        if not self.ok or not self.samples:
            return None
        reasons = sorted(n for n, bit in self.REASONS.items() if any(r & bit for _, r in self.samples))
        return {"sm_mhz": statistics.median(c for c, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(self.samples), "source": "NVML every ~1 ms"}


# --------------------------------------------------------------------------- oracle (CPU)

def oracle_step(cfg, cpu_inp, n_sample: int, seed: int = 7):
    """One bounded oracle pass: route all T tokens, experts on a token sample.

    Returns (seconds-equivalent for the whole batch, description, threads)."""
    import numpy as np
    from oracle import moe_oracle as orc

    t0 = time.perf_counter()
    noise = ((cpu_inp["W_noise"], cpu_inp["b_noise"], cpu_inp["noise_eps"], cfg.noise_min_std)
             if cfg.noisy else None)
    r = orc.route(cpu_inp["x"], cpu_inp["W_gate"], cpu_inp["b_gate"], k=cfg.k,
                  renormalize=cfg.renormalize, cf=cfg.cf, noise=noise)
    t_route = time.perf_counter() - t0
    rng = np.random.default_rng(seed)
    tok = np.sort(rng.choice(cfg.T, size=min(n_sample, cfg.T), replace=False))
    t1 = time.perf_counter()
    orc.output_rows(cpu_inp["x"], cpu_inp["W1"], cpu_inp["W3"], cpu_inp["W2"], cpu_inp["b1"],
                    cpu_inp["b2"], r.idx, r.gates, r.dropped, E=cfg.E, S=cfg.S,
                    act_name=cfg.act, residual_mode=cfg.residual_mode, tokens=tok)
    t_ffn = time.perf_counter() - t1
    kept_all = int((r.dropped == 0).sum()) + cfg.S * cfg.T
    kept_smp = int((r.dropped[tok] == 0).sum()) + cfg.S * len(tok)
    scale = kept_all / max(kept_smp, 1)
    secs = t_route + t_ffn * scale
    desc = (f"routing of all {cfg.T} tokens timed directly ({t_route:.2f} s); experts on a seeded "
            f"sample of {len(tok)} tokens ({kept_smp} kept slots, {t_ffn:.2f} s) extrapolated "
            f"per kept slot to {kept_all} slots")
    return secs, desc, orc.num_threads()


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    from sparse_mixture_experts_scan_b300 import make_inputs

    cfg = bench_config(args)
    inp = make_inputs(cfg, 0, device="cpu")
    # size the per-step token sample so that warm-up + timed steps take ~2 minutes
    t0 = time.perf_counter()
    oracle_step(cfg, inp, 16)
    probe = time.perf_counter() - t0
    per_step_budget = 120.0 / max(args.steps + args.warmup, 1)
    n_sample = int(max(16, min(cfg.T, 16 * per_step_budget / max(probe, 1e-3))))
    for _ in range(max(args.warmup - 1, 0)):
        oracle_step(cfg, inp, n_sample)
    secs, descs, threads = [], None, 1
    t_wall = time.perf_counter()
    for _ in range(args.steps):
        s, descs, threads = oracle_step(cfg, inp, n_sample)
        secs.append(s)
    wall = time.perf_counter() - t_wall
    per_step = sum(secs) / len(secs)  # seconds the whole batch would take (extrapolated)
    value = cfg.T / per_step
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        # wall time each step actually spent (routing of all T tokens + the expert sample)
        "ms_per_step": wall / max(args.steps, 1) * 1e3,
        # the whole batch's time, the expert part extrapolated per kept slot: value = T / this
        "extrapolated_ms_per_step": per_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; shapes and distributions of the workload)",
        "config": {"workload": workload_name(cfg), "tokens_per_step": cfg.T},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": descs + f"; {args.steps} steps in {wall:.1f} s wall; value = T / "
                                           "extrapolated_ms_per_step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------- GPU arm

def algorithmic_gemm_work(cfg, out, direct=False):
    """Bytes and flops the grouped-GEMM stage must move/do for this batch.

    Bytes: weights of every expert that received >= 1 kept row (W1, W3, W2), the
    permuted activations read once, the hidden activations written and read once,
    the expert outputs written once (shared experts: x read once, their S * d_ff hidden
    columns written and read once and one summed output row per token; with the combine
    finished in the stage, the kept rows of y plus their token and gate).  Flops: 2 per
    multiply-add on kept rows only."""
    import torch
    kept = (out["dropped"] == 0)
    idx = out["expert_idx"].long()
    kept_per_e = torch.zeros(cfg.E, dtype=torch.long, device=idx.device)
    kept_per_e.scatter_add_(0, idx[kept], torch.ones_like(idx[kept]))
    touched = int((kept_per_e > 0).sum()) + cfg.S
    rows = int(kept.sum())
    esz = 2 if cfg.dtype == "bf16" else 4
    nmat = 3 if cfg.act == "swiglu" else 2
    if cfg.weights == "int8":  # 1-byte weights and one fp32 scale per output row
        w_bytes = touched * (nmat * cfg.d * cfg.F + 4 * ((nmat - 1) * cfg.F + cfg.d))
    elif cfg.weights == "int4":  # half-byte weights and one fp32 scale per 128 inputs
        w_bytes = touched * (nmat * cfg.d * cfg.F // 2 + 4 * nmat * cfg.d * cfg.F // 128)
    else:
        w_bytes = touched * nmat * cfg.d * cfg.F * esz
    srows = cfg.S * cfg.T
    act_bytes = (rows * (cfg.d + 2 * cfg.F + cfg.d) + (2 * cfg.T * cfg.d if cfg.S else 0)
                 + srows * 2 * cfg.F) * esz + (rows * 8 if direct else 0)
    flops = cfg.expert_flops(rows)
    return {"bytes": w_bytes + act_bytes, "weight_bytes": w_bytes, "flops": flops,
            "kept_rows": rows, "touched_experts": touched}


def direct_combine(cfg, args) -> bool:
    """True when the library finishes the combine inside the expert stage: a top-1 bf16
    layer on the fused tensor-core kernel without shared experts or the residual on every
    token (the GEMM2 epilogue writes y, the dispatch copies the dropped tokens)."""
    return (cfg.k == 1 and cfg.S == 0 and cfg.residual_mode == 0 and cfg.dtype == "bf16"
            and cfg.weights == "dtype" and not getattr(args, "ep", None) and not getattr(args, "backward", False))


def stage_bytes(cfg, out, gemm, direct=False):
    """Minimum HBM bytes of the memory-bound stages (router, dispatch, combine).  With the
    combine finished in the expert stage, the combine moves nothing and the dispatch also
    copies the dropped tokens' rows into y."""
    esz = 2 if cfg.dtype == "bf16" else 4
    T, d, k, E = cfg.T, cfg.d, cfg.k, cfg.E
    rows = gemm["kept_rows"]
    router = T * d * esz + E * d * 4 + T * k * 8
    if cfg.noisy:
        router += E * d * 4 + T * E * 4  # W_noise and the normal draws
    dispatch = T * k * 4 + rows * d * esz * 2 + T * k * (1 + 4 + 4)
    pass_tok = int((out["dropped"].bool().all(dim=1)).sum()) if cfg.residual_mode == 0 else T
    if direct:
        dispatch += 2 * pass_tok * d * esz + rows * 8
        return {"moe_router": router, "moe_dispatch": dispatch, "moe_combine": 0}
    combine = rows * d * esz + T * d * esz + pass_tok * d * esz + T * k * 8 + \
        (T * d * esz if cfg.S else 0)
    return {"moe_router": router, "moe_dispatch": dispatch, "moe_combine": combine}


def traffic_from_profiles(kernel_file: str, workload: str):
    """DRAM bytes per launch recorded by an ncu capture, if the kernel source is unchanged."""
    path = os.path.join(ROOT, "profiles", "traffic.md")
    src = os.path.join(ROOT, "sparse_mixture_experts_scan_b300", "csrc", kernel_file)
    if not os.path.exists(path) or not os.path.exists(src):
        return None
    with open(src, "rb") as f:
        h = hashlib.sha256(f.read()).hexdigest()[:16]
    pat = re.compile(r"^traffic\s+(\S+)\s+(\S+)\s+bytes_per_step=(\d+)\s+source=([0-9a-f]+)")
    with open(path) as f:
        for line in f:
            m = pat.match(line.strip())
            if m and m.group(1) == kernel_file and m.group(2) == workload and m.group(4) == h:
                return int(m.group(3))
    return None


def run_gpu(args):
    import torch
    import torch.distributed as dist

    from sparse_mixture_experts_scan_b300 import MoELayer, _lib, make_inputs

    world, rank, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    cfg = bench_config(args)
    inp = make_inputs(cfg, seed=rank, device=dev)
    if cfg.weights in ("int8", "int4"):
        from sparse_mixture_experts_scan_b300 import quantize_expert_weights
        inp = quantize_expert_weights(inp, bits=8 if cfg.weights == "int8" else 4)
    # bf16 layers: the router weights' three-term split is made once, as after a weight update
    prepared = cfg.dtype == "bf16" and not args.split_router_per_call
    layer = MoELayer(cfg, inp, device=dev, ep_ranks=args.ep, prepared_router=prepared)
    stream = torch.cuda.current_stream(dev)
    # an expert-parallel layer runs only the whole forward: its stage pass is that one call
    stages = ["moe_forward"] if args.ep else ["moe_router", "moe_dispatch", "moe_grouped_gemm", "moe_combine"]
    if args.profile_only:
        # the command ncu captures: warm-up + steps forwards, direct launches, nothing else
        for _ in range(max(args.warmup, 0) + args.steps):
            layer.run("moe_forward", stream)
        torch.cuda.synchronize()
        status = layer.device_status()
        if rank == 0:
            print(json.dumps({"profile_only": True, "workload": workload_name(cfg),
                              "forwards": max(args.warmup, 0) + args.steps, "device_status": status}),
                  flush=True)
        return 0 if status == 0 else 1

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 64 << 20), dtype=torch.uint8, device=dev)

    def stage_step(evs=None):
        for i, st_name in enumerate(stages):
            if evs is not None:
                evs[i].record(stream)
            layer.run(st_name, stream)
        if evs is not None:
            evs[-1].record(stream)

    def full_step():
        layer.run("moe_forward", stream)

    n_launch0 = _lib.moe_kernel_launches()
    for _ in range(max(args.warmup, 0)):
        flush.zero_()
        full_step()
    torch.cuda.synchronize()
    # kernels one moe_forward enqueues, from the library's own launch counter
    launches_per_step = (_lib.moe_kernel_launches() - n_launch0) // max(args.warmup, 1)

    if not args.no_graph:
        # CUDA graphs of the library's calls (it only enqueues kernels, so it is
        # capturable): one of the whole forward (kernels chained by programmatic
        # dependent launch) and one per stage for the stage breakdown
        g_full = torch.cuda.CUDAGraph()
        n_launch0 = _lib.moe_kernel_launches()
        with torch.cuda.graph(g_full):
            layer.run("moe_forward")
        launches_per_step = _lib.moe_kernel_launches() - n_launch0  # kernels in the replayed graph
        g_stage = []
        for st_name in stages:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                layer.run(st_name)
            g_stage.append(g)
        torch.cuda.synchronize()

        def full_step():  # noqa: F811
            g_full.replay()

        def stage_step(evs=None):  # noqa: F811
            for i, g in enumerate(g_stage):
                if evs is not None:
                    evs[i].record(stream)
                g.replay()
            if evs is not None:
                evs[-1].record(stream)

        for _ in range(2):
            flush.zero_()
            full_step()
            stage_step()
        torch.cuda.synchronize()

    K = args.steps
    ev_step = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)] for _ in range(K)]
    clk = ClockSampler(dev.index, clocks_path(args, rank))
    nvml = NvmlSampler(dev.index)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with clk, nvml:
        t_wall0 = time.perf_counter()
        # timed region: K whole-layer steps, events only at step boundaries
        for i in range(K):
            flush.zero_()
            ev_step[i][0].record(stream)
            full_step()
            ev_step[i][1].record(stream)
        if nvml.ok:
            nvml._sample()  # while the last steps are still running on the device
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        t_wall = time.perf_counter() - t_wall0
        # second timed pass: the same K steps with events between the four stages
        for i in range(K):
            flush.zero_()
            stage_step(evs[i])
        torch.cuda.synchronize()
    stage_ms = {st_name: 0.0 for st_name in stages}
    for i in range(K):
        for j, st_name in enumerate(stages):
            stage_ms[st_name] += evs[i][j].elapsed_time(evs[i][j + 1])
    stage_ms = {k_: v / K for k_, v in stage_ms.items()}
    ms_step = sum(a.elapsed_time(b) for a, b in ev_step) / K
    if world > 1:
        ms_step = max_over_ranks(ms_step, dev)
    value = replica_throughput(world, cfg.T, ms_step)

    out = layer.out
    direct = direct_combine(cfg, args)
    gemm = algorithmic_gemm_work(cfg, out, direct)
    sbytes = stage_bytes(cfg, out, gemm, direct)
    pk = peaks()
    g_ms = stage_ms.get("moe_grouped_gemm", ms_step)
    hbm_bound = gemm["bytes"] == 0 or \
        gemm["flops"] / gemm["bytes"] < pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    if gemm["bytes"] == 0 or g_ms <= 0:
        # capacity 0: every slot is dropped, the expert stage has no work
        roof = {"bound": "hbm", "achieved": 0.0, "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": 0.0,
                "note": "no kept rows: the expert stage does no work"}
    elif hbm_bound:
        achieved = gemm["bytes"] / (g_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"]}
    else:
        achieved = gemm["flops"] / (g_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / pk["bf16_tflops"],
                # the same kernel against the power-capped, seconds-long cuBLAS figure
                "peak_sustained": pk["bf16_tflops_sustained"],
                "frac_sustained": achieved / pk["bf16_tflops_sustained"]}
    wl_key = args.config + ("_noisy" if cfg.noisy else "")
    if args.tokens is not None or args.d_ff is not None:
        wl_key += f"_T{cfg.T}_F{cfg.F}"
    fused = cfg.dtype == "bf16"
    if args.ep:
        wl_key += f"_ep{args.ep}"
        tr = None
        kname = (f"the whole expert-parallel forward over {args.ep} emulated ranks (moe_forward_ep; the "
                 "owners' expert kernels dominate)")
    elif cfg.weights in ("int8", "int4"):
        wl_key += "_" + cfg.weights
        max_rows = min(cfg.T, int(cfg.T * cfg.cf / cfg.E)) if cfg.cf else cfg.T
        if cfg.weights == "int4" or max_rows <= 128:
            tr = traffic_from_profiles("grouped_gemm_wq.cu", wl_key)
            kname = (f"moe_grouped_gemm stage: two k_grouped_gemm_wq launches ({cfg.weights} weights converted "
                     "into tensor memory, tcgen05 with A from TMEM)")
        else:
            tr = traffic_from_profiles("grouped_gemm_q8.cu", wl_key)
            kname = "moe_grouped_gemm stage: two k_grouped_gemm_q8 launches (int8 weights, tcgen05)"
    else:
        tr = traffic_from_profiles("ffn_fused_tc.cu" if fused else "grouped_gemm_ffma.cu", wl_key)
        kname = ("moe_grouped_gemm stage: k_ffn_fused_tc (both expert layers, one persistent tcgen05 launch)"
                 + (" + shared-expert k_grouped_gemm_tc launches" if cfg.S else "")) if fused else \
            "moe_grouped_gemm stage: k_grouped_gemm_ffma (fp32)"
    roof.update({"traffic": tr, "kernel": kname,
                 "algorithmic_bytes": gemm["bytes"], "algorithmic_flops": gemm["flops"],
                 "touched_experts": gemm["touched_experts"], "kept_rows": gemm["kept_rows"],
                 "peak_source": pk["source"] + " (burst)",
                 "tensor_tflops": gemm["flops"] / max(g_ms * 1e-3, 1e-12) / 1e12,
                 "tensor_frac": gemm["flops"] / max(g_ms * 1e-3, 1e-12) / 1e12 / pk["bf16_tflops"],
                 "hbm_gbs": gemm["bytes"] / max(g_ms * 1e-3, 1e-12) / 1e9,
                 "hbm_frac": gemm["bytes"] / max(g_ms * 1e-3, 1e-12) / 1e9 / pk["hbm_gbs"]})
    mem_stages, rdc = {}, None
    if not args.ep:
        for s in ("moe_router", "moe_dispatch", "moe_combine"):
            gbs = sbytes[s] / (stage_ms[s] * 1e-3) / 1e9
            mem_stages[s] = {"ms": stage_ms[s], "bytes": sbytes[s], "GB/s": gbs, "frac": gbs / pk["hbm_gbs"]}
        rdc_bytes = sum(sbytes.values())
        rdc_ms = sum(stage_ms[s] for s in ("moe_router", "moe_dispatch", "moe_combine"))
        rdc = {"bytes": rdc_bytes, "ms": rdc_ms, "GB/s": rdc_bytes / (rdc_ms * 1e-3) / 1e9,
               "frac": rdc_bytes / (rdc_ms * 1e-3) / 1e9 / pk["hbm_gbs"]}

    # ---- end to end through the public API with host buffers: every step copies its x
    # from pinned host memory to the device, runs the layer, and copies y and aux back.
    # Steps are pipelined over three streams (copy in / compute / copy out) with two
    # layer instances, so step i+1's upload and step i-1's download overlap step i.
    e2e = None
    if not args.no_e2e:
        x_host = inp["x"].cpu().pin_memory()
        layers = [layer, MoELayer(cfg, dict(inp), device=dev, ep_ranks=args.ep, prepared_router=prepared)]
        x_dev = [inp["x"].clone() for _ in layers]  # valid data before the first forward
        for L, xd in zip(layers, x_dev):
            L.set_x(xd)
        fwd = [(lambda L=L: L.run("moe_forward")) for L in layers]
        if not args.no_graph:
            for b_, L in enumerate(layers):
                L.run("moe_forward")
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    L.run("moe_forward")
                fwd[b_] = g.replay
        y_host = [torch.empty_like(out["y"], device="cpu").pin_memory() for _ in range(K)]
        aux_host = [torch.empty(1, dtype=torch.float32).pin_memory() for _ in range(K)]
        s_in, s_run, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev = lambda: torch.cuda.Event(enable_timing=False)  # noqa: E731
        def run_e2e(nsteps, t0=None, t1=None):
            up, comp, down = [None] * nsteps, [None] * nsteps, [None] * nsteps
            if t0 is not None:
                t0.record(s_in)
            for i in range(nsteps):
                b = i % 2
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(comp[i - 2])  # x buffer b is free again
                    x_dev[b].copy_(x_host, non_blocking=True)
                    up[i] = ev(); up[i].record(s_in)
                with torch.cuda.stream(s_run):
                    s_run.wait_event(up[i])
                    if i >= 2:
                        s_run.wait_event(down[i - 2])  # outputs of buffer b downloaded
                    fwd[b]()
                    comp[i] = ev(); comp[i].record(s_run)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(comp[i])
                    y_host[i % K].copy_(layers[b].out["y"], non_blocking=True)
                    aux_host[i % K].copy_(layers[b].out["aux"], non_blocking=True)
                    down[i] = ev(); down[i].record(s_out)
            if t1 is not None:
                s_out.wait_event(down[nsteps - 1])
                t1.record(s_out)
        run_e2e(max(args.warmup, 2))
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        run_e2e(K, t0, t1)
        torch.cuda.synchronize()
        e_ms = t0.elapsed_time(t1) / K
        if world > 1:
            e_ms = max_over_ranks(e_ms, dev)
        esz = x_host.element_size()
        h2d = x_host.numel() * esz
        d2h = y_host[0].numel() * y_host[0].element_size() + 4
        e2e = {"value": replica_throughput(world, cfg.T, e_ms), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e_ms, "pcie_GB/s": (h2d + d2h) / (e_ms * 1e-3) / 1e9,
               "method": "moe_forward per step (its CUDA graph) on pinned host buffers; upload, "
                         "compute and download of consecutive steps overlap on three streams"}
        layer = layers[0]

    status = layer.device_status()
    if status != 0:
        print(f"device status {status}", file=sys.stderr)
        return 1
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    cpu_base = None
    if not args.no_cpu_baseline:
        cpu_inp = {k: (None if v is None else v.cpu()) for k, v in inp.items()}
        if cfg.weights in ("int8", "int4"):  # the oracle runs on the exactly dequantised weights
            from oracle import moe_oracle as orc
            for k_ in ("W1", "W3", "W2"):
                q_ = cpu_inp.get(k_)
                if q_ is None:
                    continue
                if cfg.weights == "int8":
                    cpu_inp[k_] = orc.dequantize_int8(q_.numpy().reshape(-1, q_.shape[-1]),
                                                      cpu_inp[k_ + "_scale"].numpy().reshape(-1)).reshape(q_.shape)
                else:
                    cpu_inp[k_] = orc.dequantize_int4(q_.numpy(), cpu_inp[k_ + "_scale"].numpy())
        # about 10 G multiply-adds of expert work: ~10-30 s on the host cores
        per_tok = cfg.d * cfg.F * (3 if cfg.act == "swiglu" else 2) * (cfg.k + cfg.S)
        secs, desc, threads = oracle_step(cfg, cpu_inp, int(max(16, min(cfg.T, 1e10 / per_tok))))
        cpu_base = {"value": cfg.T / secs, "unit": UNIT, "cores": threads, "kind": "oracle",
                    "sample": desc}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": cfg.dtype,
        "data": "synthetic (seeded; shapes and distributions of the workload; random-init weights)",
        "config": {"workload": workload_name(cfg), "tokens_per_step": cfg.T,
                   "l2": "flushed between steps (2x L2 buffer written outside the timed events)",
                   "router_weights": ("split into three bf16 terms once (moe_prepare_router_weights), as "
                                      "after a weight update" if prepared else "split on every call"),
                   "parallelism": (f"replicas x{world}" if world > 1 else "single GPU")
                   + (f"; expert parallel over {args.ep} ranks emulated on each GPU" if args.ep else ""),
                   "launch": ("direct C-ABI calls" if args.no_graph else
                              "one CUDA graph of moe_forward per step (kernels chained by programmatic "
                              "dependent launch)"),
                   "stage_timing": "second timed pass of the same K steps, CUDA events between the "
                                   "four stage calls (events break the launch overlap, so the stage "
                                   "times add up to slightly more than ms_per_step)",
                   "stage_ms": stage_ms,
                   "memory_stages": mem_stages,
                   "router_dispatch_combine": rdc,
                   "wall_s_timed_region": t_wall},
        "roofline": roof,
        "cpu_baseline": cpu_base,
        "e2e": e2e,
        "gpu_launches": launches_per_step * K,
        "clocks": (nvml.summary() or clk.summary()),
        "clocks_nvidia_smi": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def backward_work(cfg, out):
    """Minimum work of the backward's expert stage for this batch.

    Flops: dgrad and wgrad of every expert matrix on the kept rows (2 x the
    forward's); the pre-activations the activation backward needs are kept by the
    forward, not recomputed.  Bytes: the weights of touched experts read once,
    every weight gradient written once (untouched experts get zeros), and the row
    activations read or written once: Xp, H, dYp, dXp (d, F, d, d per kept row)
    plus the saved pre-activations (GELU: F, SwiGLU: 2F per kept row)."""
    import torch
    kept = (out["dropped"] == 0)
    idx = out["expert_idx"].long()
    kept_per_e = torch.zeros(cfg.E, dtype=torch.long, device=idx.device)
    kept_per_e.scatter_add_(0, idx[kept], torch.ones_like(idx[kept]))
    touched = int((kept_per_e > 0).sum()) + cfg.S
    rows = int(kept.sum()) + cfg.S * cfg.T
    esz = 2 if cfg.dtype == "bf16" else 4
    nmat = 3 if cfg.act == "swiglu" else 2
    n_pre = {"relu": 0, "swiglu": 2}.get(cfg.act, 1)
    flops = 2.0 * rows * cfg.d * cfg.F * 2 * nmat
    w = nmat * cfg.d * cfg.F * esz
    nbytes = touched * w + (cfg.E + cfg.S) * w + rows * esz * (3 * cfg.d + (1 + n_pre) * cfg.F)
    return {"flops": flops, "bytes": nbytes, "rows": rows, "touched_experts": touched}


def run_gpu_backward(args):
    """Training step of the layer: moe_forward + moe_backward, CUDA graph per step."""
    import torch

    from sparse_mixture_experts_scan_b300 import MoELayer, _lib, make_inputs

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    cfg = bench_config(args)
    inp = make_inputs(cfg, seed=rank, device=dev)
    layer = MoELayer(cfg, inp, device=dev, flags=_lib.MOE_FLAG_TRAINING)
    g = torch.Generator(device=dev).manual_seed(100 + rank)
    dy = torch.randn(cfg.T, cfg.d, generator=g, device=dev).to(cfg.torch_dtype)
    stream = torch.cuda.current_stream(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 64 << 20), dtype=torch.uint8, device=dev)
    for _ in range(max(args.warmup, 1)):
        layer.run("moe_forward")
        layer.backward(dy, 0.01)
    torch.cuda.synchronize()
    n0 = _lib.moe_kernel_launches()
    g_fwd, g_bwd = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_fwd):
        layer.run("moe_forward")
    with torch.cuda.graph(g_bwd):
        layer.backward(dy, 0.01)
    launches = _lib.moe_kernel_launches() - n0
    for _ in range(2):
        g_fwd.replay()
        g_bwd.replay()
    torch.cuda.synchronize()
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    nvml = NvmlSampler(dev.index)
    with nvml:
        for i in range(K):
            flush.zero_()
            ev[i][0].record(stream)
            g_fwd.replay()
            ev[i][1].record(stream)
            g_bwd.replay()
            ev[i][2].record(stream)
        torch.cuda.synchronize()
    fwd_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / K
    bwd_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / K
    ms = fwd_ms + bwd_ms
    if world > 1:
        ms = max_over_ranks(ms, dev)
    status = layer.device_status()
    if status != 0:
        print(f"device status {status}", file=sys.stderr)
        return 1
    if rank != 0:
        return 0
    work = backward_work(cfg, layer.out)
    pk = peaks()
    hbm_bound = work["flops"] / work["bytes"] < pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    if hbm_bound:
        ach = work["bytes"] / (bwd_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": ach / pk["hbm_gbs"]}
    else:
        ach = work["flops"] / (bwd_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": ach / pk["bf16_tflops"]}
    roof.update({"traffic": None, "kernel": "the whole moe_backward call (every backward kernel; expert work only "
                 "counted)", "algorithmic_bytes": work["bytes"], "algorithmic_flops": work["flops"],
                 "peak_source": pk["source"] + " (burst)"})
    line = {
        "metric": "MoE layer training step (fwd + bwd) tokens/s on 1 B300", "value": replica_throughput(world, cfg.T, ms),
        "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": cfg.dtype,
        "data": "synthetic (seeded; shapes and distributions of the workload; random-init weights)",
        "config": {"workload": workload_name(cfg), "tokens_per_step": cfg.T, "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
                   "l2": "flushed before each step", "launch": "CUDA graphs of moe_forward and moe_backward"},
        "roofline": roof, "gpu_launches": launches * K, "clocks": nvml.summary(),
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.backward:
        return run_gpu_backward(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
