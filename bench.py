#!/usr/bin/env python3
"""Benchmark of the routed NVFP4 MoE layer at decode (one JSON line on rank 0).

A step is one pass of the whole hot path over one batch: router GEMV + top-k
(moe_route) and the routed expert FFN with its combine (moe_forward), on
inputs already resident in HBM.  Default workload: the K3-shape layer (896
experts, top-16, hidden 3584, FFN 3072, NVFP4, ~16.6 GB resident) at decode
batch 1.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

Timed region: K steps replayed from CUDA graphs (16 rotating token sets, so
the routed experts change every step; the 297 MB of expert bytes a step reads
exceed the 129 MB L2), bracketed by barrier + synchronize, timed with CUDA
events, max over ranks.  Every graph is replayed once before timing, and the
K steps are timed in three windows: the line reports the median window and
the spread.  Under torchrun each rank runs its own replica of the
layer on its own tokens (weak scaling, no collective on the data path).

The JSON line also carries: the gate/up kernel's roofline (algorithmic bytes /
CUDA-event duration, from a second loop with per-stage events), an end-to-end
number through the C ABI with host buffers (H2D of x and D2H of y inside the
timed region), SM clocks sampled during the timed region, and the float64
oracle timed on the host cores on a bounded sample (cpu_baseline).
``--impl reference`` times only that oracle as the reference arm.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer decode tok/s (896 experts, top-16, NVFP4); expert-weight HBM GB/s"
EXPERT_BYTES_K3 = 18_579_480

CONFIGS = {
    # name: experts, top_k, hidden, inter, tokens per step, layers, zipf router
    "k3b1": dict(E=896, k=16, H=3584, I=3072, C=1, layers=1, zipf=False,
                 workload="K3-shape MoE layer, decode batch 1, top-16 of 896, NVFP4, uniform routing"),
    "k3c7k16": dict(E=896, k=16, H=3584, I=3072, C=7, layers=1, zipf=False,
                    workload="K3-shape MoE layer, decode batch 7, top-16 of 896, NVFP4, uniform routing"),
    "k3c7k8": dict(E=896, k=8, H=3584, I=3072, C=7, layers=1, zipf=False,
                   workload="K3-shape MoE layer, decode batch 7, top-8 of 896, NVFP4, uniform routing"),
    "k3c16": dict(E=896, k=16, H=3584, I=3072, C=16, layers=1, zipf=False,
                  workload="K3-shape MoE layer, batch of 16 tokens, top-16 of 896, NVFP4, uniform routing "
                           "(decode kernels in groups of 8, below the grouped path's crossover)"),
    "k3c64": dict(E=896, k=16, H=3584, I=3072, C=64, layers=1, zipf=False,
                  workload="K3-shape MoE layer, batch of 64 tokens, top-16 of 896, NVFP4, uniform routing "
                           "(grouped tcgen05 path)"),
    "k3x8zipf": dict(E=896, k=16, H=3584, I=3072, C=1, layers=8, zipf=True,
                     workload="8 K3-shape MoE layers (133 GB resident), decode batch 1, top-16 of 896, NVFP4, "
                              "Zipf-biased routing (s = 1.1, per-layer permutation)"),
    "prefill512": dict(E=896, k=16, H=3584, I=3072, C=512, layers=1, zipf=True,
                       workload="K3-shape MoE layer, prefill of 512 tokens, top-16 of 896, NVFP4, "
                                "Zipf-biased routing (s = 1.1)"),
    "k3verify4": dict(E=896, k=16, H=3584, I=3072, C=4, layers=1, zipf=False, draft_rho=0.95,
                      workload="K3-shape MoE layer, multi-row verify pass: 4 draft rows of one stream "
                               "(pairwise correlation 0.95), top-16 of 896, NVFP4"),
    "k3verify8": dict(E=896, k=16, H=3584, I=3072, C=8, layers=1, zipf=False, draft_rho=0.95,
                      workload="K3-shape MoE layer, multi-row verify pass: 8 draft rows of one stream "
                               "(pairwise correlation 0.95), top-16 of 896, NVFP4"),
    "k3b1mx": dict(E=896, k=16, H=3584, I=3072, C=1, layers=1, zipf=False, fmt="mxfp4",
                   workload="K3-shape MoE layer, decode batch 1, top-16 of 896, MXFP4 (e8m0 scale per 32), "
                            "uniform routing"),
    "k3c7mx": dict(E=896, k=16, H=3584, I=3072, C=7, layers=1, zipf=False, fmt="mxfp4",
                   workload="K3-shape MoE layer, decode batch 7, top-16 of 896, MXFP4 (e8m0 scale per 32), "
                            "uniform routing"),
    "k3ffnb1": dict(E=896, k=16, H=3584, I=3072, C=1, layers=1, zipf=False,
                    ffn=dict(hidden=7168, shared=2, shared_inter=3072),
                    workload="K3-shape MoE FFN at decode batch 1: routed_down 7168->3584, router + top-16 of 896 "
                             "experts, routed_norm, routed_up 3584->7168, 2 shared experts (7168->3072->7168), "
                             "NVFP4"),
    "prefill512w4a4": dict(E=896, k=16, H=3584, I=3072, C=512, layers=1, zipf=True, w4a4=True,
                           workload="K3-shape MoE layer, prefill of 512 tokens, top-16 of 896, NVFP4 weights, "
                                    "W4A4 (x and h quantized to NVFP4 with each expert's static input scales), "
                                    "Zipf-biased routing (s = 1.1)"),
    "k3b1w4a4": dict(E=896, k=16, H=3584, I=3072, C=1, layers=1, zipf=False, w4a4=True,
                     workload="K3-shape MoE layer, decode batch 1, top-16 of 896, NVFP4 weights, W4A4 "
                              "(x and h quantized to NVFP4 in the decode kernels' fragments), uniform routing"),
    "tiny": dict(E=32, k=4, H=256, I=192, C=1, layers=1, zipf=False,
                 workload="tiny MoE layer, 32 experts, top-4, hidden 256, FFN 192, batch 1 (L2-resident)"),
}
ROTATE = 16          # distinct token sets cycled through the timed steps


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=200)
    p.add_argument("--config", default="k3b1", choices=sorted(CONFIGS))
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-budget-s", type=float, default=20.0)
    p.add_argument("--experts", type=int, default=None,
                   help="use this many experts instead of the workload's (a smaller case for profiler captures)")
    return p.parse_args()


# ---------------------------------------------------------------- utilities

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class ClockSampler:
    """nvidia-smi clocks/throttle sampling while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        try:
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
            if self.gpu_id is not None:
                cmd += ["-i", str(self.gpu_id)]
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.reader.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [q.strip() for q in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs"), "measured"
    return 6800.0, "fallback"


# every source file that goes into a kernel: the .cu and the headers it includes
KERNEL_SOURCES = {
    "expert_gemv.cu": ("csrc/expert_gemv.cu", "csrc/gemv_core.cuh", "csrc/moe_internal.cuh", "csrc/kernels.h",
                       "../include/moe.h"),
    "grouped.cu": ("csrc/grouped.cu", "csrc/gemv_core.cuh", "csrc/moe_internal.cuh", "csrc/kernels.h",
                   "../include/moe.h"),
}


def kernel_sources_sha256(kernel_file):
    """sha256 over the kernel's source files (the .cu and its headers, in a
    fixed order): the key under which an ncu summary stays valid."""
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel_file]:
        with open(os.path.join(ROOT, "quantized_moe_expert_router_gb300", rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def ncu_traffic(kernel_file, tag):
    """DRAM bytes per unit from a committed ncu summary, if none of the
    kernel's source files has changed since the capture (their combined
    sha256 is recorded in the summary).  Returns (bytes, source) or
    (None, reason)."""
    prof = os.path.join(ROOT, "profiles", f"{tag}.md")
    if not os.path.exists(prof):
        return None, f"no ncu summary profiles/{tag}.md"
    txt = open(prof).read()
    m = re.search(r"dram_bytes_per_expert:\s*([0-9.eE+]+)", txt)
    h = re.search(r"sources_sha256:\s*([0-9a-f]{64})", txt)
    if not m or not h:
        return None, f"profiles/{tag}.md records no DRAM bytes or source hash"
    if kernel_sources_sha256(kernel_file) != h.group(1):
        return None, f"profiles/{tag}.md was captured on other kernel sources"
    return float(m.group(1)), (f"ncu dram__bytes_read.sum + dram__bytes_write.sum per expert from "
                               f"profiles/{tag}.md (sources sha256 {h.group(1)[:12]}), times the experts "
                               f"of one launch")


def host_cpu():
    """(cores this process may use, CPU model name) of the host."""
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        cores = os.cpu_count() or 1
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                model = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        import platform
        model = platform.processor() or platform.machine()
    return cores, model


# ---------------------------------------------------------------- oracle legs

def oracle_sample(cfg, seed, layer_id, weights_for, budget_s, Wr, bias, x_bits, threads=1):
    """Time the float64 oracle on whole tokens of the workload, one token after
    the other, until ``budget_s`` is used (at least one token): router logits
    and top-k on one thread, the token's expert FFNs on ``threads`` threads
    (oracle_moe_forward_mt spreads its (token, slot) evaluations; one thread
    runs the plain loop).  Returns (tokens, seconds)."""
    import oracle
    done, t_total = 0, 0.0
    for t in range(x_bits.shape[0]):
        xb = x_bits[t:t + 1]
        t0 = time.perf_counter()
        logits = oracle.router_logits(Wr, xb, bias)
        ids, w, _ = oracle.route(logits, cfg["k"])
        sel = sorted(set(int(e) for e in ids.ravel()))
        t_prep0 = time.perf_counter()
        weights = weights_for(sel)                       # input staging, not timed
        t_prep = time.perf_counter() - t_prep0
        remap = {e: i for i, e in enumerate(sel)}
        if cfg.get("w4a4"):
            oracle.moe_forward_w4a4(weights, xb, np.vectorize(remap.get)(ids).astype(np.int32), w, threads=threads)
        else:
            oracle.moe_forward(weights, xb, np.vectorize(remap.get)(ids).astype(np.int32), w, threads=threads,
                               fmt=cfg.get("fmt", "nvfp4"))
        t_total += time.perf_counter() - t0 - t_prep
        done += 1
        if t_total >= budget_s:
            break
    return done, t_total


def run_reference(args, cfg, rank):
    """Reference arm: the float64 oracle on the host cores, on this config."""
    from quantized_moe_expert_router_gb300 import synth
    import oracle
    oracle.build()
    if rank != 0:
        return
    E, k, H, I, C = cfg["E"], cfg["k"], cfg["H"], cfg["I"], cfg["C"]
    Wr = synth.router_weights(args.seed, 0, E, H, synth.ZIPF_ROUTER_STD if cfg["zipf"] else 1.0)
    bias = synth.zipf_bias(args.seed, 0, E) if cfg["zipf"] else None
    cache = {}

    def weights_for(sel):
        need = [e for e in sel if e not in cache]
        if need:
            part = synth.canonical_layer(args.seed, 0, E, H, I, experts=need, fmt=cfg.get("fmt", "nvfp4"))
            for j, e in enumerate(need):
                cache[e] = {n: {f: m[f][j] for f in ("codes", "scales", "g", "a")} for n, m in part.items()}
        return {n: {f: np.stack([cache[e][n][f] for e in sel]) for f in ("codes", "scales", "g", "a")}
                for n in ("gate", "up", "down")}

    # one step = one token of the workload; the step count is capped so the
    # whole run stays within a few minutes
    x_all = synth.tokens(args.seed, 0, max(1, args.steps + args.warmup), H) if args.steps + args.warmup <= 64 \
        else synth.tokens(args.seed, 0, 64, H)
    threads = min(oracle.default_threads(), k)     # a step is one token: k expert FFNs at most in parallel
    cores, model = host_cpu()
    warm = min(args.warmup, 3)                     # oracle warm-up steps, capped (each is a whole token)
    for t in range(warm):
        oracle_sample(cfg, args.seed, 0, weights_for, 0.0, Wr, bias, x_all[t:t + 1], threads)
    steps_done, elapsed = 0, 0.0
    budget = 150.0
    for s in range(args.steps):
        xb = x_all[(warm + s) % x_all.shape[0]: (warm + s) % x_all.shape[0] + 1]
        n, dt = oracle_sample(cfg, args.seed, 0, weights_for, 0.0, Wr, bias, xb, threads)
        steps_done += 1
        elapsed += dt
        if elapsed >= budget:
            break
    tok_s = steps_done / elapsed
    line = {
        "impl": "reference", "metric": METRIC, "value": tok_s, "unit": "tok/s", "n_gpus": args.gpus,
        "steps": steps_done, "warmup": warm, "ms_per_step": 1e3 * elapsed / steps_done,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": cfg["workload"], "tokens_per_step": 1},
        "cpu_baseline": {"value": tok_s, "unit": "tok/s", "cores": threads, "kind": "oracle",
                         "host_cores": cores, "cpu_model": model,
                         "sample": f"{steps_done} whole token(s) of the workload (router and top-k on one "
                                   f"thread, the {k} expert FFNs on {threads} threads), float64 C oracle"},
        "e2e": {"value": tok_s, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "note": "; ".join(n_ for n_ in (("step count capped by a 150 s budget" if steps_done < args.steps else ""),
                                        (f"warm-up capped at {warm} oracle steps" if warm < args.warmup else ""))
                          if n_),
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- our arm

def main():
    args = parse()
    cfg = dict(CONFIGS[args.config])
    if args.experts:
        cfg["E"] = args.experts
        cfg["workload"] += f" [reduced to {args.experts} experts for profiling]"
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, cfg, rank)
        return

    import torch
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    torch.cuda.set_device(local)
    dev = torch.device(f"cuda:{local}")

    from quantized_moe_expert_router_gb300 import build as pkg_build
    if rank == 0:
        pkg_build.build()
    if world > 1:
        dist.barrier()
    from quantized_moe_expert_router_gb300 import moe, synth
    from quantized_moe_expert_router_gb300.synth import device as synth_dev

    E, k, H, I, C = cfg["E"], cfg["k"], cfg["H"], cfg["I"], cfg["C"]
    NL = cfg["layers"]
    free, total = torch.cuda.mem_get_info(dev)
    # the layers' packed weights plus one canonical copy while a layer is packed
    need = (NL + 1.2) * E * EXPERT_BYTES_K3 * (H * I) / (3584 * 3072)
    if need > free:
        print(json.dumps({"metric": METRIC, "error": f"needs {need / 1e9:.1f} GB free HBM, {free / 1e9:.1f} GB free"}))
        sys.exit(1)

    # one handle serves every layer (it holds the shapes only); per layer its
    # packed weights, router and (Zipf) router bias
    fmt = cfg.get("fmt", "nvfp4")
    w4a4 = bool(cfg.get("w4a4"))
    layer = moe.Layer(E, k, H, I, C, device=local,
                      flags=(moe.CONFIG_MXFP4 if fmt == "mxfp4" else 0) | (moe.CONFIG_W4A4 if w4a4 else 0))
    grouped = C >= 28                             # the path moe_forward takes
    router_std = synth.ZIPF_ROUTER_STD if cfg["zipf"] else 1.0
    packed, Wr_ds, bias_ds, biases = [], [], [], []
    canon = None
    for li in range(NL):
        cl = synth_dev.canonical_layer_device(args.seed, li, E, H, I, dev, fmt=fmt)
        pk = moe.alloc_packed(layer, dev)
        moe.moe_pack_weights(layer, cl, pk)
        packed.append(pk)
        if li == 0:
            canon = cl                          # kept for the oracle's sample (layer 0)
        else:
            del cl
            torch.cuda.empty_cache()
        Wl = synth.router_weights(args.seed, li, E, H, router_std)
        bl = synth.zipf_bias(args.seed, li, E) if cfg["zipf"] else None
        Wr_ds.append(torch.from_numpy(Wl).to(dev))
        bias_ds.append(None if bl is None else torch.from_numpy(bl).to(dev))
        biases.append(bl)
        if li == 0:
            Wr, bias = Wl, bl

    FFN = cfg.get("ffn")
    if FFN:
        # the FFN around the routed sum (one layer): its weights on the device
        Hd = FFN["hidden"]
        fw = synth_dev.ffn_weights_device(args.seed, 0, Hd, H, FFN["shared"], FFN["shared_inter"], dev)
        ffn = moe.Ffn(layer, Hd, FFN["shared"], FFN["shared_inter"], eps=fw["eps"])
        fpacked = moe.alloc_ffn_packed(ffn, dev)
        moe.moe_ffn_pack_weights(ffn, fw, fpacked)
        ffn_ws = moe.alloc_ffn_workspace(ffn, C, dev)
        ffn_bytes = sum(m["codes"].numel() + m["scales"].numel() + 8 * m["g"].numel()
                        for m in [fw["routed_down"], fw["routed_up"]] + list(fw["shared"].values()))
    # rotating token sets, distinct per rank
    if FFN:
        x_host = [synth.tokens(args.seed + 1000 * rank, r, C, FFN["hidden"]) for r in range(ROTATE)]
        outs = [torch.empty((C, FFN["hidden"]), dtype=torch.float32, device=dev) for _ in range(ROTATE)]
    elif cfg.get("draft_rho") is not None:
        x_host = [synth.draft_rows(args.seed + 1000 * rank, r, C, H, cfg["draft_rho"]) for r in range(ROTATE)]
    else:
        x_host = [synth.tokens(args.seed + 1000 * rank, r, C, H) for r in range(ROTATE)]
    xs = [torch.from_numpy(xh.view(np.int16)).to(dev) for xh in x_host]
    ids = [[torch.empty((C, k), dtype=torch.int32, device=dev) for _ in range(NL)] for _ in range(ROTATE)]
    wts = [[torch.empty((C, k), dtype=torch.float32, device=dev) for _ in range(NL)] for _ in range(ROTATE)]
    ys = [torch.empty((C, H), dtype=torch.float32, device=dev) for _ in range(ROTATE)]
    ws = moe.alloc_workspace(layer, C, dev)

    # the oracle's sample needs the canonical bytes of the experts it selects
    cpu_sample = None
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        sample_x = np.concatenate(x_host, axis=0)[:16]
        host_cache = {}

        def weights_for(sel):
            need_e = [e for e in sel if e not in host_cache]
            if need_e:
                part = synth_dev.gather_to_host(canon, need_e)
                for j, e in enumerate(need_e):
                    host_cache[e] = {n: {f: m[f][j] for f in ("codes", "scales", "g", "a")} for n, m in part.items()}
            return {n: {f: np.stack([host_cache[e][n][f] for e in sel]) for f in ("codes", "scales", "g", "a")}
                    for n in ("gate", "up", "down")}
        cpu_sample = (sample_x, weights_for)
        threads = min(oracle.default_threads(), k)     # one token at a time: k expert FFNs in parallel
        cores, model = host_cpu()
        if FFN:
            fw_host = {"routed_down": {f: (fw["routed_down"][f].cpu().numpy() if f in ("codes", "scales")
                                           else float(fw["routed_down"][f][0])) for f in ("codes", "scales", "g")},
                       "routed_up": {f: (fw["routed_up"][f].cpu().numpy() if f in ("codes", "scales")
                                         else float(fw["routed_up"][f][0])) for f in ("codes", "scales", "g")},
                       "shared": {n: {f: m[f].cpu().numpy() for f in ("codes", "scales", "g", "a")}
                                  for n, m in fw["shared"].items()},
                       "gamma": fw["gamma"].cpu().numpy(), "eps": fw["eps"]}

            def ffn_sample(budget_s, th):
                done_, tt_, fetch = 0, 0.0, [0.0]

                def fetch_w(sel):
                    f0 = time.perf_counter()
                    r_ = weights_for(sel)
                    fetch[0] += time.perf_counter() - f0
                    return r_
                for t in range(sample_x.shape[0]):
                    fetch[0] = 0.0
                    t0_ = time.perf_counter()
                    oracle.ffn_layer(fw_host, fetch_w, Wr, sample_x[t:t + 1], k, bias, threads=th)
                    tt_ += time.perf_counter() - t0_ - fetch[0]
                    done_ += 1
                    if tt_ >= budget_s:
                        break
                return done_, tt_
            done_t, secs_t = ffn_sample(args.cpu_budget_s / 4, threads)
            done, secs = ffn_sample(args.cpu_budget_s, 1)
            cpu_baseline = {"value": done_t / secs_t, "unit": "tok/s", "cores": threads, "kind": "oracle",
                            "host_cores": cores, "cpu_model": model,
                            "sample": f"{done_t} whole token(s) of this workload (routed_down, router + top-{k}, "
                                      f"routed_norm, routed_up and the shared experts on one thread, the {k} routed "
                                      f"expert FFNs on {threads} threads), float64 C oracle, {secs_t:.1f} s",
                            "single_thread": {"value": done / secs, "unit": "tok/s", "cores": 1,
                                              "sample": f"{done} whole token(s), one thread, {secs:.1f} s"}}
        # the threaded oracle (expert FFNs of a token over all the cores), then
        # the plain one-thread loop on the same tokens
        if not FFN:
            done_t, secs_t = oracle_sample(cfg, args.seed, 0, weights_for, args.cpu_budget_s / 4, Wr, bias, sample_x,
                                           threads)
            done, secs = oracle_sample(cfg, args.seed, 0, weights_for, args.cpu_budget_s, Wr, bias, sample_x)
            cpu_baseline = {"value": done_t / secs_t, "unit": "tok/s", "cores": threads, "kind": "oracle",
                            "host_cores": cores, "cpu_model": model,
                            "sample": f"{done_t} whole token(s) of this workload (router + top-{k} on one thread, "
                                      f"the {k} expert FFNs on {threads} threads, combine), float64 C oracle, "
                                      f"{secs_t:.1f} s",
                            "single_thread": {"value": done / secs, "unit": "tok/s", "cores": 1,
                                              "sample": f"{done} whole token(s), one thread, {secs:.1f} s"}}
    del canon
    torch.cuda.empty_cache()

    stream = torch.cuda.Stream(dev)

    def step(r, s, x=None):
        x = xs[r] if x is None else x
        for li in range(NL):
            if FFN:
                moe.moe_ffn_forward(ffn, x, C, Wr_ds[li], bias_ds[li], packed[li], fpacked, ids[r][li], wts[r][li],
                                    outs[r], ffn_ws, s)
            else:
                moe.moe_route_forward(layer, x, C, Wr_ds[li], bias_ds[li], packed[li], ids[r][li], wts[r][li],
                                      ys[r], ws, s)

    # distinct experts each rotating input selects, summed over the layers
    # (the bytes a step streams)
    with torch.cuda.stream(stream):
        for r in range(ROTATE):
            step(r, stream)
    stream.synchronize()
    distinct = [sum(len(set(ids[r][li].cpu().numpy().ravel().tolist())) for li in range(NL)) for r in range(ROTATE)]
    zipf_stats = None
    if cfg["zipf"]:
        # share of the picks that fall on each layer's 104 hottest experts (by bias)
        hits = picks = 0
        for li in range(NL):
            hot = set(np.argsort(-biases[li], kind="stable")[:104].tolist())
            for r in range(ROTATE):
                got = ids[r][li].cpu().numpy().ravel().tolist()
                hits += sum(e in hot for e in got)
                picks += len(got)
        zipf_stats = {"top104_pick_share": hits / picks, "picks": picks}
    flags = moe.moe_get_device_status(layer, ws, stream)
    if flags:
        raise RuntimeError(f"device flags {flags:#x} after the first pass")

    def capture(nsteps, offset):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(nsteps):
                step((offset + i) % ROTATE, stream)
        return g

    g_full = capture(ROTATE, 0)
    rem = args.steps % ROTATE
    g_rem = capture(rem, 0) if rem else None
    wrem = args.warmup % ROTATE
    g_wrem = capture(wrem, 0) if wrem else None

    def run_steps():
        for _ in range(args.steps // ROTATE):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()

    # warm-up: the requested steps, and every graph the timed region replays
    # at least once (its first replay uploads it)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup // ROTATE):
            g_full.replay()
        if g_wrem is not None:
            g_wrem.replay()
        g_full.replay()
        if g_rem is not None:
            g_rem.replay()
    stream.synchronize()

    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = None
    sampler = ClockSampler(gpu_id)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)
    # three timed windows of exactly K steps each, every one bracketed by a
    # barrier and a synchronize; the line reports the median window (max over
    # ranks) and the spread of the three
    windows = []
    t_host = 0.0
    for _ in range(3):
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t_host0 = time.perf_counter()
        ev0.record(stream)
        with torch.cuda.stream(stream):
            run_steps()
        ev1.record(stream)
        stream.synchronize()
        t_host += time.perf_counter() - t_host0
        torch.cuda.synchronize(dev)
        wms = ev0.elapsed_time(ev1)
        if world > 1:
            dist.barrier()
            tt = torch.tensor([wms], device=dev, dtype=torch.float64)
            dist.all_reduce(tt, op=dist.ReduceOp.MAX)
            wms = float(tt.item())
        windows.append(wms)
    clocks = sampler.stop()
    ms = float(np.median(windows))
    ms_per_step = ms / args.steps
    # one MoE layer's throughput: a step runs NL layers on the same C tokens
    tokens = C * args.steps * NL * world
    tok_s = tokens / (ms / 1e3)
    avg_distinct = sum(distinct[(i % ROTATE)] for i in range(args.steps)) / args.steps
    if fmt == "mxfp4":
        expert_bytes = 3 * (I * H // 2 + I * H // 32 + 8)
    else:
        expert_bytes = EXPERT_BYTES_K3 if (H, I) == (3584, 3072) else 3 * (I * H // 2 + I * H // 16 + 8)
    hbm_gbs = avg_distinct * expert_bytes * world / (ms_per_step * 1e-3) / 1e9

    # ---- roofline of the dominant kernel (gate/up), per-stage CUDA events
    n_prof = 256 if C == 1 else 128
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_prof)]
    for trio in evs:
        for e_ in trio:
            e_.record(stream)
    stream.synchronize()
    with torch.cuda.stream(stream):
        for i in range(n_prof):
            r = i % ROTATE
            if FFN:                          # the events bracket the routed kernels inside the layer
                moe.moe_set_stage_events(layer, evs[i])
                step(r, stream)
                continue
            moe.moe_route(layer, xs[r], C, Wr_ds[0], bias_ds[0], ids[r][0], wts[r][0], ws, stream)
            moe.moe_set_stage_events(layer, evs[i])
            moe.moe_forward(layer, xs[r], C, ids[r][0], wts[r][0], packed[0], ys[r], ws, stream)
    moe.moe_set_stage_events(layer, None)
    stream.synchronize()
    gu_ms = [evs[i][0].elapsed_time(evs[i][1]) for i in range(n_prof)]
    dn_ms = [evs[i][1].elapsed_time(evs[i][2]) for i in range(n_prof)]
    gu_bytes_per_expert = 2 * (I * H // 2 + I * H // (32 if fmt == "mxfp4" else 16))
    # the stage events bracket the first gate/up launch of the call: on the
    # decode path that is the first group of at most 8 tokens
    first = C if grouped else min(C, 8)
    gu_units = sum(len(set(ids[i % ROTATE][0][:first].cpu().numpy().ravel().tolist()))
                   for i in range(n_prof)) / n_prof
    gu_avg = float(np.mean(gu_ms))
    dn_avg = float(np.mean(dn_ms))
    hbm_peak, peak_src = measured_peaks()
    achieved = gu_units * gu_bytes_per_expert / (gu_avg * 1e-3) / 1e9
    if grouped:
        # grouped path: the stage events bracket dispatch, x-row prep and the gate/up GEMM
        traffic_per_expert, traffic_src = ncu_traffic("grouped.cu", f"group_tc_gu_{args.config}")
        kernel_label = (f"group_tc_kernel<{2 if w4a4 else 0}> (grouped gate/up + SwiGLU on tcgen05; the timed span "
                        f"also holds the dispatch and x-row {'quantization ' if w4a4 else ''}kernels)")
    else:
        traffic_per_expert, traffic_src = ncu_traffic("expert_gemv.cu", f"expert_gemv_gu_{args.config}")
        kernel_label = (f"expert_gemv_kernel<{2 if C <= 2 else 0}> (gate/up + SwiGLU, "
                        f"{'two tiles' if C <= 2 else 'one tile'} per stage"
                        f"{'; the first group of 8 tokens' if C > 8 else ''})")
    roofline = {"kernel": kernel_label, "bound": "hbm",
                "achieved": achieved, "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                "peak_source": peak_src,
                "traffic": None if traffic_per_expert is None else traffic_per_expert * gu_units,
                "traffic_source": traffic_src,
                "algorithmic_bytes_per_launch": gu_units * gu_bytes_per_expert,
                "avg_launch_us": gu_avg * 1e3,
                "down_kernel": {"avg_launch_us": dn_avg * 1e3,
                                "achieved_gbs": gu_units * (gu_bytes_per_expert / 2) / (dn_avg * 1e-3) / 1e9}}

    # ---- end to end through the C ABI with host buffers
    n_e2e = min(args.steps, 2000)
    Hin = FFN["hidden"] if FFN else H
    x_pin = [torch.from_numpy(xh.view(np.int16)).pin_memory() for xh in x_host]
    y_pin = torch.empty((C, Hin), dtype=torch.float32).pin_memory()
    x_stage = torch.empty((C, Hin), dtype=torch.int16, device=dev)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(n_e2e):
            r = i % ROTATE
            x_stage.copy_(x_pin[r], non_blocking=True)
            step(r, stream, x_stage)
            y_pin.copy_(outs[r] if FFN else ys[r], non_blocking=True)
    stream.synchronize()
    e2e_s = time.perf_counter() - t0
    if world > 1:
        tt = torch.tensor([e2e_s], device=dev, dtype=torch.float64)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        e2e_s = float(tt.item())
    e2e = {"value": C * n_e2e * NL * world / e2e_s, "unit": "tok/s", "steps": n_e2e,
           "h2d_bytes_per_step": C * Hin * 2, "d2h_bytes_per_step": C * Hin * 4,
           "path": ("pinned host u -> H2D -> moe_ffn_forward -> D2H out" if FFN else
                    "pinned host x -> H2D -> moe_route_forward -> D2H y") + ", per step, host-timed"}

    flags = moe.moe_get_device_status(layer, ws, stream)
    if rank == 0:
        line = {
            "metric": METRIC, "value": tok_s, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": ("nvfp4 weights and activations (W4A4), f16 mma of the exact e2m1 x e4m3 values, "
                      "f32 accumulate" if w4a4 else "nvfp4 weights, f16 mma, f32 accumulate"),
            "data": "synthetic",
            "config": {"workload": cfg["workload"], "experts": E, "top_k": k, "hidden": H,
                       "intermediate": I, "tokens_per_step": C, "layers": NL,
                       "value": "tokens per second through one MoE layer" + (f" ({NL} layers per step)" if NL > 1 else ""),
                       "parallelism": f"replicas x{world}",
                       "l2": f"{ROTATE} rotating token sets; each step streams ~{avg_distinct * expert_bytes / 1e6:.0f} MB "
                             "of expert weights (> 129 MB L2)" if H == 3584 else "L2-resident (tiny)",
                       "timing": "CUDA graphs of moe_route_forward, CUDA events on the launching stream"},
            "us_per_layer": 1e3 * ms_per_step / NL,
            "windows_ms_per_step": [w_ / args.steps for w_ in windows],
            "window_spread": (max(windows) - min(windows)) / ms,
            "expert_hbm_gbs": hbm_gbs, "expert_hbm_frac": hbm_gbs / world / hbm_peak,
            **({"ffn": {"weight_bytes_per_step": avg_distinct * expert_bytes + ffn_bytes,
                        "ffn_matrix_bytes": ffn_bytes,
                        "weight_hbm_gbs": (avg_distinct * expert_bytes + ffn_bytes) / (ms_per_step * 1e-3) / 1e9,
                        "weight_hbm_frac": (avg_distinct * expert_bytes + ffn_bytes) / (ms_per_step * 1e-3) / 1e9
                                           / hbm_peak}} if FFN else {}),
            "distinct_experts_per_step": avg_distinct,
            **({"routing": zipf_stats} if zipf_stats else {}),
            "roofline": roofline,
            "e2e": e2e,
            # FFN: + routed_down (2), routed_norm (1), routed_up (2) and 4 per shared expert
            # routed layer per call: C <= 8: fused router, gate/up, down, combine;
            # 9 .. 27 tokens: tiled router + top-k, then 3 decode kernels per group
            # of 8; 28 or more: router, then 7 grouped kernels per pass of 512;
            # (W4A4 from 28 tokens: 6 grouped kernels per pass)
            "gpu_launches": args.steps * NL * ((4 if C <= 8 else 2 + 3 * ((C + 7) // 8) if C < 28
                                                else 2 + (6 if w4a4 else 7) * ((C + 511) // 512))
                                               # FFN: GEMV A (2), norm (1), GEMV B (2; 3 for C > 4)
                                               + ((5 if C <= 4 else 6) if FFN else 0)),
            "clocks": clocks,
            "host_s": t_host,                 # host time of the three windows
            "device_flags": flags,
        }
        if cpu_sample is not None:
            line["cpu_baseline"] = cpu_baseline
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
