#!/usr/bin/env python3
"""Benchmark of the GB300 routed-expert FFN library: prints one JSON line.

Default workload: one K3-shaped routed layer (d_model 7168, d_ff 1536, 896
experts, top-16, MXFP4 weights resident in HBM), decode batches of T = 1, 4
and 16 tokens; one step = moe_plan + the expert FFN for each of the three
batches (21 tokens). The FFN call of each batch takes the faster entry point
as measured on GB300, which is moe_forward (tcgen05 grouped GEMMs) at every
batch size, down to one token (89 vs 101 us for moe_decode, the CUDA-core
streaming path); CROSSOVER_T keeps the rule explicit, and `--path
decode|forward` forces one of them. `--workload prefill4k|skewed8k` times moe_plan +
moe_forward on one prefill batch instead; `--workload router16k` times the
long prefill whose logits come from the library's own fp32 router (x . W_r)
and which adds one bf16 shared expert.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Timing: CUDA events on the library's stream, barrier + synchronize on both
sides, max over ranks. Each step's weight working set (>= 280 MB) exceeds L2
and the router logits rotate through pre-generated sets, so the selected
experts change every step. N > 1 runs independent replicas (the layer does
not shard here): value = tokens of all ranks / slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s + % roofline (decode HBM GB/s; prefill FP4 TFLOP/s), 1xGB300"
K3_SHAPE = (7168, 1536, 896, 16)   # d_model, d_ff, experts, top-k
D_MODEL, D_FF, N_EXPERTS, TOP_K = K3_SHAPE
EXPERT_BYTES = 17547264            # one expert's three MXFP4 matrices (codes + scales)
GATEUP_BYTES = 2 * (D_FF * D_MODEL // 2 + D_FF * D_MODEL // 32)
DOWN_BYTES = D_MODEL * D_FF // 2 + D_MODEL * D_FF // 32


def use_shape(wl: dict) -> None:
    """Layer shape of the chosen workload (K3 unless it names another)."""
    global D_MODEL, D_FF, N_EXPERTS, TOP_K, EXPERT_BYTES, GATEUP_BYTES, DOWN_BYTES
    D_MODEL, D_FF, N_EXPERTS, TOP_K = wl.get("shape", K3_SHAPE)
    GATEUP_BYTES = 2 * (D_FF * D_MODEL // 2 + D_FF * D_MODEL // 32)
    DOWN_BYTES = D_MODEL * D_FF // 2 + D_MODEL * D_FF // 32
    EXPERT_BYTES = GATEUP_BYTES + DOWN_BYTES


def base_workload(name: str):
    """The seeded generator's workload a bench workload draws its inputs from."""
    import synth
    wl = BENCH_WORKLOADS[name]
    if "base" in wl:
        return synth.WORKLOADS[wl["base"]]
    return synth.WORKLOADS["decode1"] if name.startswith("decode") else synth.WORKLOADS[name]
N_SETS = 8
CROSSOVER_T = 0   # largest batch the CUDA-core decode path takes under --path auto

BENCH_WORKLOADS = {
    "decode": {"Ts": [1, 4, 16], "path": "auto",
               "desc": "K3 routed layer decode, T=1,4,16 (d_model 7168, d_ff 1536, 896 experts, top-16, MXFP4)"},
    "prefill4k": {"Ts": [4096], "path": "forward",
                  "desc": "K3 routed layer prefill, T=4096, uniform routing"},
    "skewed8k": {"Ts": [8192], "path": "forward",
                 "desc": "K3 routed layer prefill, T=8192, Zipf(1.1)-skewed routing"},
    "router16k": {"Ts": [16384], "path": "forward", "router": True, "sets": 2,
                  "desc": "K3 routed layer long prefill, T=16384, in-library fp32 router "
                          "(x . W_r) + one bf16 shared expert"},
    "decode_stream": {"Ts": [1, 4, 16], "path": "forward", "stream_slots": 448,
                      "desc": "K3 routed layer decode, T=1,4,16, all 896 experts in pinned host "
                              "memory behind a 448-slot HBM expert cache (expert streaming)"},
    "decode_stream_store": {"Ts": [1, 4, 16], "path": "forward", "stream_slots": 448,
                            "store": True, "codes": 1,   # synth.CODES_PEAKED
                            "desc": "K3 routed layer decode, T=1,4,16, all 896 experts rANS-coded "
                                    "in pinned host memory (compressed expert store; peaked E2M1 "
                                    "codes) behind a 448-slot HBM expert cache, misses decoded "
                                    "on the GPU"},
    # MiMo V2.6 Flash lane: 256 experts, top-8, the same MXFP4 expert FFN; its
    # hidden sizes are not on the pages (d_model 4096, d_ff 2048 give the
    # stated 310B total over 48 layers)
    "mimo_decode": {"Ts": [1, 4, 16], "path": "forward", "shape": (4096, 2048, 256, 8),
                    "base": "mimo_decode",
                    "desc": "MiMo-shaped routed layer decode, T=1,4,16 (d_model 4096, d_ff 2048, "
                            "256 experts, top-8, MXFP4)"},
    "mimo_prefill4k": {"Ts": [4096], "path": "forward", "shape": (4096, 2048, 256, 8),
                       "base": "mimo_prefill4k",
                       "desc": "MiMo-shaped routed layer prefill, T=4096, uniform routing "
                               "(d_model 4096, d_ff 2048, 256 experts, top-8, MXFP4)"},
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 1000 for decode, 60 for prefill)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(BENCH_WORKLOADS), default="decode")
    ap.add_argument("--path", choices=["decode", "forward", "auto"], default=None,
                    help="entry point for the batches (default: auto -- moe_decode up to "
                         "CROSSOVER_T tokens, moe_forward above; measured fastest: forward throughout)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="wall-time budget of the CPU-oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--experts", type=int, default=None,
                    help="experts in the layer (default: the workload's); fewer only for profiling small "
                         "cases, and the line is then marked as such")
    ap.add_argument("--tokens", type=int, default=None,
                    help="one batch of this many tokens instead of the workload's batches; only "
                         "for profiling small cases (the line is then marked as such)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# Replicas: every rank runs the same workload on its own GPU; the job's time is
# the slowest rank's, and its throughput counts the tokens of all ranks.
# ---------------------------------------------------------------------------
def max_over_ranks(times_ms: list, dist=None, device="cpu") -> list:
    """Element-wise maximum of per-rank times (all ranks get the result)."""
    import torch
    t = torch.tensor(times_ms, dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_tokens_per_s(world: int, tokens_per_step: int, steps: int, ms: float) -> float:
    """Whole-job throughput: tokens of all ranks over the (slowest rank's) time."""
    return world * tokens_per_step * steps / (ms * 1e-3)


# ---------------------------------------------------------------------------
# CPU oracle leg (the reference arm and the cpu_baseline object)
# ---------------------------------------------------------------------------
def oracle_tokens_per_s(workload_name: str, budget_s: float):
    """Time the CPU oracle, as it stands, one token at a time until the budget
    is used (at least one token). Returns (tokens/s, tokens, seconds, threads)."""
    import numpy as np
    import synth
    import oracle
    from oracle.run import reference
    oracle.build()
    wl = BENCH_WORKLOADS[workload_name]
    base = base_workload(workload_name)
    done, t0 = 0, time.perf_counter()
    it = 0
    while True:
        T = wl["Ts"][it % len(wl["Ts"])]
        w = synth.Workload(base.name, T=T, D=base.D, F=base.F, E=base.E, k=base.k, seed=base.seed,
                           zipf_s=base.zipf_s, router=base.router, shared=base.shared,
                           codes=wl.get("codes", synth.CODES_UNIFORM))
        x = synth.make_x(w, it % N_SETS)
        lg = None if w.router == "xwr" else synth.make_logits(w, it % N_SETS)
        reference(w, x, lg, tokens=[it % T])
        done += 1
        it += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return done / el, done, el, threads


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    per_step = []
    total_tok = 0
    budget = 90.0 / max(args.steps + args.warmup, 1)   # at least one token per step
    for i in range(args.warmup + args.steps):
        tps, tok, el, threads = oracle_tokens_per_s(args.workload, budget)
        if i >= args.warmup:
            per_step.append(el)
            total_tok += tok
    el = sum(per_step)
    value = total_tok / el
    wl = BENCH_WORKLOADS[args.workload]
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * el / max(args.steps, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl["desc"], "sample": "one token per oracle call, full routing of its batch"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"{total_tok} tokens of the {args.workload} workload, one at a time"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", gpu_id, "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        window = "timed"
        if not inside:
            inside = [p for (_, p) in self.samples]
            window = "run"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(p[0]) for p in inside if num(p[0]) is not None]
        smax = [num(p[1]) for p in inside if num(p[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4) if p[4 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(inside), "window": window}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def kernel_traffic(name: str, source: str, workload: str):
    """DRAM bytes per launch of `name` in `workload` from the committed ncu
    summary (profiles/traffic.txt: name, sha256[:16] of the kernel source,
    workload, bytes), or None when it was taken on another version of the
    kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    src = os.path.join(ROOT, "mxfp4_routed_expert_03_gb300", "csrc", source)
    if not (os.path.exists(path) and os.path.exists(src)):
        return None
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    for line in open(path):
        parts = line.split()
        if len(parts) == 4 and parts[0] == name and parts[1] == sha and parts[2] == workload:
            return float(parts[3])
    return None


def run_ours(args):
    import numpy as np
    import torch
    import synth
    import mxfp4_routed_expert_03_gb300 as moe
    from mxfp4_routed_expert_03_gb300 import (MOE_PROF_DECODE_GATEUP, MOE_PROF_FORWARD_GEMM1,
                                              MOE_PROF_NONE, MOE_ROUTER_XWR, check,
                                              moe_profile_kernel)
    from mxfp4_routed_expert_03_gb300.layer import Layer, Plan, alloc_weights

    n_exp = args.experts or N_EXPERTS
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    wl = dict(BENCH_WORKLOADS[args.workload])
    if args.tokens:
        wl["Ts"] = [args.tokens]
    path = args.path or wl["path"]
    base = base_workload(args.workload)

    # weights: the full layer, generated in HBM by the device half of the generator
    weights = alloc_weights(n_exp, D_MODEL, D_FF)
    synth.dev_fill_layer(base.seed, n_exp, D_MODEL, D_FF,
                         {k: v.data_ptr() for k, v in weights.items()},
                         torch.cuda.current_stream().cuda_stream,
                         dist=wl.get("codes", synth.CODES_UNIFORM))
    use_router = bool(wl.get("router"))
    n_slots = wl.get("stream_slots")
    store_info = None
    n_sets = wl.get("sets", N_SETS)
    if use_router:
        import dataclasses
        w_router = torch.from_numpy(synth.make_w_router(dataclasses.replace(base, E=n_exp))).to(dev)
        shared = {k: torch.from_numpy(v.view(np.int16)).to(dev)
                  for k, v in synth.make_shared(base).items()}
        layer = Layer(D_MODEL, D_FF, n_exp, TOP_K, weights, MOE_ROUTER_XWR, w_router, shared)
    elif n_slots:
        # the store: all experts in pinned host memory; the layer caches n_slots in HBM
        from mxfp4_routed_expert_03_gb300.layer import StreamingLayer
        host = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in weights.items()}
        for k, v in weights.items():
            host[k].copy_(v)
        del weights
        torch.cuda.empty_cache()
        if wl.get("store"):
            # the compressed store, built by the library's host encoder
            from mxfp4_routed_expert_03_gb300.layer import ExpertStore
            t_enc = time.perf_counter()
            store = ExpertStore(n_exp, D_MODEL, D_FF, host)
            store_info = {"encode_s": time.perf_counter() - t_enc,
                          "stored_over_raw": store.blob_bytes / store.raw_bytes}
            del host
            layer = StreamingLayer(D_MODEL, D_FF, n_exp, TOP_K, None, min(n_slots, n_exp),
                                   store=store)
        else:
            layer = StreamingLayer(D_MODEL, D_FF, n_exp, TOP_K, host, min(n_slots, n_exp))
    else:
        layer = Layer(D_MODEL, D_FF, n_exp, TOP_K, weights)
    def path_of(T):
        if path == "auto":
            return "decode" if T <= CROSSOVER_T else "forward"
        return path
    if use_router or any(path_of(T) == "forward" for T in wl["Ts"]):
        layer.prepare()
    stream = torch.cuda.current_stream()

    # inputs: seeded (x, logits) sets per batch size, resident in HBM (x only
    # when the library computes the logits)
    batches = []
    for T in wl["Ts"]:
        w = synth.Workload(base.name, T=T, D=D_MODEL, F=D_FF, E=n_exp, k=TOP_K,
                           seed=base.seed, zipf_s=base.zipf_s)
        xs_h = [synth.make_x(w, rank * 97 + i) for i in range(n_sets)]
        ls_h = [np.zeros((T, n_exp), np.float32) if use_router else
                synth.make_logits(w, rank * 97 + i) for i in range(n_sets)]
        xs = [torch.from_numpy(a.view(np.int16)).to(dev) for a in xs_h]
        ls = [torch.from_numpy(a).to(dev) for a in ls_h]
        pin_x = [torch.from_numpy(a.view(np.int16)).pin_memory() for a in xs_h]
        pin_l = [torch.from_numpy(a).pin_memory() for a in ls_h]
        batches.append({"T": T, "x": xs, "l": ls, "px": pin_x, "pl": pin_l,
                        "plan": Plan(T, n_exp, TOP_K),
                        "out": torch.empty((T, D_MODEL), dtype=torch.int16, device=dev),
                        "dx": torch.empty((T, D_MODEL), dtype=torch.int16, device=dev),
                        "dl": torch.empty((T, n_exp), dtype=torch.float32, device=dev),
                        "hout": torch.empty((T, D_MODEL), dtype=torch.int16).pin_memory(),
                        "path": path_of(T)})
    for b in batches:  # size the workspace once for the largest call
        for op in (0, 1, 2):
            layer.workspace(b["T"], op)
    # the kernel whose launches are timed in each batch: the path's main one
    main_kind = {"decode": MOE_PROF_DECODE_GATEUP,
                 "forward": moe.MOE_PROF_STREAM_COPY if n_slots else MOE_PROF_FORWARD_GEMM1}

    def step(i, events=None, e2e=False, prof_kind=None):
        for bi, b in enumerate(batches):
            s = i % n_sets
            run = layer.decode if b["path"] == "decode" else layer.forward
            if events is not None:
                ev0, ev1 = events[bi]
                kind = prof_kind if prof_kind is not None else main_kind[b["path"]]
                check(moe_profile_kernel(layer.h, kind, ev0, ev1), "profile")
            if e2e:
                b["dx"].copy_(b["px"][s], non_blocking=True)
                if not use_router:
                    b["dl"].copy_(b["pl"][s], non_blocking=True)
                x, lg = b["dx"], b["dl"]
            else:
                x, lg = b["x"][s], b["l"][s]
            if use_router:
                check(layer.plan(b["T"], None, x, b["plan"], stream), "moe_plan")
            else:
                check(layer.plan(b["T"], lg, None, b["plan"], stream), "moe_plan")
            check(run(b["T"], x, b["plan"], b["out"], stream), "moe_" + b["path"])
            if e2e:
                b["hout"].copy_(b["out"], non_blocking=True)

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    sampler = ClockSampler(gpu_id)
    for i in range(args.warmup):
        step(i)
    barrier()
    # per-launch events of the dominant kernel over the timed region
    n_b = len(batches)
    kev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(n_b)] for _ in range(args.steps)]
    for row in kev:
        for a, b in row:
            a.record()
            b.record()
    torch.cuda.synchronize()
    stats0 = layer.stats() if n_slots else None
    t_start = time.time()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(args.steps):
        step(args.warmup + i, events=kev[i])
    e1.record()
    barrier()
    t_end = time.time()
    check(moe_profile_kernel(layer.h, MOE_PROF_NONE), "profile")
    stats1 = layer.stats() if n_slots else None
    elapsed_ms = e0.elapsed_time(e1)
    kern_ms = [[a.elapsed_time(b) for (a, b) in row] for row in kev]
    check(layer.status(), "device status")

    # end to end through the same calls with host buffers (copies inside the region)
    for i in range(args.warmup):
        step(i, e2e=True)
    barrier()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record()
    for i in range(args.steps):
        step(args.warmup + i, e2e=True)
    f1.record()
    barrier()
    e2e_ms = f0.elapsed_time(f1)
    sampler.stop()
    clocks = sampler.summary(t_start, t_end)

    elapsed_ms, e2e_ms = max_over_ranks([elapsed_ms, e2e_ms], dist, dev)

    # per-kernel breakdown (separate untimed pass, one kernel bracketed at a time)
    breakdown = {}
    kinds = []
    if any(b["path"] == "decode" for b in batches):
        kinds += [("decode_gateup", moe.MOE_PROF_DECODE_GATEUP), ("decode_down", moe.MOE_PROF_DECODE_DOWN)]
    if any(b["path"] == "forward" for b in batches):
        kinds += [("gemm1_gateup", moe.MOE_PROF_FORWARD_GEMM1), ("gemm2_down", moe.MOE_PROF_FORWARD_GEMM2)]
    if n_slots:
        kinds += [("stream_copy", moe.MOE_PROF_STREAM_COPY)]
    if use_router:
        kinds += [("router", moe.MOE_PROF_ROUTER), ("shared_gateup", moe.MOE_PROF_SHARED_GATEUP),
                  ("shared_down", moe.MOE_PROF_SHARED_DOWN)]
    n_bd = min(args.steps, 5)
    for name, kid in kinds:
        ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n_b)] for _ in range(n_bd)]
        for row in ev:
            for a, b in row:
                a.record()
                b.record()
        for i in range(n_bd):
            step(i, events=ev[i], prof_kind=kid)
        torch.cuda.synchronize()
        # mean per call of the batches that launch this kernel
        used = [bi for bi, b in enumerate(batches)
                if (b["path"] == "decode") == name.startswith("decode") or name in
                ("router", "shared_gateup", "shared_down")]
        breakdown[name] = float(np.mean([ev[i][bi][0].elapsed_time(ev[i][bi][1])
                                         for i in range(n_bd) for bi in used]))
    check(moe_profile_kernel(layer.h, MOE_PROF_NONE), "profile")
    tokens_step = sum(wl["Ts"])
    value = job_tokens_per_s(world, tokens_step, args.steps, elapsed_ms)
    e2e_value = job_tokens_per_s(world, tokens_step, args.steps, e2e_ms)

    # roofline of the dominant kernel: the timed kernel (per batch, its path's
    # main kernel) with the largest share of the timed region; its bound is
    # the one its arithmetic intensity puts it under
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) \
        if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    hbm_peak = peaks.get("hbm_gbs", 6800.0)
    fp8_peak = 2.0 * peaks.get("bf16_tflops", 1900.0)  # kind::mxf8f6f4 runs at the FP8 rate
    act = [int(b["plan"].active[0].item()) for b in batches]
    per_batch_ms = np.mean(np.array(kern_ms), axis=0)   # mean launch time per batch
    kinds_t = {}
    for bi, b in enumerate(batches):
        kinds_t.setdefault(b["path"], []).append(bi)
    dom = max(kinds_t, key=lambda k: sum(per_batch_ms[bi] for bi in kinds_t[k]))
    bis = kinds_t[dom]
    ms_avg = float(np.mean([per_batch_ms[bi] for bi in bis]))
    if dom == "decode":
        # gate/up kernel: active experts' gate+up codes and scales, f16 x rows read,
        # f16 h and its exponents written (active counts from the last step's plans)
        nbytes = [act[bi] * GATEUP_BYTES + wl["Ts"][bi] * D_MODEL * 2 +
                  wl["Ts"][bi] * TOP_K * (D_FF * 2 + D_FF // 32) for bi in bis]
        nflop = [2.0 * wl["Ts"][bi] * TOP_K * 2 * D_MODEL * D_FF for bi in bis]
        kname, src, tkey = "moe_decode_gateup_kernel", "decode.cu", args.workload
    else:
        # GEMM1: active experts' gate+up weights, two-term activation tiles in,
        # two-term h tiles out (one byte per term and element)
        nbytes = [act[bi] * GATEUP_BYTES + wl["Ts"][bi] * TOP_K * (2 * D_MODEL + 2 * D_FF)
                  for bi in bis]
        nflop = [2.0 * wl["Ts"][bi] * TOP_K * 2 * D_MODEL * D_FF for bi in bis]
        kname, src, tkey = "moe_grouped_gemm_kernel<0>", "grouped_gemm.cu", args.workload
    b_avg, f_avg = float(np.mean(nbytes)), float(np.mean(nflop))
    gbs = b_avg / (ms_avg * 1e-3) / 1e9
    tfs = f_avg / (ms_avg * 1e-3) / 1e12
    mem_bound = (b_avg / hbm_peak) >= (f_avg / 1e3 / fp8_peak)  # time at peak: bytes vs flops
    src_peak = "measured" if peaks else "fallback"
    if mem_bound:
        roof = {"bound": "hbm", "kernel": kname, "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                "frac": gbs / hbm_peak, "peak_source": src_peak + " (copy bandwidth)",
                "bytes_per_launch": b_avg, "tensor_TFLOPs": tfs, "frac_of_fp8_peak": tfs / fp8_peak}
    else:
        roof = {"bound": "tensor", "kernel": kname, "achieved": tfs, "peak": fp8_peak,
                "unit": "TFLOP/s", "frac": tfs / fp8_peak,
                "peak_source": src_peak + " bf16 x 2 (FP8 rate; the two-term activation split "
                               "issues 2 MMAs per algorithmic one, so frac <= 0.5)",
                "flop_per_launch": f_avg, "hbm_GBs": gbs, "frac_of_hbm": gbs / hbm_peak}
    roof["frac_of_fp4_peak"] = tfs / (6.0 * peaks.get("bf16_tflops", 1900.0))
    roof["traffic"] = kernel_traffic(kname, src, tkey)
    stream_info = None
    if n_slots:
        # the copy of the missing experts is bound by the host-to-device link:
        # miss bytes in the timed region over the summed copy-kernel time, against
        # the link's copy bandwidth measured here (pinned host -> device, 2 GiB)
        hits = stats1[0] - stats0[0]
        misses = stats1[1] - stats0[1]
        copy_ms = float(np.sum(np.array(kern_ms)))
        link = torch.empty(1 << 31, dtype=torch.uint8, pin_memory=True)
        dst = torch.empty(1 << 31, dtype=torch.uint8, device=dev)
        best = None
        for _ in range(3):
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record()
            dst.copy_(link, non_blocking=True)
            a1.record()
            torch.cuda.synchronize()
            t = a0.elapsed_time(a1)
            best = t if best is None else min(best, t)
        h2d = (1 << 31) / (best * 1e-3) / 1e9
        del link, dst
        # bytes crossing the link per missing expert: the expert itself, or
        # from a store its stored tiles (the store's mean per expert)
        store = getattr(layer, "store", None)
        link_bytes = store.blob_bytes / n_exp if store is not None else EXPERT_BYTES
        gbs_c = misses * link_bytes / (copy_ms * 1e-3) / 1e9 if copy_ms > 0 else 0.0
        roof = {"bound": "host-to-device link",
                "kernel": "moe_store_decode_kernel" if store is not None else "moe_stream_copy_kernel",
                "achieved": gbs_c, "peak": h2d, "unit": "GB/s",
                "frac": gbs_c / h2d if h2d else None,
                "peak_source": "measured in this run: cudaMemcpyAsync of 2 GiB pinned host memory "
                               "to the device",
                "bytes_per_launch": misses * link_bytes / max(1, args.steps * len(batches)),
                "traffic": None}
        stream_info = {"slots": layer.n_slots, "hit_rate": hits / max(1, hits + misses),
                       "misses_per_step": misses / args.steps,
                       "copy_ms_per_step": copy_ms / args.steps}
        if store is not None:
            roof["decoded_GBs"] = misses * EXPERT_BYTES / (copy_ms * 1e-3) / 1e9 if copy_ms > 0 else 0.0
            roof["link_bytes_per_expert"] = "stored bytes, the store's mean per expert"
            stream_info["store"] = store_info

    # plan: one fused kernel for T <= 64, else top-k, count, scan, scatter;
    # decode: gate/up, down, combine; forward: quant, schedule, gather, two GEMMs,
    # finalize (T <= 16: one fused quant/gather kernel, two GEMMs, finalize)
    launches = 0
    for b in batches:
        launches += 1 if b["T"] <= 64 else 4
        launches += 3 if b["path"] == "decode" else (4 if b["T"] <= 16 else 6)
        if n_slots:
            launches += 4   # cache: replacement, copy of the misses, two scale re-layouts
        if use_router:
            launches += 1 + 2   # router GEMM; shared gate/up and down GEMMs
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": " / ".join(sorted({"mxfp4 x f16 -> f32" if b["path"] == "decode" else
                                    "mxfp4 x 2-term e4m3 -> f32" for b in batches})),
        "data": "synthetic (seeded Philox weights, N(0,1) activations and logits)",
        "config": {"workload": wl["desc"],
                   "path": ("moe_plan (router)" if use_router else "moe_plan") + " + " +
                           ", ".join(f"moe_{b['path']} (T={b['T']})" for b in batches),
                   "tokens_per_step": tokens_step, "active_experts_last_step": act,
                   "kernel_ms_per_call": breakdown,
                   **({"expert_cache": stream_info} if stream_info else {}),
                   "l2": f"inputs larger than L2: a step reads {sum(act) * EXPERT_BYTES / 1e6:.0f} MB "
                         f"of expert weights (L2 129 MB) before any batch recurs, and "
                         f"{wl.get('sets', N_SETS)} rotating logit sets change the experts of "
                         "each batch from step to step",
                   "parallelism": f"replicas x{world}"},
        "roofline": roof,
        **({"profiling_case": f"{n_exp} experts, batches {wl['Ts']}; not a bench value"}
           if n_exp != N_EXPERTS or args.tokens else {}),
        "e2e": {"value": e2e_value, "unit": "tokens/s",
                "h2d_bytes_per_step": sum(T * D_MODEL * 2 + (0 if use_router else T * n_exp * 4)
                                          for T in wl["Ts"]),
                "d2h_bytes_per_step": sum(T * D_MODEL * 2 for T in wl["Ts"])},
        "gpu_launches": launches * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tps, tok, el, threads = oracle_tokens_per_s(args.workload, args.cpu_seconds)
        line["cpu_baseline"] = {"value": tps, "unit": "tokens/s", "cores": threads,
                                "kind": "oracle",
                                "sample": f"{tok} tokens of the {args.workload} workload "
                                          f"in {el:.1f} s (full routing of each batch, expert FFN "
                                          "of the sampled token, fp64)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    layer.close()
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    args = parse_args()
    use_shape(BENCH_WORKLOADS[args.workload])
    if args.steps is None:
        args.steps = 1000 if args.workload in ("decode", "mimo_decode") else 60
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
