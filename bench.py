#!/usr/bin/env python3
"""Benchmark of the GB300 routed-expert FFN library: prints one JSON line.

Default workload (the headline): one K3-shaped routed layer (d_model 7168,
d_ff 1536, 896 experts, top-16, MXFP4 weights resident in HBM), decode
batches of T = 1, 4 and 16 tokens; one step = moe_plan + the expert FFN for
each of the three batches (21 tokens). The FFN call of each batch takes the
faster entry point as measured on GB300, which is moe_forward (tcgen05
grouped GEMMs) at every batch size, down to one token; CROSSOVER_T keeps the
rule explicit, and `--path decode|forward` forces one of them.

The default run adds, in the same line under "workloads", one record per
workload measured on the same generated layer: decode_T1, decode_T4,
decode_T16, prefill4k (T = 4096, uniform routing), skewed8k (T = 8192,
Zipf-skewed routing) and router16k (T = 16384, the library's own fp32 router
x . W_r plus one bf16 shared expert). Each record has its time per step,
tokens/s (device-resident inputs and end to end), its dominant kernel's mean
launch time with the roofline that bounds it, and the clocks of its timed
window. `--workload NAME` times one workload alone.

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
    "decode_T1": {"Ts": [1], "path": "forward",
                  "desc": "K3 routed layer decode, T=1 (one token per step)"},
    "decode_T4": {"Ts": [4], "path": "forward", "desc": "K3 routed layer decode, T=4"},
    "decode_T16": {"Ts": [16], "path": "forward", "desc": "K3 routed layer decode, T=16"},
    "prefill4k": {"Ts": [4096], "path": "forward",
                  "desc": "K3 routed layer prefill, T=4096, uniform routing"},
    "decode_fp8": {"Ts": [1, 4, 16], "path": "decode", "fp8": True, "base": "decode1",
                   "desc": "K3-shaped FP8 (E4M3FN, fp32 scale per 128 x 128) routed layer decode, "
                           "T=1,4,16, fused CUDA-core GEMV (moe_decode)"},
    "prefill4k_fp8": {"Ts": [4096], "path": "forward", "fp8": True, "base": "prefill4k",
                      "desc": "K3-shaped FP8 routed layer prefill, T=4096, bf16 tensor-core GEMMs "
                              "on the bf16 copy moe_prepare makes (BF16-dequant prefill)"},
    "prefill4k_fp4": {"Ts": [4096], "path": "forward", "act": 1, "base": "prefill4k",
                      "desc": "K3 routed layer prefill, T=4096, uniform routing, FP4 x FP4 mode "
                              "(MXFP4 activations, kind::mxf4; not the parity path)"},
    "router16k_fp4": {"Ts": [16384], "path": "forward", "router": True, "sets": 2, "act": 1,
                      "base": "router16k",
                      "desc": "K3 routed layer long prefill, T=16384, in-library fp32 router + "
                              "one bf16 shared expert, FP4 x FP4 mode for the routed experts"},
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
    ap.add_argument("--no-records", action="store_true",
                    help="the headline workload only (no per-workload records)")
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
def bind_host_to_gpu(uuid: str):
    """Runs this process on the CPU cores NVML names as the GPU's neighbours
    (a read-only query), so the pinned host buffers of the end-to-end pass are
    placed in memory next to it. Returns the cores, or None when NVML is not
    there or names none (the process then keeps its cores)."""
    import ctypes
    try:
        nvml = ctypes.CDLL("libnvidia-ml.so.1")
    except OSError:
        return None
    if nvml.nvmlInit_v2() != 0:
        return None
    try:
        dev = ctypes.c_void_p()
        if nvml.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(dev)) != 0:
            return None
        words = ((os.cpu_count() or 64) + 63) // 64
        mask = (ctypes.c_ulong * words)()
        if nvml.nvmlDeviceGetCpuAffinity(dev, ctypes.c_uint(words), mask) != 0:
            return None
        cpus = {64 * i + b for i in range(words) for b in range(64) if (mask[i] >> b) & 1}
        cpus &= os.sched_getaffinity(0)
        if not cpus:
            return None
        os.sched_setaffinity(0, cpus)
        return sorted(cpus)
    except (AttributeError, OSError):
        return None
    finally:
        nvml.nvmlShutdown()


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
                 "--format=csv,noheader,nounits", "-lms", "50"],
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


# ---------------------------------------------------------------------------
# GPU arm: one generated layer, shared by every workload measured in the run
# ---------------------------------------------------------------------------
class Ctx:
    """Device state of a run: the routed layer's weights (generated in HBM
    once, by the device half of the seeded generator) and the library handles
    built over them."""

    def __init__(self, args, n_exp, dev, rank, world, dist):
        self.args, self.n_exp, self.dev = args, n_exp, dev
        self.rank, self.world, self.dist = rank, world, dist
        self.weights = {}     # code distribution -> weight tensors
        self.layers = {}      # kind -> Layer

    def layer_weights(self, codes, seed):
        """The layer's weights under E2M1 code distribution `codes`, or the FP8
        lane's (codes == "fp8")."""
        import torch
        import synth
        from mxfp4_routed_expert_03_gb300.layer import alloc_fp8_weights, alloc_weights
        if codes not in self.weights:
            stream = torch.cuda.current_stream().cuda_stream
            if codes == "fp8":
                w = alloc_fp8_weights(self.n_exp, D_MODEL, D_FF)
                synth.dev_fill_fp8_layer(seed, self.n_exp, D_MODEL, D_FF,
                                         {k: v.data_ptr() for k, v in w.items()}, stream)
            else:
                w = alloc_weights(self.n_exp, D_MODEL, D_FF)
                synth.dev_fill_layer(seed, self.n_exp, D_MODEL, D_FF,
                                     {k: v.data_ptr() for k, v in w.items()}, stream, dist=codes)
            self.weights[codes] = w
        return self.weights[codes]

    def barrier(self):
        import torch
        torch.cuda.synchronize()
        if self.dist is not None:
            self.dist.barrier()
        torch.cuda.synchronize()

    def close(self):
        for layer in self.layers.values():
            layer.close()
        self.layers.clear()


def make_layer(ctx, wl, base):
    """The library handle a workload runs on (built once per kind and kept)."""
    import dataclasses
    import numpy as np
    import torch
    import synth
    from mxfp4_routed_expert_03_gb300 import MOE_ROUTER_XWR
    from mxfp4_routed_expert_03_gb300.layer import Layer
    codes = "fp8" if wl.get("fp8") else wl.get("codes", synth.CODES_UNIFORM)
    n_slots = wl.get("stream_slots")
    act = wl.get("act", 0)
    wfmt = 1 if wl.get("fp8") else 0   # MOE_W_FP8 / MOE_W_MXFP4
    kind = ("router" if wl.get("router") else "stream_store" if wl.get("store") else
            "stream" if n_slots else "plain", codes, act)
    if kind in ctx.layers:
        return ctx.layers[kind], None
    weights = ctx.layer_weights(codes, base.seed)
    info = None
    if wl.get("router"):
        w_router = torch.from_numpy(
            synth.make_w_router(dataclasses.replace(base, E=ctx.n_exp))).to(ctx.dev)
        shared = {k: torch.from_numpy(v.view(np.int16)).to(ctx.dev)
                  for k, v in synth.make_shared(base).items()}
        layer = Layer(D_MODEL, D_FF, ctx.n_exp, TOP_K, weights, MOE_ROUTER_XWR, w_router, shared,
                      act_mode=act)
    elif n_slots:
        # the slow tier: all experts in pinned host memory; the layer caches
        # n_slots of them in HBM
        from mxfp4_routed_expert_03_gb300.layer import StreamingLayer
        host = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in weights.items()}
        for k, v in weights.items():
            host[k].copy_(v)
        if wl.get("store"):
            from mxfp4_routed_expert_03_gb300.layer import ExpertStore
            t_enc = time.perf_counter()
            store = ExpertStore(ctx.n_exp, D_MODEL, D_FF, host)
            info = {"encode_s": time.perf_counter() - t_enc,
                    "stored_over_raw": store.blob_bytes / store.raw_bytes}
            del host
            layer = StreamingLayer(D_MODEL, D_FF, ctx.n_exp, TOP_K, None,
                                   min(n_slots, ctx.n_exp), store=store, act_mode=act)
        else:
            layer = StreamingLayer(D_MODEL, D_FF, ctx.n_exp, TOP_K, host, min(n_slots, ctx.n_exp),
                                   act_mode=act)
    else:
        layer = Layer(D_MODEL, D_FF, ctx.n_exp, TOP_K, weights, act_mode=act, weight_format=wfmt)
    if wl["path"] != "decode" or not wl.get("fp8"):
        layer.prepare()   # (the FP8 decode reads the codes; its bf16 copy serves moe_forward)
    ctx.layers[kind] = layer
    return layer, info


def pad256(a):
    """A byte array zero-padded to a multiple of 256 bytes (keeps every input
    in the end-to-end step buffer 256-byte aligned)."""
    import numpy as np
    return np.concatenate([a, np.zeros((-len(a)) % 256, np.uint8)])


def make_batches(ctx, wl, base, path_of, use_router):
    """Seeded (x, logits) sets per batch size, resident in HBM (x only when the
    library computes the logits), their pinned host copies for the end-to-end
    pass, plan and output buffers. For the end-to-end pass the inputs of all
    of a step's batches (x, then the logits, per batch) sit side by side in
    one pinned buffer per set and the outputs in one device buffer, so a step
    moves its inputs with one copy and its outputs with one."""
    import numpy as np
    import torch
    import synth
    from mxfp4_routed_expert_03_gb300.layer import Plan
    n_sets = wl.get("sets", N_SETS)
    batches = []
    step_in = [[] for _ in range(n_sets)]   # per set: each batch's x and logits bytes
    for T in wl["Ts"]:
        w = synth.Workload(base.name, T=T, D=D_MODEL, F=D_FF, E=ctx.n_exp, k=TOP_K,
                           seed=base.seed, zipf_s=base.zipf_s)
        xs_h = [synth.make_x(w, ctx.rank * 97 + i) for i in range(n_sets)]
        ls_h = [np.zeros((T, ctx.n_exp), np.float32) if use_router else
                synth.make_logits(w, ctx.rank * 97 + i) for i in range(n_sets)]
        dev = ctx.dev
        for i, (a, l) in enumerate(zip(xs_h, ls_h)):
            step_in[i].append(pad256(a.view(np.uint8).reshape(-1)))
            if not use_router:
                step_in[i].append(pad256(l.view(np.uint8).reshape(-1)))
        batches.append({"T": T,
                        "x": [torch.from_numpy(a.view(np.int16)).to(dev) for a in xs_h],
                        "l": [torch.from_numpy(a).to(dev) for a in ls_h],
                        "plan": Plan(T, ctx.n_exp, TOP_K),
                        "out": torch.empty((T, D_MODEL), dtype=torch.int16, device=dev),
                        "path": path_of(T)})
    # the end-to-end pass's step buffers (every piece a multiple of 16 bytes)
    nin = sum(len(p) for p in step_in[0])
    pin = []
    for parts in step_in:
        buf = torch.empty(sum(len(p) for p in parts), dtype=torch.uint8).pin_memory()
        buf.copy_(torch.from_numpy(np.concatenate(parts)))
        pin.append(buf)
    din = torch.empty(pin[0].numel(), dtype=torch.uint8, device=ctx.dev)
    tot = sum(wl["Ts"])
    dout = torch.empty((tot, D_MODEL), dtype=torch.int16, device=ctx.dev)
    hout = torch.empty((tot, D_MODEL), dtype=torch.int16).pin_memory()
    off, row = 0, 0
    for b in batches:
        T = b["T"]
        xb, lb = T * D_MODEL * 2, (0 if use_router else T * ctx.n_exp * 4)
        b["dx"] = din[off:off + xb].view(torch.int16).view(T, D_MODEL)
        off += -(-xb // 256) * 256
        b["dl"] = (din[off:off + lb].view(torch.float32).view(T, ctx.n_exp) if lb else
                   torch.empty((T, ctx.n_exp), dtype=torch.float32, device=ctx.dev))
        off += -(-lb // 256) * 256
        b["dout"] = dout[row:row + T]
        row += T
    assert off == nin == din.numel()
    step_io = {"pin": pin, "din": din, "dout": dout, "hout": hout}
    return batches, step_io


def kernel_work(path: str, T: int, active: int, fp4: bool = False, fp8: bool = False):
    """Algorithmic bytes and flops of one launch of a batch's dominant kernel:
    the gate/up GEMM of moe_forward (active experts' gate+up weights, the
    two-term activation rows in and the two-term h rows out, one byte per
    term and element; in the FP4 x FP4 mode one MXFP4 term, half a byte per
    element plus a scale byte per 32) or the gate/up kernel of moe_decode
    (the same weights, bf16 x rows in, f16 h rows and their exponents out)."""
    flop = 2.0 * T * TOP_K * 2 * D_MODEL * D_FF
    if fp8:
        # FP8 lane: decode streams one code byte per weight (+ its block scales);
        # the prefill GEMM streams the bf16 copy (2 bytes per weight) and bf16
        # activation rows in and h rows out
        nb = lambda n: (n + 127) // 128
        if path == "decode":
            wb = 2 * (D_FF * D_MODEL + 4 * nb(D_FF) * nb(D_MODEL))
            nbytes = active * wb + T * D_MODEL * 2 + T * TOP_K * (D_FF * 2 + D_FF // 32)
        else:
            nbytes = active * 2 * D_FF * D_MODEL * 2 + T * TOP_K * (2 * D_MODEL + 2 * D_FF)
    elif path == "decode":
        nbytes = active * GATEUP_BYTES + T * D_MODEL * 2 + T * TOP_K * (D_FF * 2 + D_FF // 32)
    elif fp4:
        nbytes = active * GATEUP_BYTES + T * TOP_K * (D_MODEL // 2 + D_MODEL // 32 +
                                                      D_FF // 2 + D_FF // 32)
    else:
        nbytes = active * GATEUP_BYTES + T * TOP_K * (2 * D_MODEL + 2 * D_FF)
    return float(nbytes), flop


def roofline(path, nbytes, flop, ms, peaks, workload, fp4=False, fp8=False):
    """Roofline of the dominant kernel: achieved algorithmic bytes or flops per
    launch over its mean launch time, against the measured peak of the bound
    its arithmetic intensity puts it under."""
    hbm_peak = peaks.get("hbm_gbs", 6800.0)
    fp8_peak = 2.0 * peaks.get("bf16_tflops", 1900.0)  # kind::mxf8f6f4 runs at the FP8 rate
    fp4_peak = 6.0 * peaks.get("bf16_tflops", 1900.0)  # kind::mxf4 (nominal 13.5 / 2.25)
    src = "measured" if peaks else "fallback"
    gbs = nbytes / (ms * 1e-3) / 1e9
    tfs = flop / (ms * 1e-3) / 1e12
    bf16_peak = peaks.get("bf16_tflops", 1900.0)
    if path == "decode":
        kname, csrc = "moe_decode_gateup_kernel", "decode.cu"
        tensor_time = 0.0   # CUDA cores: bound by bytes
    elif fp8:
        kname, csrc = "moe_grouped_gemm_kernel<0,bf16>", "grouped_gemm.cu"
        tensor_time = flop / 1e12 / bf16_peak        # kind::f16 on the bf16 copy
    elif fp4:
        kname, csrc = "moe_grouped_gemm_kernel<0,fp4>", "grouped_gemm.cu"
        tensor_time = flop / 1e12 / fp4_peak          # one MXFP4 term, kind::mxf4
    else:
        kname, csrc = "moe_grouped_gemm_kernel<0>", "grouped_gemm.cu"
        tensor_time = 2.0 * flop / 1e12 / fp8_peak   # two MMAs per algorithmic one
    mem_bound = nbytes / 1e9 / hbm_peak >= tensor_time
    if mem_bound:
        r = {"bound": "hbm", "kernel": kname, "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
             "frac": gbs / hbm_peak, "peak_source": src + " (copy bandwidth)"}
    elif fp8:
        r = {"bound": "tensor", "kernel": kname, "achieved": tfs, "peak": bf16_peak,
             "unit": "TFLOP/s", "frac": tfs / bf16_peak, "peak_source": src + " bf16 (burst)",
             "hbm_GBs": gbs, "frac_of_hbm": gbs / hbm_peak}
    elif fp4:
        r = {"bound": "tensor", "kernel": kname, "achieved": tfs, "peak": fp4_peak,
             "unit": "TFLOP/s", "frac": tfs / fp4_peak,
             "peak_source": src + " bf16 x 6 (FP4 rate, nominal 13.5 / 2.25)",
             "hbm_GBs": gbs, "frac_of_hbm": gbs / hbm_peak}
    else:
        r = {"bound": "tensor", "kernel": kname, "achieved": tfs, "peak": fp8_peak,
             "unit": "TFLOP/s", "frac": tfs / fp8_peak,
             "peak_source": src + " bf16 x 2 (FP8 rate; the two-term activation split issues 2 "
                                  "MMAs per algorithmic one, so frac <= 0.5)",
             "hbm_GBs": gbs, "frac_of_hbm": gbs / hbm_peak}
    r.update({"bytes_per_launch": nbytes, "flop_per_launch": flop, "kernel_ms": ms,
              "tensor_TFLOPs": tfs, "frac_of_fp8_peak": tfs / fp8_peak,
              "frac_of_fp4_peak": tfs / fp4_peak,
              "binding_roof_ms": max(nbytes / 1e9 / hbm_peak, tensor_time) * 1e3,
              "traffic": kernel_traffic(kname, csrc, workload)})
    r["frac_of_binding_roof"] = r["binding_roof_ms"] / ms
    return r


def measure(ctx, name, wl, steps, warmup, sampler, peaks, breakdown=True, path_override=None):
    """Time `steps` steps of workload `name` (after `warmup` untimed ones) on
    device-resident inputs, then the same steps end to end (host inputs copied
    in and the output read back inside the timed region). Returns the
    workload's record and the figures the headline line adds."""
    import numpy as np
    import torch
    import mxfp4_routed_expert_03_gb300 as moe
    from mxfp4_routed_expert_03_gb300 import check, moe_profile_kernel
    base = base_workload(name)
    layer, store_info = make_layer(ctx, wl, base)
    use_router = bool(wl.get("router"))
    n_slots = wl.get("stream_slots")
    path = path_override or wl["path"]

    def path_of(T):
        if path == "auto":
            return "decode" if T <= CROSSOVER_T else "forward"
        return path
    batches, step_io = make_batches(ctx, wl, base, path_of, use_router)
    n_sets = wl.get("sets", N_SETS)
    for b in batches:  # size the workspace once for the largest call
        for op in (0, 1, 2):
            layer.workspace(b["T"], op)
    stream = torch.cuda.current_stream()
    main_kind = {"decode": moe.MOE_PROF_DECODE_GATEUP,
                 "forward": moe.MOE_PROF_STREAM_COPY if n_slots else moe.MOE_PROF_FORWARD_GEMM1}

    def step(i, events=None, e2e=False, prof_kind=None):
        if e2e:  # the step's inputs, all batches: one copy
            step_io["din"].copy_(step_io["pin"][i % n_sets], non_blocking=True)
        for bi, b in enumerate(batches):
            s = i % n_sets
            run = layer.decode if b["path"] == "decode" else layer.forward
            if events is not None:
                ev0, ev1 = events[bi]
                kind = prof_kind if prof_kind is not None else main_kind[b["path"]]
                check(moe_profile_kernel(layer.h, kind, ev0, ev1), "profile")
            if e2e:
                x, lg = b["dx"], b["dl"]
            else:
                x, lg = b["x"][s], b["l"][s]
            if use_router:
                check(layer.plan(b["T"], None, x, b["plan"], stream), "moe_plan")
            else:
                check(layer.plan(b["T"], lg, None, b["plan"], stream), "moe_plan")
            check(run(b["T"], x, b["plan"], b["dout"] if e2e else b["out"], stream),
                  "moe_" + b["path"])
        if e2e:  # and its outputs: one copy
            step_io["hout"].copy_(step_io["dout"], non_blocking=True)

    def events(n_rows):
        ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in batches] for _ in range(n_rows)]
        for row in ev:
            for a, b in row:
                a.record()
                b.record()
        return ev

    for i in range(warmup):
        step(i)
    ctx.barrier()
    # the timed steps: nothing recorded between the library's launches, so its
    # kernels overlap across boundaries as they do in use
    t_start = time.time()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(steps):
        step(warmup + i)
    e1.record()
    ctx.barrier()
    t_end = time.time()
    elapsed_ms = e0.elapsed_time(e1)
    check(layer.status(), "device status")
    # the same steps again with events around each batch's dominant kernel
    # (its launch durations for the roofline; the events serialise that
    # kernel with its neighbours)
    kev = events(steps)
    torch.cuda.synchronize()
    stats0 = layer.stats() if n_slots else None   # (the cache's misses during these steps)
    for i in range(steps):
        step(warmup + i, events=kev[i])
    ctx.barrier()
    stats1 = layer.stats() if n_slots else None
    check(moe_profile_kernel(layer.h, moe.MOE_PROF_NONE), "profile")
    kern_ms = [[a.elapsed_time(b) for (a, b) in row] for row in kev]
    check(layer.status(), "device status")

    for i in range(warmup):  # end to end through the same calls, host buffers
        step(i, e2e=True)
    ctx.barrier()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record()
    for i in range(steps):
        step(warmup + i, e2e=True)
    f1.record()
    ctx.barrier()
    e2e_ms = f0.elapsed_time(f1)
    clocks = sampler.summary(t_start, t_end)
    elapsed_ms, e2e_ms = max_over_ranks([elapsed_ms, e2e_ms], ctx.dist, ctx.dev)

    # per-kernel breakdown (separate untimed pass, one kernel bracketed at a time)
    bd = {}
    if breakdown:
        kinds = []
        if any(b["path"] == "decode" for b in batches):
            kinds += [("decode_gateup", moe.MOE_PROF_DECODE_GATEUP),
                      ("decode_down", moe.MOE_PROF_DECODE_DOWN)]
        if any(b["path"] == "forward" for b in batches):
            kinds += [("gemm1_gateup", moe.MOE_PROF_FORWARD_GEMM1),
                      ("gemm2_down", moe.MOE_PROF_FORWARD_GEMM2)]
        if n_slots:
            kinds += [("stream_copy", moe.MOE_PROF_STREAM_COPY)]
        if use_router:
            kinds += [("router", moe.MOE_PROF_ROUTER), ("shared_gateup", moe.MOE_PROF_SHARED_GATEUP),
                      ("shared_down", moe.MOE_PROF_SHARED_DOWN)]
        n_bd = min(steps, 5)
        for kname, kid in kinds:
            ev = events(n_bd)
            for i in range(n_bd):
                step(i, events=ev[i], prof_kind=kid)
            torch.cuda.synchronize()
            used = [bi for bi, b in enumerate(batches)
                    if (b["path"] == "decode") == kname.startswith("decode") or kname in
                    ("router", "shared_gateup", "shared_down", "stream_copy")]
            bd[kname] = float(np.mean([ev[i][bi][0].elapsed_time(ev[i][bi][1])
                                       for i in range(n_bd) for bi in used]))
        check(moe_profile_kernel(layer.h, moe.MOE_PROF_NONE), "profile")

    tokens_step = sum(wl["Ts"])
    value = job_tokens_per_s(ctx.world, tokens_step, steps, elapsed_ms)
    e2e_value = job_tokens_per_s(ctx.world, tokens_step, steps, e2e_ms)
    act = [int(b["plan"].active[0].item()) for b in batches]
    per_batch_ms = np.mean(np.array(kern_ms), axis=0)   # mean launch time per batch
    by_path = {}
    for bi, b in enumerate(batches):
        by_path.setdefault(b["path"], []).append(bi)
    dom = max(by_path, key=lambda k: sum(per_batch_ms[bi] for bi in by_path[k]))
    bis = by_path[dom]
    ms_avg = float(np.mean([per_batch_ms[bi] for bi in bis]))
    fp4, fp8 = bool(wl.get("act", 0)), bool(wl.get("fp8"))
    work = [kernel_work(dom, wl["Ts"][bi], act[bi], fp4, fp8) for bi in bis]
    nbytes, nflop = float(np.mean([w_[0] for w_ in work])), float(np.mean([w_[1] for w_ in work]))
    roof = roofline(dom, nbytes, nflop, ms_avg, peaks, name, fp4, fp8)
    stream_info = None
    if n_slots:
        roof, stream_info = stream_roofline(ctx, layer, stats0, stats1, kern_ms, steps,
                                            len(batches), store_info)
    # the bytes the end-to-end steps copy: the step's input buffer (x and
    # logits of every batch, each padded to 256 bytes) and its outputs
    h2d = step_io["din"].numel()
    d2h = step_io["dout"].numel() * step_io["dout"].element_size()
    record = {
        "workload": wl["desc"], "T": wl["Ts"], "dtype": dtype_of(wl, path),
        "path": ("moe_plan (router)" if use_router else "moe_plan") + " + " +
                ", ".join(f"moe_{b['path']} (T={b['T']})" for b in batches),
        "steps": steps, "warmup": warmup, "ms_per_step": elapsed_ms / steps,
        "tokens_per_s": value,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "active_experts_last_step": act,
        "dominant_kernel_ms": ms_avg,
        "roofline": roof,
        "clocks": clocks,
    }
    if bd:
        record["kernel_ms_per_call"] = bd
    if stream_info:
        record["expert_cache"] = stream_info
    # launches of the library's kernels per step: plan (one fused kernel for
    # T <= 64, else top-k, count, scan, scatter); decode: gate/up, down,
    # combine; forward: quant, schedule, gather, two GEMMs, finalize (T <= 16:
    # one fused quant/gather kernel, two GEMMs, finalize)
    launches = 0
    for b in batches:
        launches += 1 if b["T"] <= 64 else 4
        launches += 3 if b["path"] == "decode" else (4 if b["T"] <= 16 else 6)
        if n_slots:
            launches += 4   # cache: replacement, copy of the misses, two scale re-layouts
        if use_router:
            launches += 1 + 2   # router GEMM; shared gate/up and down GEMMs
    record["gpu_launches_per_step"] = launches
    for b in batches:
        del b["x"], b["l"]
    torch.cuda.empty_cache()
    return record


def stream_roofline(ctx, layer, stats0, stats1, kern_ms, steps, n_batches, store_info):
    """Expert streaming: the copy (or store decode) of the missing experts is
    bound by the host-to-device link; miss bytes in the timed region over the
    summed copy-kernel time, against the link's copy bandwidth measured here
    (pinned host -> device, 2 GiB)."""
    import numpy as np
    import torch
    hits = stats1[0] - stats0[0]
    misses = stats1[1] - stats0[1]
    copy_ms = float(np.sum(np.array(kern_ms)))
    link = torch.empty(1 << 31, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(1 << 31, dtype=torch.uint8, device=ctx.dev)
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
    # bytes crossing the link per missing expert: the expert itself, or from a
    # store its stored tiles (the store's mean per expert)
    store = getattr(layer, "store", None)
    link_bytes = store.blob_bytes / ctx.n_exp if store is not None else EXPERT_BYTES
    gbs_c = misses * link_bytes / (copy_ms * 1e-3) / 1e9 if copy_ms > 0 else 0.0
    roof = {"bound": "host-to-device link",
            "kernel": "moe_store_decode_kernel" if store is not None else "moe_stream_copy_kernel",
            "achieved": gbs_c, "peak": h2d, "unit": "GB/s",
            "frac": gbs_c / h2d if h2d else None,
            "peak_source": "measured in this run: cudaMemcpyAsync of 2 GiB pinned host memory "
                           "to the device",
            "bytes_per_launch": misses * link_bytes / max(1, steps * n_batches),
            "traffic": None}
    info = {"slots": layer.n_slots, "hit_rate": hits / max(1, hits + misses),
            "misses_per_step": misses / steps, "copy_ms_per_step": copy_ms / steps}
    if store is not None:
        roof["decoded_GBs"] = misses * EXPERT_BYTES / (copy_ms * 1e-3) / 1e9 if copy_ms > 0 else 0.0
        roof["link_bytes_per_expert"] = "stored bytes, the store's mean per expert"
        info["store"] = store_info
    return roof, info


def dtype_of(wl, path):
    """The arithmetic types a workload's path computes in (operands -> accumulator)."""
    if wl.get("fp8"):
        return "e4m3fn x f16 -> f32" if path == "decode" else "bf16 (from e4m3fn) x bf16 -> f32"
    if wl.get("act", 0):
        return "mxfp4 x mxfp4 -> f32"
    if path == "decode":
        return "mxfp4 x f16 -> f32"
    return "mxfp4 x 2-term e4m3 -> f32"


# Workloads that get a record of their own in the default run's line.
RECORDS = ("decode_T1", "decode_T4", "decode_T16", "prefill4k", "skewed8k", "router16k",
           "prefill4k_fp4", "router16k_fp4", "decode_fp8", "prefill4k_fp8")


def run_ours(args):
    import torch
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
    ctx = Ctx(args, n_exp, dev, rank, world, dist)
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) \
        if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    gpu_uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    host_cpus = bind_host_to_gpu(gpu_uuid)
    sampler = ClockSampler(gpu_uuid)
    wl = dict(BENCH_WORKLOADS[args.workload])
    if args.tokens:
        wl["Ts"] = [args.tokens]
    head = measure(ctx, args.workload, wl, args.steps, args.warmup, sampler, peaks,
                   path_override=args.path)
    records = {}
    if args.workload == "decode" and not (args.no_records or args.experts or args.tokens):
        rec_steps = min(args.steps, 100)   # keeps the default run within a few minutes
        for name in RECORDS:
            records[name] = measure(ctx, name, BENCH_WORKLOADS[name], rec_steps, args.warmup,
                                    sampler, peaks)
    sampler.stop()
    config = {"workload": wl["desc"], "path": head["path"],
              "tokens_per_step": sum(wl["Ts"]),
              "active_experts_last_step": head["active_experts_last_step"],
              "kernel_ms_per_call": head.get("kernel_ms_per_call", {}),
              **({"expert_cache": head["expert_cache"]} if "expert_cache" in head else {}),
              "l2": "inputs larger than L2: every step reads at least 280 MB of expert weights "
                    "(L2 129 MB) and the inputs rotate through "
                    f"{wl.get('sets', N_SETS)} pre-generated sets, so the selected experts "
                    "change from step to step",
              "parallelism": f"replicas x{world}",
              "host_cores": (f"{len(host_cpus)} next to the GPU (NVML affinity)" if host_cpus
                             else "unbound")}
    line = {
        "metric": METRIC, "value": head["tokens_per_s"], "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": dtype_of(wl, args.path or wl["path"]),
        "data": "synthetic (seeded Philox weights, N(0,1) activations and logits)",
        "config": config,
        "roofline": head["roofline"],
        **({"profiling_case": f"{n_exp} experts, batches {wl['Ts']}; not a bench value"}
           if n_exp != N_EXPERTS or args.tokens else {}),
        "e2e": head["e2e"],
        "gpu_launches": head["gpu_launches_per_step"] * args.steps,
        "clocks": head["clocks"],
    }
    if records:
        line["workloads"] = records
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tps, tok, el, threads = oracle_tokens_per_s(args.workload, args.cpu_seconds)
        line["cpu_baseline"] = {"value": tps, "unit": "tokens/s", "cores": threads,
                                "kind": "oracle",
                                "sample": f"{tok} tokens of the {args.workload} workload "
                                          f"in {el:.1f} s (full routing of each batch, expert FFN "
                                          "of the sampled token, fp64)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    ctx.close()
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
