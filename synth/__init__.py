"""Seeded synthetic inputs for the routed-expert FFN workloads.

This module is the only thing the CPU checker (``oracle/``) and the CUDA path
share: it turns (seed, tensor id, expert, row, column) into bytes with
Philox4x32-10 and holds none of the layer's arithmetic. Expert weights come out
as raw E2M1 codes (two per byte) and E8M0 scale bytes; activations, logits and
router weights as bf16 / fp32 normals.

The host half (``synth_host.c``) and the device half (``synth_dev.cu``) emit
identical expert-weight bytes, so a full 896-expert layer (15.7 GB) can be
generated directly in HBM while the CPU checker regenerates only the experts
it needs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_HOST_SO = os.path.join(_HERE, "libsynth_host.so")
_DEV_SO = os.path.join(_HERE, "libsynth_dev.so")
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]

# Tensor ids: second word of the Philox key (kept equal to philox.h).
GATE_Q, UP_Q, DOWN_Q, GATE_S, UP_S, DOWN_S = 1, 2, 3, 4, 5, 6
X, LOGITS, WR, ZIPF, SH_GATE, SH_UP, SH_DOWN = 7, 8, 9, 10, 11, 12, 13
F8_GATE_Q, F8_UP_Q, F8_DOWN_Q, F8_GATE_S, F8_UP_S, F8_DOWN_S = 14, 15, 16, 17, 18, 19

# E8M0 scale bytes uniform over 2^-4 .. 2^0  ->  {123, ..., 127}
SCALE_LO, SCALE_N = 123, 5
# E2M1 code distributions: uniform over the 16 codes, or "peaked" (shaped like
# block-scaled normal weights, half of the zeros negative; see philox.h).
CODES_UNIFORM, CODES_PEAKED = 0, 1


def _newer(target, sources):
    if not os.path.exists(target):
        return False
    t = os.path.getmtime(target)
    return all(os.path.getmtime(s) <= t for s in sources)


def build(device: bool = True, force: bool = False) -> None:
    """Compile the host generator (gcc) and, if asked, the device one (nvcc)."""
    hdr = os.path.join(_HERE, "philox.h")
    src = os.path.join(_HERE, "synth_host.c")
    if force or not _newer(_HOST_SO, [src, hdr]):
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-o", _HOST_SO, src, "-lm"])
    if device:
        dsrc = os.path.join(_HERE, "synth_dev.cu")
        if force or not _newer(_DEV_SO, [dsrc, hdr]):
            subprocess.check_call(["nvcc", *ARCH_FLAGS, "-O3", "-Xcompiler", "-fPIC", "-shared",
                                   "-o", _DEV_SO, dsrc])


_host = None
_dev = None


def _host_lib():
    global _host
    if _host is None:
        if not os.path.exists(_HOST_SO):
            build(device=False)
        L = ctypes.CDLL(_HOST_SO)
        u64, u32, i64, i32, p = (ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int64,
                                 ctypes.c_int, ctypes.c_void_p)
        L.synth_philox.argtypes = [p, p, p]
        L.synth_mx_codes.argtypes = [u64, u32, u32, i64, i64, p]
        L.synth_mx_codes.restype = i32
        L.synth_mx_codes_dist.argtypes = [u64, u32, u32, i64, i64, i32, p]
        L.synth_mx_codes_dist.restype = i32
        L.synth_mx_scales.argtypes = [u64, u32, u32, i64, i64, i32, i32, p]
        L.synth_mx_scales.restype = i32
        L.synth_normal_f32.argtypes = [u64, u32, i64, i64, ctypes.c_double, ctypes.c_double, p]
        L.synth_normal_bf16.argtypes = [u64, u32, i64, i64, ctypes.c_double, p]
        L.synth_zipf_bias.argtypes = [u64, i32, ctypes.c_double, p, p]
        L.synth_fp8_codes.argtypes = [u64, u32, u32, i64, i64, p]
        L.synth_fp8_codes.restype = i32
        L.synth_fp8_scales.argtypes = [u64, u32, u32, i64, i64, p]
        L.synth_fp8_scales.restype = i32
        _host = L
    return _host


def _dev_lib():
    global _dev
    if _dev is None:
        if not os.path.exists(_DEV_SO):
            build(device=True)
        L = ctypes.CDLL(_DEV_SO)
        u64, u32, i64, i32, p = (ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int64,
                                 ctypes.c_int, ctypes.c_void_p)
        L.synth_dev_mx_codes.argtypes = [u64, u32, u32, i64, i64, i64, p, p]
        L.synth_dev_mx_codes.restype = i32
        L.synth_dev_mx_codes_dist.argtypes = [u64, u32, u32, i64, i64, i64, i32, p, p]
        L.synth_dev_mx_codes_dist.restype = i32
        L.synth_dev_mx_scales.argtypes = [u64, u32, u32, i64, i64, i64, i32, i32, p, p]
        L.synth_dev_mx_scales.restype = i32
        L.synth_dev_fp8_codes.argtypes = [u64, u32, u32, i64, i64, i64, p, p]
        L.synth_dev_fp8_codes.restype = i32
        L.synth_dev_fp8_scales.argtypes = [u64, u32, u32, i64, i64, i64, p, p]
        L.synth_dev_fp8_scales.restype = i32
        _dev = L
    return _dev


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def philox(ctr, key):
    """Raw Philox4x32-10: 4 counter words, 2 key words -> 4 output words."""
    c = np.asarray(ctr, dtype=np.uint32).copy()
    k = np.asarray(key, dtype=np.uint32).copy()
    o = np.zeros(4, dtype=np.uint32)
    _host_lib().synth_philox(_ptr(c), _ptr(k), _ptr(o))
    return [int(v) for v in o]


def mx_codes(seed: int, tensor: int, expert: int, rows: int, K: int,
             dist: int = CODES_UNIFORM) -> np.ndarray:
    """Packed E2M1 codes of one expert matrix: uint8 [rows, K/2]."""
    out = np.empty((rows, K // 2), dtype=np.uint8)
    if _host_lib().synth_mx_codes_dist(seed, tensor, expert, rows, K, dist, _ptr(out)) != 0:
        raise ValueError("K must be a multiple of 32 and dist 0 or 1")
    return out


def mx_scales(seed: int, tensor: int, expert: int, rows: int, K: int,
              lo: int = SCALE_LO, n: int = SCALE_N) -> np.ndarray:
    """E8M0 scale bytes of one expert matrix: uint8 [rows, K/32]."""
    out = np.empty((rows, K // 32), dtype=np.uint8)
    if _host_lib().synth_mx_scales(seed, tensor, expert, rows, K, lo, n, _ptr(out)) != 0:
        raise ValueError("bad scale range or K")
    return out


def expert_weights(seed: int, e: int, D: int, F: int, lo: int = SCALE_LO, n: int = SCALE_N,
                   dist: int = CODES_UNIFORM):
    """All six byte arrays of expert e (gate/up: [F, D]; down: [D, F])."""
    return {
        "gate_q": mx_codes(seed, GATE_Q, e, F, D, dist), "gate_s": mx_scales(seed, GATE_S, e, F, D, lo, n),
        "up_q": mx_codes(seed, UP_Q, e, F, D, dist), "up_s": mx_scales(seed, UP_S, e, F, D, lo, n),
        "down_q": mx_codes(seed, DOWN_Q, e, D, F, dist), "down_s": mx_scales(seed, DOWN_S, e, D, F, lo, n),
    }


def fp8_expert_weights(seed: int, e: int, D: int, F: int) -> dict:
    """FP8 (E4M3FN) expert e: codes gate/up [F, D], down [D, F] (uint8) and fp32
    block scales [ceil(rows/128), ceil(K/128)] (see philox.h for the draws)."""
    L = _host_lib()
    out = {}
    for name, tq, ts, rows, K in (("gate", F8_GATE_Q, F8_GATE_S, F, D),
                                  ("up", F8_UP_Q, F8_UP_S, F, D),
                                  ("down", F8_DOWN_Q, F8_DOWN_S, D, F)):
        q = np.empty((rows, K), dtype=np.uint8)
        sc = np.empty(((rows + 127) // 128, (K + 127) // 128), dtype=np.float32)
        if L.synth_fp8_codes(seed, tq, e, rows, K, _ptr(q)) != 0 or \
                L.synth_fp8_scales(seed, ts, e, rows, K, _ptr(sc)) != 0:
            raise ValueError("K must be a multiple of 16")
        out[name + "_q"], out[name + "_s"] = q, sc
    return out


def dev_fill_fp8_layer(seed: int, E: int, D: int, F: int, bufs: dict, stream: int = 0) -> None:
    """Fill a whole FP8 layer on the GPU: ``bufs`` maps gate_q/up_q/down_q
    (E x rows x K bytes) and gate_s/up_s/down_s (E x ceil(rows/128) x
    ceil(K/128) fp32) to device pointers."""
    L = _dev_lib()
    for name, tq, ts, rows, K in (("gate", F8_GATE_Q, F8_GATE_S, F, D),
                                  ("up", F8_UP_Q, F8_UP_S, F, D),
                                  ("down", F8_DOWN_Q, F8_DOWN_S, D, F)):
        if L.synth_dev_fp8_codes(seed, tq, 0, E, rows, K, bufs[name + "_q"], stream) != 0 or \
                L.synth_dev_fp8_scales(seed, ts, 0, E, rows, K, bufs[name + "_s"], stream) != 0:
            raise RuntimeError("synth_dev_fp8 failed for " + name)


def normal_f32(seed: int, tensor: int, rows: int, cols: int, mean: float = 0.0,
               sigma: float = 1.0) -> np.ndarray:
    out = np.empty((rows, cols), dtype=np.float32)
    _host_lib().synth_normal_f32(seed, tensor, rows, cols, mean, sigma, _ptr(out))
    return out


def normal_bf16(seed: int, tensor: int, rows: int, cols: int, sigma: float = 1.0) -> np.ndarray:
    """bf16 bit patterns (uint16) of N(0, sigma^2) draws."""
    out = np.empty((rows, cols), dtype=np.uint16)
    _host_lib().synth_normal_bf16(seed, tensor, rows, cols, sigma, _ptr(out))
    return out


def zipf_bias(seed: int, E: int, s: float):
    """(perm, bias): bias[e] = -s * ln(perm[e] + 1) for a seeded permutation."""
    perm = np.empty(E, dtype=np.int32)
    bias = np.empty(E, dtype=np.float32)
    _host_lib().synth_zipf_bias(seed, E, s, _ptr(perm), _ptr(bias))
    return perm, bias


def dev_fill_layer(seed: int, E: int, D: int, F: int, bufs: dict, stream: int = 0,
                   lo: int = SCALE_LO, n: int = SCALE_N, dist: int = CODES_UNIFORM) -> None:
    """Fill a whole layer's weights on the GPU.

    ``bufs`` maps gate_q/gate_s/up_q/up_s/down_q/down_s to device pointers of
    sizes E*F*D/2, E*F*D/32, ... (row-major [E][rows][bytes]).
    """
    L = _dev_lib()
    plan = [("gate_q", GATE_Q, F, D), ("up_q", UP_Q, F, D), ("down_q", DOWN_Q, D, F)]
    for name, tid, rows, K in plan:
        if L.synth_dev_mx_codes_dist(seed, tid, 0, E, rows, K, dist, bufs[name], stream) != 0:
            raise RuntimeError("synth_dev_mx_codes failed for " + name)
    plan = [("gate_s", GATE_S, F, D), ("up_s", UP_S, F, D), ("down_s", DOWN_S, D, F)]
    for name, tid, rows, K in plan:
        if L.synth_dev_mx_scales(seed, tid, 0, E, rows, K, lo, n, bufs[name], stream) != 0:
            raise RuntimeError("synth_dev_mx_scales failed for " + name)


# ---------------------------------------------------------------------------
# The five workloads of the routed-expert layer.
# ---------------------------------------------------------------------------

@dataclass
class Workload:
    name: str
    T: int
    D: int
    F: int
    E: int
    k: int
    seed: int = 0
    router: str = "logits"       # "logits" (fp32 input) or "xwr" (in-library x . W_r)
    zipf_s: float = 0.0          # > 0: Zipf popularity bias on the logits
    shared: bool = False         # one bf16 shared expert added to the combine
    codes: int = CODES_UNIFORM   # E2M1 code distribution of the expert weights
    extra: dict = field(default_factory=dict)


WORKLOADS = {
    "tiny": Workload("tiny", T=8, D=256, F=128, E=32, k=4, seed=0),
    "decode1": Workload("decode1", T=1, D=7168, F=1536, E=896, k=16),
    "decode4": Workload("decode4", T=4, D=7168, F=1536, E=896, k=16),
    "decode16": Workload("decode16", T=16, D=7168, F=1536, E=896, k=16),
    "prefill4k": Workload("prefill4k", T=4096, D=7168, F=1536, E=896, k=16),
    "skewed8k": Workload("skewed8k", T=8192, D=7168, F=1536, E=896, k=16, zipf_s=1.1),
    "router16k": Workload("router16k", T=16384, D=7168, F=1536, E=896, k=16, router="xwr",
                          shared=True),
    # MiMo V2.6 Flash lane: 256 experts, top-8 (d_model 4096, d_ff 2048: a
    # reading, the hidden sizes are not stated)
    "mimo_decode": Workload("mimo_decode", T=1, D=4096, F=2048, E=256, k=8),
    "mimo_prefill4k": Workload("mimo_prefill4k", T=4096, D=4096, F=2048, E=256, k=8),
}

# Seeds of the per-call activation / logit draws (weights use Workload.seed).
X_SEED_OFFSET = 1000
LOGIT_SEED_OFFSET = 2000
SHARED_SIGMA = 1.5   # rms of an MXFP4 draw under the codes/scales above
WR_SIGMA = 0.02


def make_x(w: Workload, it: int = 0, T: int | None = None) -> np.ndarray:
    return normal_bf16(w.seed + X_SEED_OFFSET + it, X, T or w.T, w.D)


def make_logits(w: Workload, it: int = 0, T: int | None = None) -> np.ndarray:
    lg = normal_f32(w.seed + LOGIT_SEED_OFFSET + it, LOGITS, T or w.T, w.E)
    if w.zipf_s > 0:
        _, bias = zipf_bias(w.seed, w.E, w.zipf_s)
        lg = (lg + bias[None, :]).astype(np.float32)
    return lg


def make_w_router(w: Workload) -> np.ndarray:
    return normal_f32(w.seed, WR, w.E, w.D, 0.0, WR_SIGMA)


def make_shared(w: Workload):
    return {
        "sh_gate": normal_bf16(w.seed, SH_GATE, w.F, w.D, SHARED_SIGMA),
        "sh_up": normal_bf16(w.seed, SH_UP, w.F, w.D, SHARED_SIGMA),
        "sh_down": normal_bf16(w.seed, SH_DOWN, w.D, w.F, SHARED_SIGMA),
    }
