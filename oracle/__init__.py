"""CPU oracle of the routed-expert FFN (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. It loads ``liboracle.so`` built from
``moe_oracle.c`` (plain C, fp64, OpenMP across rows) and shares no code with
the CUDA library. See ``moe_oracle.c`` for what each function computes and the
passage it follows. ``oracle.store`` (``store_oracle.c``) is the oracle of the
compressed expert store.

Every function here is pinned by ``tests/test_oracle_*.py``; none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_SRC = os.path.join(_HERE, "moe_oracle.c")
_lib = None


def build(force: bool = False) -> None:
    """Compile liboracle.so and libstore_oracle.so with gcc (building the
    checker is not using it)."""
    from . import store
    store.build(force)
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                           "-o", _SO, _SRC, "-lm"])


def _L():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        i32, i64, p, d = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_double
        L.oracle_e2m1.argtypes = [i32]
        L.oracle_e2m1.restype = d
        L.oracle_e8m0.argtypes = [i32]
        L.oracle_e8m0.restype = d
        L.oracle_dequant.argtypes = [p, p, i64, i64, p]
        L.oracle_dequant.restype = i32
        L.oracle_route.argtypes = [i32, i32, i32, p, p, p]
        L.oracle_route.restype = i32
        L.oracle_plan.argtypes = [i32, i32, i32, p, p, p, p, p, p]
        L.oracle_plan.restype = i32
        L.oracle_router_logits.argtypes = [i32, i32, i32, p, p, p]
        L.oracle_ffn.argtypes = [i32, i32, i32, i32, p, p, p, i32, p, p, p, p, p, p, p, p]
        L.oracle_ffn.restype = i32
        L.oracle_shared_ffn.argtypes = [i32, i32, i32, p, p, p, p, p]
        _lib = L
    return _lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def e2m1(code: int) -> float:
    return _L().oracle_e2m1(int(code))


def e8m0(b: int) -> float:
    return _L().oracle_e8m0(int(b))


def dequant(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Decoded fp64 matrix [rows, K] from codes [rows, K/2] and scales [rows, K/32]."""
    q = _c(q, np.uint8)
    s = _c(s, np.uint8)
    rows, K = q.shape[0], q.shape[1] * 2
    out = np.empty((rows, K), dtype=np.float64)
    if _L().oracle_dequant(q.ctypes.data, s.ctypes.data, rows, K, out.ctypes.data) != 0:
        raise ValueError("K must be a multiple of 32")
    return out


def route(logits: np.ndarray, k: int):
    """(idx int32 [T,k], w float64 [T,k]) from logits [T,E]."""
    lg = _c(logits, np.float64)
    T, E = lg.shape
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    rc = _L().oracle_route(T, E, k, lg.ctypes.data, idx.ctypes.data, w.ctypes.data)
    if rc == -2:
        raise ValueError("NaN logit")
    if rc != 0:
        raise ValueError("bad k")
    return idx, w


def plan(idx: np.ndarray, E: int) -> dict:
    idx = _c(idx, np.int32)
    T, k = idx.shape
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    perm = np.empty(T * k, dtype=np.int32)
    inv = np.empty(T * k, dtype=np.int32)
    active = np.empty(E + 1, dtype=np.int32)
    rc = _L().oracle_plan(T, E, k, idx.ctypes.data, counts.ctypes.data, offsets.ctypes.data,
                          perm.ctypes.data, inv.ctypes.data, active.ctypes.data)
    if rc != 0:
        raise ValueError("expert index out of range")
    return {"counts": counts, "offsets": offsets, "perm": perm, "inv": inv,
            "active": active[: 1 + active[0]]}


def router_logits(x_bf16: np.ndarray, w_router: np.ndarray) -> np.ndarray:
    x = _c(x_bf16, np.uint16)
    wr = _c(w_router, np.float32)
    T, D = x.shape
    E = wr.shape[0]
    out = np.empty((T, E), dtype=np.float64)
    _L().oracle_router_logits(T, D, E, x.ctypes.data, wr.ctypes.data, out.ctypes.data)
    return out


def ffn(x_bf16: np.ndarray, idx: np.ndarray, w: np.ndarray, store: dict) -> np.ndarray:
    """fp64 combined expert output [n, D] for n tokens.

    ``store`` holds ``experts`` (int32 [S]) and per-slot byte arrays
    gate_q/up_q [S,F,D/2], gate_s/up_s [S,F,D/32], down_q [S,D,F/2], down_s [S,D,F/32].
    """
    x = _c(x_bf16, np.uint16)
    idx = _c(idx, np.int32)
    w = _c(w, np.float64)
    n, D = x.shape
    k = idx.shape[1]
    ex = _c(store["experts"], np.int32)
    S = ex.shape[0]
    F = store["gate_q"].shape[1]
    arrs = [_c(store[nm], np.uint8) for nm in ("gate_q", "gate_s", "up_q", "up_s",
                                               "down_q", "down_s")]
    out = np.empty((n, D), dtype=np.float64)
    rc = _L().oracle_ffn(n, D, F, k, x.ctypes.data, idx.ctypes.data, w.ctypes.data, S,
                         ex.ctypes.data, *[a.ctypes.data for a in arrs], out.ctypes.data)
    if rc == -3:
        raise KeyError("selected expert missing from the store")
    if rc != 0:
        raise ValueError("D and F must be multiples of 32")
    return out


def shared_ffn(x_bf16: np.ndarray, sg: np.ndarray, su: np.ndarray, sd: np.ndarray,
               out: np.ndarray) -> None:
    """out += shared-expert SwiGLU FFN of x (bf16 weights), in place (fp64)."""
    x = _c(x_bf16, np.uint16)
    n, D = x.shape
    F = sg.shape[0]
    assert out.dtype == np.float64 and out.flags["C_CONTIGUOUS"] and out.shape == (n, D)
    _L().oracle_shared_ffn(n, D, F, x.ctypes.data, _c(sg, np.uint16).ctypes.data,
                           _c(su, np.uint16).ctypes.data, _c(sd, np.uint16).ctypes.data,
                           out.ctypes.data)
