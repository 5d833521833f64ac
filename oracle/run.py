"""Oracle over a workload: regenerate the needed experts and run the checker.

Test infrastructure only (tests, smoke check, CPU-baseline leg of the
benchmark). The expert weights come from the seeded generator in ``synth``;
nothing here reads anything the GPU produced.
"""
from __future__ import annotations

import numpy as np

import synth
from . import ffn, plan, route, router_logits, shared_ffn


def store_for(w: synth.Workload, experts) -> dict:
    """Compacted weights of the given experts, regenerated on the host."""
    experts = np.asarray(sorted(set(int(e) for e in experts)), dtype=np.int32)
    S, D, F = len(experts), w.D, w.F
    st = {"experts": experts,
          "gate_q": np.empty((S, F, D // 2), np.uint8), "gate_s": np.empty((S, F, D // 32), np.uint8),
          "up_q": np.empty((S, F, D // 2), np.uint8), "up_s": np.empty((S, F, D // 32), np.uint8),
          "down_q": np.empty((S, D, F // 2), np.uint8), "down_s": np.empty((S, D, F // 32), np.uint8)}
    for i, e in enumerate(experts):
        ew = synth.expert_weights(w.seed, int(e), D, F, dist=w.codes)
        for nm, a in ew.items():
            st[nm][i] = a
    return st


def logits_for(w: synth.Workload, x: np.ndarray, logits: np.ndarray | None) -> np.ndarray:
    """fp64 logits the oracle routes on (given, or x . W_r for the router workload)."""
    if w.router == "xwr":
        return router_logits(x, synth.make_w_router(w))
    return np.asarray(logits, dtype=np.float64)


def reference(w: synth.Workload, x: np.ndarray, logits: np.ndarray | None,
              tokens=None, route_override=None) -> dict:
    """Full integer plan for all T tokens, fp64 outputs for ``tokens`` (default: all).

    ``route_override`` = (idx, w) replaces the oracle's own routing for the FFN
    (used where the two sides may legitimately route a near-tie differently).
    """
    lg = logits_for(w, x, logits)
    idx, wts = route(lg, w.k)
    p = plan(idx, w.E)
    T = x.shape[0]
    tok = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    fidx, fw = (idx, wts) if route_override is None else route_override
    sel_idx, sel_w = fidx[tok], fw[tok]
    store = store_for(w, np.unique(sel_idx))
    out = ffn(x[tok], sel_idx, sel_w, store)
    if w.shared:
        sh = synth.make_shared(w)
        shared_ffn(x[tok], sh["sh_gate"], sh["sh_up"], sh["sh_down"], out)
    return {"logits": lg, "idx": idx, "w": wts, "plan": p, "tokens": tok, "out": out}
