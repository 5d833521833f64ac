"""Independent numpy (float64) brute-force evaluator used to pin the C oracle.

Written separately from ``oracle/moe_oracle.c``: it decodes E2M1 through the
OCP value table in ``golden/ocp_e2m1_values.txt`` and E8M0 through torch's
float8_e8m0fnu decoder, evaluates every expert densely with numpy matmuls, and
masks the non-selected ones, so a slip in the oracle's decode, indexing or
combine shows up as a mismatch here.
"""
from __future__ import annotations

import os

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))


def ocp_e2m1_table() -> np.ndarray:
    vals = np.zeros(16, dtype=np.float64)
    with open(os.path.join(HERE, "golden", "ocp_e2m1_values.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            c, v = line.split()
            vals[int(c)] = float(v)
    return vals


def e8m0_torch(b: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(b, dtype=np.uint8)).view(torch.float8_e8m0fnu)
    return t.to(torch.float64).numpy()


def decode(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """[rows, K] float64 from packed codes [rows, K/2] and scales [rows, K/32]."""
    tab = ocp_e2m1_table()
    lo = q & 0x0F
    hi = q >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(q.shape[0], q.shape[1] * 2)
    scale = np.repeat(e8m0_torch(s), 32, axis=1)
    return tab[codes] * scale


def bf16_to_f64(x: np.ndarray) -> np.ndarray:
    return (np.asarray(x, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def silu(z):
    return z / (1.0 + np.exp(-z))


def expert_ffn_dense(xf: np.ndarray, Wg, Wu, Wd) -> np.ndarray:
    """SwiGLU FFN of every token through one expert: [n, D]."""
    return (silu(xf @ Wg.T) * (xf @ Wu.T)) @ Wd.T


def topk_stable(logits: np.ndarray, k: int):
    order = np.argsort(-logits, axis=1, kind="stable")
    return order[:, :k].astype(np.int32)


def moe_dense(x_bf16, logits, k, weights_by_expert) -> np.ndarray:
    """All experts computed for all tokens; non-selected ones masked to weight 0.

    ``weights_by_expert[e]`` = (Wg, Wu, Wd) decoded float64 matrices.
    """
    xf = bf16_to_f64(x_bf16)
    lg = np.asarray(logits, dtype=np.float64)
    T, E = lg.shape
    sel = topk_stable(lg, k)
    mask = np.zeros((T, E), dtype=bool)
    np.put_along_axis(mask, sel, True, axis=1)
    z = np.where(mask, np.exp(lg - lg.max(axis=1, keepdims=True)), 0.0)
    gate_w = z / z.sum(axis=1, keepdims=True)
    out = np.zeros((T, xf.shape[1]), dtype=np.float64)
    for e in range(E):
        Wg, Wu, Wd = weights_by_expert[e]
        out += gate_w[:, e:e + 1] * expert_ffn_dense(xf, Wg, Wu, Wd)
    return out
