"""Activation-precision study on the CPU (test infrastructure only).

How far the layer's output moves when the tensor cores see the activations
(x into gate/up, h into down) in a narrower format than bf16, all else in
fp64. It is the evidence behind the GEMMs' two-term E4M3 activations and the
measured error of an FP4 x FP4 mode (MXFP4 activations): the formats are the
OCP Microscaling (MX) v1.0 ones, an element format with one shared E8M0 scale
per 32 consecutive values, the scale 2^(floor(log2(amax)) - emax_elem)
(OCP MX v1.0, section 6.3: the conversion from a vector of higher-precision
values), elements rounded to nearest, ties to even, clamped to the largest
finite magnitude. Only ``tests/`` import this module.

Pinned by ``tests/test_oracle_act_study.py`` (exact values stay exact,
midpoint ties, saturation, the scale rule, and the bf16 case reducing to the
oracle's own FFN).
"""
from __future__ import annotations

import numpy as np

from . import dequant, e2m1, route


def _magnitudes(fmt: str) -> np.ndarray:
    """Finite non-negative magnitudes of an element format, in code order."""
    if fmt == "e2m1":
        return np.array([e2m1(c) for c in range(8)])
    if fmt == "e4m3":  # OCP E4M3 (FN): bias 7, no infinities, S.1111.111 is NaN
        vals = []
        for c in range(127):  # 0x00 .. 0x7E
            e, m = c >> 3, c & 7
            vals.append(m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
        return np.array(vals)
    raise ValueError(fmt)


_EMAX = {"e2m1": 2, "e4m3": 8}


def round_to_format(v: np.ndarray, fmt: str) -> np.ndarray:
    """Round to the nearest finite value of the format (ties to the even code),
    magnitudes above the largest clamped to it."""
    mags = _magnitudes(fmt)
    a = np.minimum(np.abs(v), mags[-1])
    hi = np.searchsorted(mags, a, side="left")          # first magnitude >= a
    hi = np.minimum(hi, len(mags) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = a - mags[lo], mags[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    q = np.where(pick_hi, mags[hi], mags[lo])
    q = np.where(a == mags[hi], mags[hi], q)
    return np.copysign(q, v)


def mx_quantise(v: np.ndarray, fmt: str) -> np.ndarray:
    """Decoded value of v (last axis a multiple of 32) in MX format `fmt`:
    per block of 32, X = 2^(floor(log2(amax)) - emax_elem), elements
    round_to_format(v / X). All-zero blocks stay zero."""
    shp = v.shape
    b = v.reshape(-1, 32)
    amax = np.max(np.abs(b), axis=1, keepdims=True)
    with np.errstate(divide="ignore"):
        k = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))), 0.0)
    X = 2.0 ** (k - _EMAX[fmt])
    q = round_to_format(b / X, fmt) * X
    return np.where(amax > 0, q, 0.0).reshape(shp)


def two_term(v: np.ndarray, fmt: str = "e4m3") -> np.ndarray:
    """hi + lo: hi = MX(v), lo = MX(v - hi), each with its own block scales."""
    hi = mx_quantise(v, fmt)
    return hi + mx_quantise(v - hi, fmt)


def _bf16(v: np.ndarray) -> np.ndarray:
    """Round fp64 to bf16 (through fp32, nearest even)."""
    f = v.astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


TREATMENTS = {
    "exact": lambda v: v,
    "bf16_h": _bf16,
    "two_term_e4m3": lambda v: two_term(v, "e4m3"),
    "one_term_e4m3": lambda v: mx_quantise(v, "e4m3"),
    "mxfp4": lambda v: mx_quantise(v, "e2m1"),
}


def ffn(x: np.ndarray, logits: np.ndarray, k: int, expert, treats) -> dict:
    """fp64 routed FFN of tokens x [T, D] (the bf16 inputs as fp64) under each
    activation treatment in `treats`: the activations into gate/up (x) and
    into down (h) pass through it ("bf16_h" rounds only h; x is bf16 already).
    expert(e) returns expert e's decoded fp64 matrices gate [F, D], up [F, D],
    down [D, F]; experts are visited one at a time. Returns treat -> [T, D]."""
    idx, wts = route(logits, k)
    out = {tr: np.zeros_like(x) for tr in treats}
    for e in sorted(set(int(v) for v in idx.ravel())):
        m = expert(e)
        for t, j in zip(*np.nonzero(idx == e)):
            for tr in treats:
                q = TREATMENTS[tr]
                xa = x[t] if tr == "bf16_h" else q(x[t])
                g = m["gate"] @ xa
                u = m["up"] @ xa
                h = g / (1.0 + np.exp(-g)) * u
                out[tr][t] += wts[t, j] * (m["down"] @ q(h))
    return out


def decoded(ew: dict) -> dict:
    """Decoded fp64 matrices of one expert from its byte arrays (synth layout)."""
    return {"gate": dequant(ew["gate_q"], ew["gate_s"]),
            "up": dequant(ew["up_q"], ew["up_s"]),
            "down": dequant(ew["down_q"], ew["down_s"])}


def errors(y: np.ndarray, ref: np.ndarray) -> dict:
    """Normwise errors against the reference's largest magnitude."""
    s = float(np.max(np.abs(ref)))
    d = np.abs(y - ref)
    return {"max_rel": float(d.max() / s), "mae_rel": float(d.mean() / s)}
