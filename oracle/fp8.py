"""CPU oracle of an FP8 expert variant (test infrastructure only).

The pages' third lane keeps routed experts in FP8 E4M3FN and qualifies an
exhaustive OCP E4M3FN oracle beside a fused decode GEMV and a bf16-dequant
prefill (Moonshine GitHub README, "GLM 5.3 Flash status"). They give no
scale layout; the reading taken here is E4M3FN weight codes [N][K] with one
fp32 scale per 128 x 128 block ([ceil(N/128)][ceil(K/128)]), dequantised as
value(code) * scale. Only ``tests/`` import this module.

Pinned by ``tests/test_oracle_fp8.py``: all 256 codes against torch's
float8_e4m3fn decoder and the OCP special values, block boundaries of the
scales, and the FFN against the (pinned) MXFP4 oracle on experts whose MXFP4
values are re-encoded exactly as FP8.
"""
from __future__ import annotations

import numpy as np

from . import route

BLOCK = 128


def e4m3fn(code: int) -> float:
    """Value of an OCP E4M3FN byte: sign, 4 exponent bits (bias 7), 3 mantissa
    bits; exponent 0 is subnormal (m * 2^-9); S.1111.111 is NaN; no infinities."""
    s = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 0xF, code & 7
    if e == 0xF and m == 7:
        return float("nan")
    if e == 0:
        return s * m * 2.0 ** -9
    return s * (1 + m / 8) * 2.0 ** (e - 7)


TABLE = np.array([e4m3fn(c) for c in range(256)])


def dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """fp64 matrix [N][K] from E4M3FN codes [N][K] and fp32 block scales
    [ceil(N/128)][ceil(K/128)]."""
    codes = np.asarray(codes, dtype=np.uint8)
    N, K = codes.shape
    sc = np.asarray(scales, dtype=np.float64)
    if sc.shape != ((N + BLOCK - 1) // BLOCK, (K + BLOCK - 1) // BLOCK):
        raise ValueError("scale shape")
    full = np.repeat(np.repeat(sc, BLOCK, axis=0), BLOCK, axis=1)[:N, :K]
    return TABLE[codes] * full


def ffn(x: np.ndarray, logits: np.ndarray, k: int, expert) -> np.ndarray:
    """fp64 routed SwiGLU FFN of tokens x [T, D] (bf16 inputs as fp64) over
    FP8 experts: expert(e) returns its codes and scales as
    (gate_q, gate_s, up_q, up_s, down_q, down_s)."""
    idx, wts = route(logits, k)
    out = np.zeros_like(x)
    for e in sorted(set(int(v) for v in idx.ravel())):
        gq, gs, uq, us, dq, ds = expert(e)
        G, U, Dn = dequant(gq, gs), dequant(uq, us), dequant(dq, ds)
        for t, j in zip(*np.nonzero(idx == e)):
            g = G @ x[t]
            u = U @ x[t]
            out[t] += wts[t, j] * (Dn @ (g / (1.0 + np.exp(-g)) * u))
    return out


def encode_exact(values: np.ndarray) -> np.ndarray:
    """E4M3FN codes of values that are exactly representable (raises if one
    is not): the inverse of the table on its finite entries."""
    flat = np.asarray(values, dtype=np.float64).ravel()
    finite = ~np.isnan(TABLE)
    codes_by_value = {}
    for c in np.nonzero(finite)[0]:
        v = TABLE[c]
        if v == 0 and c & 0x80:
            continue  # encode zero as +0
        codes_by_value.setdefault(v, c)
    try:
        out = np.array([codes_by_value[v] for v in flat.tolist()], dtype=np.uint8)
    except KeyError as err:
        raise ValueError(f"not representable in E4M3FN: {err}") from None
    return out.reshape(np.shape(values))
