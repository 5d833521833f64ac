"""Activations across bf16's range, for every entry point that takes x.

bf16 reaches from about 1e-38 to 3e38. The decode path converts x to f16
with a power-of-two exponent per 32-element block and the forward path
splits it into two E4M3 terms with an E8M0 scale per block; both must give
the oracle's answer (token by token, normwise per token) when x is scaled far
away from N(0, 1): uniformly tiny, uniformly large, a different power of two
per token, and a different power of two per 32-element block within a row.
Scaling by a power of two is exact in bf16, and the oracle's exact linearity
in x is pinned separately (tests/test_oracle_ffn.py).

The largest scale keeps the layer's output inside fp32's range: g and u grow
like the scale, h like its square, so for N(0,1) rows scaled by 2^s the
output is about 2^(2s + 18) at these shapes; s <= 40 keeps it below 2^100.
"""
import numpy as np
import pytest
import torch

import synth
from harness import MAE_REL, MAX_REL, assert_close, bf16_dev_to_f64, host_layer_weights, to_dev_bf16
from oracle.run import reference

pytestmark = pytest.mark.gpu

# the decode path's products are exact; the same bound its other tests use
DECODE_MAX_REL = 6e-3
DECODE_MAE_REL = 6e-4


def scale_bf16(x: np.ndarray, exps: np.ndarray) -> np.ndarray:
    """x (bf16 bits [T][D]) times 2^exps, exps broadcast per element; exact."""
    f = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    y = (f * np.exp2(exps)).astype(np.float32)
    bits = y.view(np.uint32)
    assert np.all(bits & 0xFFFF == 0), "power-of-two scaling left bf16"
    return (bits >> 16).astype(np.uint16)


def scaled_inputs(w, case: str, T: int, seed: int):
    x = synth.make_x(w, seed, T=T)
    lg = synth.make_logits(w, seed, T=T)
    rng = np.random.default_rng(seed)
    nb = w.D // 32
    if case == "tiny":
        e = np.full((T, 1), -24.0)
    elif case == "large":
        e = np.full((T, 1), 20.0)
    elif case == "per_token":
        e = np.linspace(-60, 40, T).round()[:, None]
    elif case == "per_block":
        e = np.repeat(rng.integers(-40, 31, size=(T, nb)).astype(np.float64), 32, axis=1)
    else:
        raise ValueError(case)
    return scale_bf16(x, e), lg


def run_all_paths(w, weights, x_np, lg_np):
    """moe_decode, moe_decode_noalloc and moe_forward on the same plan."""
    from mxfp4_routed_expert_03_gb300 import check, moe_decode_noalloc
    from mxfp4_routed_expert_03_gb300.layer import Layer, Plan
    T = x_np.shape[0]
    layer = Layer(w.D, w.F, w.E, w.k, weights)
    layer.prepare()
    plan = Plan(T, w.E, w.k)
    x = to_dev_bf16(x_np)
    check(layer.plan(T, torch.from_numpy(lg_np).cuda(), None, plan), "plan")
    outs = {}
    for name in ("decode", "noalloc", "forward"):
        out = torch.empty((T, w.D), dtype=torch.int16, device="cuda")
        if name == "decode":
            check(layer.decode(T, x, plan, out), name)
        elif name == "noalloc":
            check(moe_decode_noalloc(layer.h, T, x, plan.buf, out), name)
        else:
            check(layer.forward(T, x, plan, out), name)
        outs[name] = bf16_dev_to_f64(out)
    st = layer.status()
    layer.close()
    assert st == 0, st
    return outs


def check_per_token(outs, ref):
    worst = {}
    for name, got in outs.items():
        tol = (MAX_REL, MAE_REL) if name == "forward" else (DECODE_MAX_REL, DECODE_MAE_REL)
        for t in range(ref.shape[0]):
            assert np.abs(ref[t]).max() > 0
            e = assert_close(got[t], ref[t], *tol)
            worst[name] = max(worst.get(name, 0.0), e["max_rel"])
    return worst


@pytest.fixture(scope="module")
def tiny_weights():
    return host_layer_weights(synth.WORKLOADS["tiny"])


@pytest.mark.parametrize("case", ["tiny", "large", "per_token", "per_block"])
def test_tiny_layer_input_magnitudes(tiny_weights, case):
    w = synth.WORKLOADS["tiny"]
    x, lg = scaled_inputs(w, case, 12, 31)
    outs = run_all_paths(w, tiny_weights, x, lg)
    ref = reference(w, x, lg)["out"]
    print(case, check_per_token(outs, ref))


@pytest.mark.parametrize("case", ["per_token", "per_block"])
def test_k3_layer_input_magnitudes(k3_layer, case):
    w = synth.WORKLOADS["decode4"]
    x, lg = scaled_inputs(w, case, 4, 32)
    outs = run_all_paths(w, k3_layer, x, lg)
    ref = reference(w, x, lg)["out"]
    print("k3", case, check_per_token(outs, ref))
