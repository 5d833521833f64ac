"""The FP8 expert lane (weight_format MOE_W_FP8) against the FP8 oracle.

Experts are E4M3FN codes with an fp32 scale per 128 x 128 block
(oracle/fp8.py, pinned by tests/test_oracle_fp8.py). moe_decode and
moe_decode_noalloc stream the codes on CUDA cores with exact products (the
decode path's tighter bound applies); moe_forward runs bf16 tensor-core GEMMs
on the bf16 copy moe_prepare makes (each weight rounded once to bf16, h in
bf16), within the layer's normwise tolerance. Integer routing is the same
plan for every path.
"""
import numpy as np
import pytest
import torch

import oracle.fp8 as F8
import synth
from harness import MAE_REL, MAX_REL, assert_close, bf16_dev_to_f64, to_dev_bf16

pytestmark = pytest.mark.gpu

DECODE_MAX_REL = 6e-3
DECODE_MAE_REL = 6e-4
TINY = synth.WORKLOADS["tiny"]
K3 = synth.WORKLOADS["decode4"]


def _host_fp8_layer(w):
    from mxfp4_routed_expert_03_gb300.layer import alloc_fp8_weights
    wts = alloc_fp8_weights(w.E, w.D, w.F)
    for e in range(w.E):
        for name, arr in synth.fp8_expert_weights(w.seed, e, w.D, w.F).items():
            wts[name][e].copy_(torch.from_numpy(arr))
    return wts


def _device_fp8_layer(w):
    from mxfp4_routed_expert_03_gb300.layer import alloc_fp8_weights
    wts = alloc_fp8_weights(w.E, w.D, w.F)
    synth.dev_fill_fp8_layer(w.seed, w.E, w.D, w.F, {k: v.data_ptr() for k, v in wts.items()},
                             torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return wts


def _oracle(w, x_np, lg_np, tokens):
    """fp64 FP8 layer of `tokens` (the experts regenerated on the host)."""
    x = (x_np[tokens].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    cache = {}

    def expert(e):
        if e not in cache:
            ew = synth.fp8_expert_weights(w.seed, e, w.D, w.F)
            cache[e] = tuple(ew[n] for n in ("gate_q", "gate_s", "up_q", "up_s", "down_q",
                                             "down_s"))
        return cache[e]
    return F8.ffn(x, np.asarray(lg_np[tokens], np.float64), w.k, expert)


def _run(w, weights, x_np, lg_np, paths):
    from mxfp4_routed_expert_03_gb300 import MOE_W_FP8, check, moe_decode_noalloc
    from mxfp4_routed_expert_03_gb300.layer import Layer, Plan
    T = x_np.shape[0]
    layer = Layer(w.D, w.F, w.E, w.k, weights, weight_format=MOE_W_FP8)
    plan = Plan(T, w.E, w.k)
    x = to_dev_bf16(x_np)
    check(layer.plan(T, torch.from_numpy(lg_np).cuda(), None, plan), "plan")
    outs = {}
    for p in paths:
        out = torch.empty((T, w.D), dtype=torch.int16, device="cuda")
        if p == "decode":
            check(layer.decode(T, x, plan, out), p)
        elif p == "noalloc":
            check(moe_decode_noalloc(layer.h, T, x, plan.buf, out), p)
        else:
            check(layer.forward(T, x, plan, out), p)
        outs[p] = bf16_dev_to_f64(out)
    st = layer.status()
    layer.close()
    assert st == 0, st
    return outs


def _check(outs, ref):
    res = {}
    for p, got in outs.items():
        tol = (MAX_REL, MAE_REL) if p == "forward" else (DECODE_MAX_REL, DECODE_MAE_REL)
        res[p] = assert_close(got, ref, *tol)
    return res


@pytest.fixture(scope="module")
def tiny_fp8():
    return _host_fp8_layer(TINY)


def test_device_generator_matches_host():
    from mxfp4_routed_expert_03_gb300.layer import alloc_fp8_weights
    w = K3
    E = 2
    wts = alloc_fp8_weights(E, w.D, w.F)
    synth.dev_fill_fp8_layer(w.seed, E, w.D, w.F, {k: v.data_ptr() for k, v in wts.items()})
    torch.cuda.synchronize()
    for e in range(E):
        for name, arr in synth.fp8_expert_weights(w.seed, e, w.D, w.F).items():
            np.testing.assert_array_equal(wts[name][e].cpu().numpy(), arr, err_msg=name)


@pytest.mark.parametrize("T", [1, 8, 16, 37, 300])
def test_tiny_fp8_layer(tiny_fp8, T):
    """Decode and forward (narrow tiles up to 16 tokens, wide above)."""
    w = TINY
    x, lg = synth.make_x(w, 100 + T, T=T), synth.make_logits(w, 100 + T, T=T)
    paths = ("decode", "noalloc", "forward") if T <= 64 else ("decode", "forward")
    outs = _run(w, tiny_fp8, x, lg, paths)
    tok = np.arange(T) if T <= 37 else np.random.default_rng(T).choice(T, 40, replace=False)
    res = _check({p: o[tok] for p, o in outs.items()}, _oracle(w, x, lg, tok))
    print("tiny fp8 T=%d" % T, res)


@pytest.fixture(scope="module")
def k3_fp8():
    wts = _device_fp8_layer(K3)
    yield wts
    del wts
    torch.cuda.empty_cache()


@pytest.mark.parametrize("T", [1, 4, 16])
def test_k3_fp8_decode_and_forward(k3_fp8, T):
    w = K3
    x, lg = synth.make_x(w, 110 + T, T=T), synth.make_logits(w, 110 + T, T=T)
    outs = _run(w, k3_fp8, x, lg, ("decode", "forward"))
    tok = np.arange(T) if T <= 4 else np.array([0, 7, T - 1])
    res = _check({p: o[tok] for p, o in outs.items()}, _oracle(w, x, lg, tok))
    print("k3 fp8 T=%d" % T, res)


def test_k3_fp8_prefill_sampled_tokens(k3_fp8):
    """A wide-tile batch over most experts."""
    w = K3
    T = 512
    x, lg = synth.make_x(w, 120, T=T), synth.make_logits(w, 120, T=T)
    outs = _run(w, k3_fp8, x, lg, ("forward",))
    tok = np.array([0, 100, 311, T - 1])
    res = _check({p: o[tok] for p, o in outs.items()}, _oracle(w, x, lg, tok))
    print("k3 fp8 prefill T=%d" % T, res)
