"""GPU router (x . W_r in fp32 on tensor cores) and bf16 shared expert vs the oracle.

Routing follows each side's own logits. Where the GPU's top-k differs from
the oracle's, the difference is accepted only at a near-tie: the oracle's
sorted logits at the first differing position are closer than TIE_GAP. Such
tokens are excluded from the float comparison and counted.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from harness import (assert_close, bf16_dev_to_f64, host_layer_weights, router_and_shared,
                     to_dev_bf16)
from oracle.run import reference

pytestmark = pytest.mark.gpu

TIE_GAP = 1e-5
TINY_XWR = synth.Workload("tiny_xwr", T=300, D=256, F=128, E=32, k=4, seed=0, router="xwr",
                          shared=True)


def logit_atol(D: int) -> float:
    """Bound on |GPU logits - exact logits|.

    For the GPU plan to equal the oracle's except at near-ties (gap <
    TIE_GAP), each logit must be within TIE_GAP / 2 of the exact value. fp32
    summation of D exact products stays well inside that for D <= 16384:
    about sqrt(D / 64 + 3 D / 16) rounding steps of a half ulp of a sum of
    size ~0.02 sqrt(D) (under 2e-6 at D = 7168).
    """
    return TIE_GAP / 2


def _layer(w, weights, wr, shared):
    from mxfp4_routed_expert_03_gb300 import MOE_ROUTER_XWR
    from mxfp4_routed_expert_03_gb300.layer import Layer
    return Layer(w.D, w.F, w.E, w.k, weights, MOE_ROUTER_XWR if wr is not None else 0, wr, shared)


def tie_tokens(lg: np.ndarray, ref_idx: np.ndarray, got_idx: np.ndarray, k: int) -> np.ndarray:
    """Tokens whose GPU top-k differs from the oracle's; asserts each is a near-tie."""
    bad = np.nonzero(np.any(ref_idx != got_idx, axis=1))[0]
    for t in bad:
        p = int(np.argmax(ref_idx[t] != got_idx[t]))
        srt = np.sort(lg[t])[::-1]
        gap = srt[p] - srt[p + 1] if p + 1 < len(srt) else np.inf
        assert gap < TIE_GAP, (int(t), p, float(gap))
    return bad


def check_plan_against_own_topk(plan, E: int, k: int):
    """Integer plan properties that hold for any routing (no oracle values)."""
    idx = plan.topk_idx.cpu().numpy().reshape(-1)
    counts = plan.counts.cpu().numpy()
    offsets = plan.offsets.cpu().numpy()
    perm = plan.perm.cpu().numpy()
    inv = plan.inv.cpu().numpy()
    np.testing.assert_array_equal(counts, np.bincount(idx, minlength=E))
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    np.testing.assert_array_equal(perm, np.argsort(idx, kind="stable"))
    np.testing.assert_array_equal(inv[perm], np.arange(len(perm)))


def _route_and_run(w, layer, x_np, T, path):
    from mxfp4_routed_expert_03_gb300 import check
    from mxfp4_routed_expert_03_gb300.layer import Plan
    plan = Plan(T, w.E, w.k)
    x = to_dev_bf16(x_np)
    check(layer.plan(T, None, x, plan), "plan")
    out = torch.empty((T, w.D), dtype=torch.int16, device="cuda")
    fn = layer.forward if path == "forward" else layer.decode
    check(fn(T, x, plan, out), path)
    assert layer.status() == 0
    return bf16_dev_to_f64(out), plan


@pytest.mark.parametrize("T,D,E", [(300, 256, 32), (450, 512, 200), (1, 256, 32), (193, 768, 129)])
def test_router_logits_match_oracle(T, D, E):
    from mxfp4_routed_expert_03_gb300 import check
    w = synth.Workload("r", T=T, D=D, F=128, E=E, k=4, seed=3, router="xwr")
    weights = host_layer_weights(w)
    wr, _ = router_and_shared(w, shared=False)
    layer = _layer(w, weights, wr, None)
    x_np = synth.make_x(w)
    lg = torch.full((T, E), float("nan"), dtype=torch.float32, device="cuda")
    check(layer.router_logits(T, to_dev_bf16(x_np), lg), "router_logits")
    assert layer.status() == 0
    got = lg.cpu().numpy().astype(np.float64)
    ref = oracle.router_logits(x_np, synth.make_w_router(w))
    err = np.abs(got - ref).max()
    print("router T=%d D=%d E=%d max_abs=%.3g bound=%.3g" % (T, D, E, err, logit_atol(D)))
    assert np.all(np.isfinite(got))
    assert err <= logit_atol(D), (err, logit_atol(D))
    layer.close()


def test_router_needs_prepare_and_rejects_logits_mode():
    import mxfp4_routed_expert_03_gb300 as m
    w = synth.Workload("r", T=4, D=256, F=128, E=32, k=4, seed=3, router="xwr")
    weights = host_layer_weights(w)
    wr, _ = router_and_shared(w, shared=False)
    layer = _layer(w, weights, wr, None)
    x = to_dev_bf16(synth.make_x(w))
    lg = torch.empty((4, 32), dtype=torch.float32, device="cuda")
    assert m.moe_router_logits(layer.h, 4, x, lg) == m.MOE_ERR_NOT_PREPARED
    from mxfp4_routed_expert_03_gb300.layer import Plan
    plan = Plan(4, 32, 4)
    ws, n = layer.workspace(4, m.MOE_OP_PLAN)
    assert m.moe_plan(layer.h, 4, None, x, plan.buf, ws, ws.numel()) == m.MOE_ERR_NOT_PREPARED
    layer.prepare()
    assert m.moe_plan(layer.h, 4, lg, x, plan.buf, ws, ws.numel()) == m.MOE_ERR_INVALID_ARG
    assert m.moe_plan(layer.h, 4, None, None, plan.buf, ws, ws.numel()) == m.MOE_ERR_INVALID_ARG
    assert m.moe_router_logits(layer.h, 0, x, lg) == m.MOE_OK
    layer.close()
    plain = _layer(w, weights, None, None)
    assert m.moe_router_logits(plain.h, 4, x, lg) == m.MOE_ERR_INVALID_ARG
    plain.close()


@pytest.fixture(scope="module")
def tiny_xwr():
    w = TINY_XWR
    weights = host_layer_weights(w)
    wr, sh = router_and_shared(w)
    return weights, wr, sh


@pytest.mark.parametrize("T", [1, 5, 300])
@pytest.mark.parametrize("path", ["forward", "decode"])
def test_tiny_router_and_shared_expert_layer(tiny_xwr, T, path):
    w = TINY_XWR
    weights, wr, sh = tiny_xwr
    layer = _layer(w, weights, wr, sh)
    x_np = synth.make_x(w, 7, T=T)
    got, plan = _route_and_run(w, layer, x_np, T, path)
    layer.close()
    ref = reference(w, x_np, None)
    ties = tie_tokens(ref["logits"], ref["idx"], plan.topk_idx.cpu().numpy(), w.k)
    assert len(ties) == 0
    p = ref["plan"]
    for name in ("counts", "offsets", "perm", "inv"):
        np.testing.assert_array_equal(getattr(plan, name).cpu().numpy(), p[name])
    np.testing.assert_allclose(plan.topk_w.cpu().numpy(), ref["w"], atol=1e-5)
    e = assert_close(got, ref["out"])
    print("tiny xwr+shared T=%d %s" % (T, path), e)


def test_shared_expert_alone_matches_oracle(tiny_xwr):
    """Routed weights all zero codes: the output is the shared expert alone."""
    w = TINY_XWR
    weights, wr, sh = tiny_xwr
    zero = {k: (torch.zeros_like(v) if k.endswith("_q") else v) for k, v in weights.items()}
    layer = _layer(w, zero, wr, sh)
    T = 200
    x_np = synth.make_x(w, 9, T=T)
    got, _ = _route_and_run(w, layer, x_np, T, "forward")
    layer.close()
    ref = np.zeros((T, w.D))
    s = synth.make_shared(w)
    oracle.shared_ffn(x_np, s["sh_gate"], s["sh_up"], s["sh_down"], ref)
    e = assert_close(got, ref)
    print("shared alone", e)


def test_k3_router16k_full_size(k3_layer):
    """The fused-router workload at full size: T=16384, all 896 experts, shared expert."""
    from mxfp4_routed_expert_03_gb300 import check
    w = synth.WORKLOADS["router16k"]
    wr, sh = router_and_shared(w)
    layer = _layer(w, k3_layer, wr, sh)
    x_np = synth.make_x(w)
    T = w.T
    # the router alone, on sampled tokens
    lg = torch.empty((T, w.E), dtype=torch.float32, device="cuda")
    check(layer.router_logits(T, to_dev_bf16(x_np), lg), "router_logits")
    rng = np.random.default_rng(16)
    samp = np.sort(rng.choice(T, 64, replace=False))
    ref_lg = oracle.router_logits(x_np[samp], synth.make_w_router(w))
    err = np.abs(lg.cpu().numpy()[samp].astype(np.float64) - ref_lg).max()
    print("router16k logits max_abs=%.3g bound=%.3g" % (err, logit_atol(w.D)))
    assert err <= logit_atol(w.D)
    del lg
    # the whole layer
    got, plan = _route_and_run(w, layer, x_np, T, "forward")
    layer.close()
    full = oracle.router_logits(x_np, synth.make_w_router(w))
    ref_idx, ref_w = oracle.route(full, w.k)
    ties = tie_tokens(full, ref_idx, plan.topk_idx.cpu().numpy(), w.k)
    print("router16k near-tie tokens:", len(ties))
    check_plan_against_own_topk(plan, w.E, w.k)
    if len(ties) == 0:
        p = oracle.plan(ref_idx, w.E)
        for name in ("counts", "offsets", "perm", "inv"):
            np.testing.assert_array_equal(getattr(plan, name).cpu().numpy(), p[name])
    ok = np.setdiff1d(np.arange(T), ties)
    np.testing.assert_allclose(plan.topk_w.cpu().numpy()[ok], ref_w[ok], atol=1e-5)
    tok = np.sort(rng.choice(ok, 12, replace=False))
    ref = reference(w, x_np, None, tokens=tok)
    e = assert_close(got[tok], ref["out"])
    print("router16k forward", e)


@pytest.mark.parametrize("T", [1, 4])
def test_k3_router_shared_decode_and_forward_agree(k3_layer, T):
    w = synth.WORKLOADS["router16k"]
    wr, sh = router_and_shared(w)
    layer = _layer(w, k3_layer, wr, sh)
    x_np = synth.make_x(w, 40 + T, T=T)
    got_f, plan_f = _route_and_run(w, layer, x_np, T, "forward")
    got_d, plan_d = _route_and_run(w, layer, x_np, T, "decode")
    layer.close()
    np.testing.assert_array_equal(plan_f.perm.cpu().numpy(), plan_d.perm.cpu().numpy())
    ref = reference(w, x_np, None)
    assert len(tie_tokens(ref["logits"], ref["idx"], plan_f.topk_idx.cpu().numpy(), w.k)) == 0
    ef, ed = assert_close(got_f, ref["out"]), assert_close(got_d, ref["out"])
    print("router+shared T=%d forward" % T, ef, "decode", ed)
