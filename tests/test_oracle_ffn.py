"""Pins of the oracle's expert FFN and weighted combine."""
import numpy as np
from scipy.special import softmax

import oracle
import synth
from bruteforce import bf16_to_f64, decode, expert_ffn_dense, moe_dense, silu
from oracle.run import reference, store_for


def _decoded_layer(w):
    out = {}
    for e in range(w.E):
        ew = synth.expert_weights(w.seed, e, w.D, w.F)
        out[e] = (decode(ew["gate_q"], ew["gate_s"]), decode(ew["up_q"], ew["up_s"]),
                  decode(ew["down_q"], ew["down_s"]))
    return out


def _rel(a, b):
    return np.max(np.abs(a - b)) / np.max(np.abs(b))


def test_tiny_layer_matches_bruteforce_dense():
    w = synth.WORKLOADS["tiny"]
    x, lg = synth.make_x(w), synth.make_logits(w)
    ref = reference(w, x, lg)
    dense = moe_dense(x, lg, w.k, _decoded_layer(w))
    assert _rel(ref["out"], dense) < 1e-12


def test_tiny_layer_other_draws_and_k():
    base = synth.WORKLOADS["tiny"]
    for it, k in ((1, 1), (2, 7), (3, 32)):
        w = synth.Workload("t", T=5, D=base.D, F=base.F, E=base.E, k=k, seed=4)
        x, lg = synth.make_x(w, it), synth.make_logits(w, it)
        ref = reference(w, x, lg)
        assert _rel(ref["out"], moe_dense(x, lg, k, _decoded_layer(w))) < 1e-12


def test_single_expert_is_textbook_swiglu():
    w = synth.Workload("e1", T=3, D=64, F=96, E=1, k=1, seed=11)
    x = synth.make_x(w)
    ew = synth.expert_weights(w.seed, 0, w.D, w.F)
    idx = np.zeros((3, 1), np.int32)
    got = oracle.ffn(x, idx, np.ones((3, 1)), store_for(w, [0]))
    Wg, Wu, Wd = (decode(ew["gate_q"], ew["gate_s"]), decode(ew["up_q"], ew["up_s"]),
                  decode(ew["down_q"], ew["down_s"]))
    xf = bf16_to_f64(x)
    expect = np.stack([Wd @ (silu(Wg @ xf[t]) * (Wu @ xf[t])) for t in range(3)])
    assert _rel(got, expect) < 1e-13


def test_k_equals_e_is_full_softmax_mixture():
    w = synth.Workload("kE", T=2, D=64, F=32, E=6, k=6, seed=2)
    x, lg = synth.make_x(w), synth.make_logits(w)
    ref = reference(w, x, lg)
    p = softmax(lg.astype(np.float64), axis=1)
    layer = _decoded_layer(w)
    xf = bf16_to_f64(x)
    expect = sum(p[:, e:e + 1] * expert_ffn_dense(xf, *layer[e]) for e in range(w.E))
    assert _rel(ref["out"], expect) < 1e-13


def test_all_ones_expert_closed_form():
    # Every code 2 (= 1.0) at scale 127: W = ones, so g = u = sum(x) and
    # y_d = F * silu(S) * S for S = sum_d x_d.
    D, F = 64, 32
    st = {"experts": np.array([0], np.int32),
          "gate_q": np.full((1, F, D // 2), 0x22, np.uint8), "gate_s": np.full((1, F, D // 32), 127, np.uint8),
          "up_q": np.full((1, F, D // 2), 0x22, np.uint8), "up_s": np.full((1, F, D // 32), 127, np.uint8),
          "down_q": np.full((1, D, F // 2), 0x22, np.uint8), "down_s": np.full((1, D, F // 32), 127, np.uint8)}
    x = synth.normal_bf16(1, synth.X, 2, D)
    got = oracle.ffn(x, np.zeros((2, 1), np.int32), np.ones((2, 1)), st)
    S = bf16_to_f64(x).sum(axis=1)
    expect = (F * S / (1 + np.exp(-S)) * S)[:, None] * np.ones((1, D))
    np.testing.assert_allclose(got, expect, rtol=1e-13)


def test_power_of_two_scale_steps_scale_output_exactly():
    w = synth.Workload("p2", T=2, D=64, F=64, E=2, k=2, seed=3)
    x, lg = synth.make_x(w), synth.make_logits(w)
    idx, wt = oracle.route(lg, w.k)
    st = store_for(w, [0, 1])
    base = oracle.ffn(x, idx, wt, st)
    for name in ("down_s", "up_s"):
        st2 = {kk: v.copy() for kk, v in st.items()}
        st2[name] = st2[name] + 1
        np.testing.assert_array_equal(oracle.ffn(x, idx, wt, st2), 2.0 * base)


def test_missing_expert_raises():
    w = synth.Workload("m", T=1, D=64, F=32, E=4, k=1, seed=0)
    try:
        oracle.ffn(synth.make_x(w), np.array([[3]], np.int32), np.ones((1, 1)), store_for(w, [0]))
    except KeyError:
        return
    raise AssertionError("expected KeyError")


def test_token_subset_equals_full_rows():
    w = synth.WORKLOADS["tiny"]
    x, lg = synth.make_x(w), synth.make_logits(w)
    full = reference(w, x, lg)["out"]
    sub = reference(w, x, lg, tokens=[6, 1])["out"]
    np.testing.assert_array_equal(sub, full[[6, 1]])


def test_router_logits_and_shared_expert_match_numpy():
    w = synth.Workload("r", T=3, D=64, F=32, E=8, k=2, seed=5, router="xwr", shared=True)
    x = synth.make_x(w)
    wr = synth.make_w_router(w)
    lg = oracle.router_logits(x, wr)
    np.testing.assert_allclose(lg, bf16_to_f64(x) @ wr.astype(np.float64).T, rtol=1e-12, atol=1e-15)
    sh = synth.make_shared(w)
    out = np.zeros((3, w.D))
    oracle.shared_ffn(x, sh["sh_gate"], sh["sh_up"], sh["sh_down"], out)
    xf = bf16_to_f64(x)
    expect = expert_ffn_dense(xf, bf16_to_f64(sh["sh_gate"]), bf16_to_f64(sh["sh_up"]),
                              bf16_to_f64(sh["sh_down"]))
    assert _rel(out, expect) < 1e-13
    ref = reference(w, x, None)
    layer = _decoded_layer(w)
    assert _rel(ref["out"], moe_dense(x, lg, w.k, layer) + expect) < 1e-12
