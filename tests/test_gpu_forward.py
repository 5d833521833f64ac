"""GPU layer-major path (moe_plan + moe_forward, tcgen05 grouped GEMMs) vs the oracle."""
import numpy as np
import pytest
import torch

import synth
from harness import assert_close, bf16_dev_to_f64, errors, host_layer_weights, to_dev_bf16
from oracle.run import reference

pytestmark = pytest.mark.gpu


def _run(w, weights, x_np, lg_np, path="forward"):
    from mxfp4_routed_expert_03_gb300 import check
    from mxfp4_routed_expert_03_gb300.layer import Layer, Plan
    T = x_np.shape[0]
    layer = Layer(w.D, w.F, w.E, w.k, weights)
    plan = Plan(T, w.E, w.k)
    x = to_dev_bf16(x_np)
    check(layer.plan(T, torch.from_numpy(lg_np).cuda(), None, plan), "plan")
    out = torch.empty((T, w.D), dtype=torch.int16, device="cuda")
    fn = layer.forward if path == "forward" else layer.decode
    check(fn(T, x, plan, out), path)
    st = layer.status()
    layer.close()
    assert st == 0, st
    return bf16_dev_to_f64(out), plan


@pytest.fixture(scope="module")
def tiny_weights():
    return host_layer_weights(synth.WORKLOADS["tiny"])


def test_tiny_layer_all_tokens(tiny_weights):
    w = synth.WORKLOADS["tiny"]
    x, lg = synth.make_x(w), synth.make_logits(w)
    got, _ = _run(w, tiny_weights, x, lg)
    e = assert_close(got, reference(w, x, lg)["out"])
    print("tiny forward", e)


@pytest.mark.parametrize("T", [1, 3, 17, 130, 1000])
def test_tiny_shapes_ragged_and_multi_tile_segments(tiny_weights, T):
    w = synth.WORKLOADS["tiny"]
    x, lg = synth.make_x(w, 11, T=T), synth.make_logits(w, 11, T=T)
    tok = np.arange(T) if T <= 130 else np.random.default_rng(T).choice(T, 48, replace=False)
    got, plan = _run(w, tiny_weights, x, lg)
    ref = reference(w, x, lg, tokens=tok)
    if T == 1000:
        assert plan.counts.cpu().numpy().max() > 112   # several token tiles per expert
    e = assert_close(got[tok], ref["out"])
    print("tiny forward T=%d" % T, e)


@pytest.mark.parametrize("T", [16, 111, 112, 113, 224, 500])
def test_tiny_one_expert_holds_all_rows(tiny_weights, T):
    """T = 16 fills one narrow (16-row) token tile; 111..113 and 224 sit at
    the wide tile's 112 rows and its multiples; 500 spans five wide tiles."""
    w = synth.WORKLOADS["tiny"]
    x, lg = synth.make_x(w, 5, T=T), synth.make_logits(w, 5, T=T)
    lg[:, 9] = 60.0
    got, plan = _run(w, tiny_weights, x, lg)
    assert plan.counts.cpu().numpy()[9] == T
    tok = np.arange(T) if T <= 16 else np.unique(np.r_[np.arange(0, T, 11), 110, 111, 112,
                                                            T - 2, T - 1])
    tok = tok[tok < T]
    assert_close(got[tok], reference(w, x, lg, tokens=tok)["out"])


NT_WIDE = 112   # token rows per tile of the prefill GEMMs


def tile_edge_tokens(perm: np.ndarray, offsets: np.ndarray, k: int, e: int) -> np.ndarray:
    """Tokens at the edges of expert e's token tiles: the GEMMs split a segment
    of c rows into ceil(c / 112) tiles of near-equal size (rows j*c/ntt ..),
    so these are the first and last row of every tile, the last tile being
    the partial one when c is not a multiple of 112."""
    s0, c = int(offsets[e]), int(offsets[e + 1] - offsets[e])
    ntt = -(-c // NT_WIDE)
    rows = set()
    for j in range(ntt):
        r0, r1 = j * c // ntt, (j + 1) * c // ntt
        rows.update((r0, r1 - 1))
    return np.array(sorted({int(perm[s0 + r]) // k for r in rows}), dtype=np.int64)


@pytest.mark.parametrize("name,n_check", [("prefill4k", 16), ("skewed8k", 16)])
def test_k3_prefill_sampled_tokens(k3_layer, name, n_check):
    """Random tokens plus the tokens at the tile edges of the longest segment
    (skewed8k: the most popular Zipf expert, several tiles, the last partial)
    and of one segment with a single tile."""
    w = synth.WORKLOADS[name]
    x, lg = synth.make_x(w), synth.make_logits(w)
    got, plan = _run(w, k3_layer, x, lg)
    perm, offsets = plan.perm.cpu().numpy(), plan.offsets.cpu().numpy()
    counts = np.diff(offsets)
    longest = int(np.argmax(counts))
    single = int(np.flatnonzero((counts > 0) & (counts <= NT_WIDE))[0])
    edges = np.concatenate([tile_edge_tokens(perm, offsets, w.k, longest),
                            tile_edge_tokens(perm, offsets, w.k, single)])
    rnd = np.random.default_rng(1).choice(w.T, n_check, replace=False)
    tok = np.unique(np.concatenate([rnd, edges]))
    if name == "skewed8k":
        assert counts[longest] > 2 * NT_WIDE and counts[longest] % NT_WIDE != 0
    ref = reference(w, x, lg, tokens=tok)
    np.testing.assert_array_equal(perm, ref["plan"]["perm"])
    e = assert_close(got[tok], ref["out"])
    assert np.all(np.isfinite(got))
    print(name, "longest segment", counts[longest], "tokens checked", len(tok), e)


@pytest.mark.parametrize("T", [1, 4, 8, 16])
def test_crossover_decode_and_forward_agree(k3_layer, T):
    w = synth.WORKLOADS["decode16"]
    x, lg = synth.make_x(w, 20 + T, T=T), synth.make_logits(w, 20 + T, T=T)
    got_f, plan_f = _run(w, k3_layer, x, lg, "forward")
    got_d, plan_d = _run(w, k3_layer, x, lg, "decode")
    for name in ("topk_idx", "counts", "offsets", "perm", "inv"):
        np.testing.assert_array_equal(getattr(plan_f, name).cpu().numpy(),
                                      getattr(plan_d, name).cpu().numpy())
    af, ad = plan_f.active.cpu().numpy(), plan_d.active.cpu().numpy()
    np.testing.assert_array_equal(af[: 1 + af[0]], ad[: 1 + ad[0]])
    ref = reference(w, x, lg)["out"]
    ef = assert_close(got_f, ref)
    ed = assert_close(got_d, ref)
    print("crossover T=%d forward" % T, ef, "decode", ed)


def test_zero_tokens_is_a_noop(tiny_weights):
    from mxfp4_routed_expert_03_gb300.layer import Layer, Plan
    w = synth.WORKLOADS["tiny"]
    layer = Layer(w.D, w.F, w.E, w.k, tiny_weights)
    plan = Plan(0, w.E, w.k)
    x = torch.empty((1, w.D), dtype=torch.int16, device="cuda")
    out = torch.full((1, w.D), 7, dtype=torch.int16, device="cuda")
    assert layer.forward(0, x, plan, out) == 0
    assert layer.decode(0, x, plan, out) == 0
    assert int(out[0, 0].item()) == 7   # nothing written
    assert layer.status() == 0
    layer.close()
