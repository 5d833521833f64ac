"""GPU routing (K1 top-k, K2 plan) against the oracle: integers bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


def _layer(E, k, D=256, F=128):
    from mxfp4_routed_expert_03_gb300.layer import Layer, alloc_weights
    wts = alloc_weights(E, D, F)
    for t in wts.values():
        t.zero_()
    return Layer(D, F, E, k, wts)


def _run_plan(lg_np, k):
    from mxfp4_routed_expert_03_gb300 import check
    from mxfp4_routed_expert_03_gb300.layer import Plan
    T, E = lg_np.shape
    layer = _layer(E, k)
    plan = Plan(T, E, k)
    check(layer.plan(T, torch.from_numpy(np.ascontiguousarray(lg_np, dtype=np.float32)).cuda(),
                     None, plan), "moe_plan")
    st = layer.status()
    return layer, plan, st


def _compare(lg_np, k):
    layer, plan, st = _run_plan(lg_np, k)
    assert st == 0
    T, E = lg_np.shape
    idx, w = oracle.route(lg_np.astype(np.float64), k)
    p = oracle.plan(idx, E)
    np.testing.assert_array_equal(plan.topk_idx.cpu().numpy(), idx)
    np.testing.assert_allclose(plan.topk_w.cpu().numpy(), w, rtol=2e-6, atol=1e-7)
    np.testing.assert_array_equal(plan.counts.cpu().numpy(), p["counts"])
    np.testing.assert_array_equal(plan.offsets.cpu().numpy(), p["offsets"])
    np.testing.assert_array_equal(plan.perm.cpu().numpy()[: T * k], p["perm"])
    np.testing.assert_array_equal(plan.inv.cpu().numpy()[: T * k], p["inv"])
    act = plan.active.cpu().numpy()
    np.testing.assert_array_equal(act[: 1 + act[0]], p["active"])
    layer.close()
    return p


@pytest.mark.parametrize("name", ["tiny", "decode1", "decode4", "decode16", "prefill4k",
                                  "skewed8k"])
def test_plan_matches_oracle_on_workloads(name):
    w = synth.WORKLOADS[name]
    p = _compare(synth.make_logits(w), w.k)
    if name == "skewed8k":
        assert (p["counts"] == 0).any()


@pytest.mark.parametrize("T", [1, 63, 64, 65, 130, 1000])
def test_plan_ragged_sizes_both_paths(T):
    _compare(synth.normal_f32(T, synth.LOGITS, T, 896), 16)


def test_plan_other_k_and_e():
    for E, k in ((32, 1), (32, 32), (1024, 32), (7, 3), (100, 9)):
        _compare(synth.normal_f32(E + k, synth.LOGITS, 77, E), k)


def test_plan_ties_and_signed_zero():
    T, E = 70, 40
    lg = np.zeros((T, E), np.float32)
    lg[1::2] = -0.0
    lg[::3, ::5] = 1.0
    lg[5] = np.where(np.arange(E) % 2 == 0, 0.0, -0.0).astype(np.float32)
    _compare(lg, 8)
    _compare(lg[:9], 8)   # single-CTA path


def test_plan_one_expert_holds_all_rows():
    T, E = 300, 896
    lg = synth.normal_f32(1, synth.LOGITS, T, E)
    lg[:, 7] = 100.0
    p = _compare(lg, 16)
    assert p["counts"][7] == T


def test_plan_nan_logits_flagged_and_plan_stays_valid():
    from mxfp4_routed_expert_03_gb300 import MOE_ERR_NAN_LOGIT
    for T in (4, 200):
        lg = synth.normal_f32(2, synth.LOGITS, T, 64)
        lg[1, 3] = np.nan
        layer, plan, st = _run_plan(lg, 4)
        assert st == MOE_ERR_NAN_LOGIT
        idx = plan.topk_idx.cpu().numpy()
        assert idx.min() >= 0 and idx.max() < 64
        assert all(len(set(r)) == 4 for r in idx.tolist())
        assert 3 not in idx[1].tolist()
        assert layer.status() == 0    # cleared after reading
        layer.close()


def test_plan_zero_tokens_is_noop():
    from mxfp4_routed_expert_03_gb300.layer import Plan
    layer = _layer(32, 4)
    assert layer.plan(0, None, None, Plan(0, 32, 4)) == 0
    layer.close()


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 8, 9, 16])
def test_plan_small_batches_threshold_and_fallback(T):
    """The small-batch kernel selects each token with one warp: the keys at or
    above the k-th largest lane maximum, sorted, when there are at most 64 of
    them (normal logits; logits on a fine grid, with ties at and around the
    k-th value), else the bitwise search (a coarse grid: more equal keys than
    places at the k-th value; all-equal rows)."""
    _compare(synth.normal_f32(300 + T, synth.LOGITS, T, 896), 16)
    fine = np.round(synth.normal_f32(450 + T, synth.LOGITS, T, 896) * 16.0) / 16.0
    _compare(fine.astype(np.float32), 16)
    coarse = np.round(synth.normal_f32(400 + T, synth.LOGITS, T, 896) * 2.0) / 2.0
    _compare(coarse.astype(np.float32), 16)
    flat = np.zeros((T, 1024), np.float32)
    flat[:, 1::3] = -0.0
    _compare(flat, 32)
    _compare(synth.normal_f32(500 + T, synth.LOGITS, T, 7), 3)


def test_plan_nan_logit_single_token():
    from mxfp4_routed_expert_03_gb300 import MOE_ERR_NAN_LOGIT
    lg = synth.normal_f32(3, synth.LOGITS, 1, 896)
    lg[0, 10] = np.nan
    layer, plan, st = _run_plan(lg, 16)
    assert st == MOE_ERR_NAN_LOGIT
    idx = plan.topk_idx.cpu().numpy()[0]
    assert len(set(idx.tolist())) == 16 and 10 not in idx.tolist()
    lg[0, 10] = -np.inf
    ref, _ = oracle.route(lg.astype(np.float64), 16)
    np.testing.assert_array_equal(idx, ref[0])
    layer.close()
