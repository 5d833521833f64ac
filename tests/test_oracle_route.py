"""Pins of the oracle's routing (top-k + weights) and route plan."""
import numpy as np
import pytest
from scipy.special import softmax

import oracle
import synth
from bruteforce import topk_stable


def _check_route(lg, k):
    idx, w = oracle.route(lg, k)
    np.testing.assert_array_equal(idx, topk_stable(lg, k))
    sel = np.take_along_axis(lg.astype(np.float64), idx.astype(np.int64), axis=1)
    np.testing.assert_allclose(w, softmax(sel, axis=1), rtol=1e-14, atol=0)
    assert np.all(np.abs(w.sum(axis=1) - 1.0) <= 1e-12)
    assert np.all(np.diff(w, axis=1) <= 0)      # descending logit -> descending weight
    return idx, w


def test_route_matches_stable_argsort_and_softmax():
    w = synth.WORKLOADS["tiny"]
    _check_route(synth.make_logits(w), w.k)
    lg = synth.normal_f32(3, synth.LOGITS, 64, 896)
    _check_route(lg, 16)


def test_route_ties_go_to_lower_index_and_signed_zero_equal():
    lg = np.zeros((3, 8), dtype=np.float64)
    lg[0] = [1, 2, 2, 2, 0, 0, 0, 0]
    lg[1] = [-0.0, 0.0, -0.0, 0.0, -1, -1, 5, -0.0]
    lg[2] = 3.0
    idx, w = _check_route(lg, 4)
    assert idx[0].tolist() == [1, 2, 3, 0]
    assert idx[1].tolist() == [6, 0, 1, 2]
    assert idx[2].tolist() == [0, 1, 2, 3]
    np.testing.assert_allclose(w[2], 0.25, rtol=0, atol=0)


def test_route_rejects_nan():
    lg = np.zeros((2, 8))
    lg[1, 3] = np.nan
    with pytest.raises(ValueError):
        oracle.route(lg, 2)


def test_route_k_equals_e_is_full_softmax():
    lg = synth.normal_f32(9, synth.LOGITS, 5, 32).astype(np.float64)
    idx, w = oracle.route(lg, 32)
    full = softmax(lg, axis=1)
    np.testing.assert_allclose(np.take_along_axis(full, idx.astype(np.int64), axis=1), w,
                               rtol=1e-13, atol=0)


def _check_plan(idx, E):
    T, k = idx.shape
    p = oracle.plan(idx, E)
    flat = idx.reshape(-1)
    np.testing.assert_array_equal(p["counts"], np.bincount(flat, minlength=E))
    np.testing.assert_array_equal(p["offsets"], np.concatenate([[0], np.cumsum(p["counts"])]))
    np.testing.assert_array_equal(p["perm"], np.argsort(flat, kind="stable"))
    assert p["offsets"][-1] == T * k
    np.testing.assert_array_equal(p["inv"][p["perm"]], np.arange(T * k))
    np.testing.assert_array_equal(np.bincount(p["perm"] // k, minlength=T), np.full(T, k))
    np.testing.assert_array_equal(p["active"][1:], np.nonzero(p["counts"])[0])
    assert p["active"][0] == np.count_nonzero(p["counts"])
    # perm is sorted by (expert, flat index)
    key = flat[p["perm"]].astype(np.int64) * (T * k) + p["perm"]
    assert np.all(np.diff(key) > 0)
    return p


def test_plan_matches_numpy_uniform_and_skewed():
    for name in ("tiny",):
        w = synth.WORKLOADS[name]
        idx, _ = oracle.route(synth.make_logits(w), w.k)
        _check_plan(idx, w.E)
    w = synth.WORKLOADS["skewed8k"]
    idx, _ = oracle.route(synth.make_logits(w, T=512), w.k)
    p = _check_plan(idx, w.E)
    assert (p["counts"] == 0).sum() > 0           # Zipf leaves experts empty
    assert p["counts"].max() > 4 * 512 * 16 / 896  # and long segments


def test_plan_one_expert_holds_all_rows():
    T, E, k = 40, 16, 1
    idx = np.full((T, k), 7, dtype=np.int32)
    p = _check_plan(idx, E)
    assert p["counts"][7] == T and p["active"].tolist() == [1, 7]


def test_plan_rejects_out_of_range():
    with pytest.raises(ValueError):
        oracle.plan(np.array([[0, 9]], dtype=np.int32), 8)


def test_zipf_bias_is_log_rank_over_a_permutation():
    perm, bias = synth.zipf_bias(0, 896, 1.1)
    assert sorted(perm.tolist()) == list(range(896))
    np.testing.assert_allclose(bias, -1.1 * np.log(perm + 1.0), rtol=1e-6)
