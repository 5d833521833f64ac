"""Pins of the activation-precision study (oracle/act_study.py) and the study
itself: which activation formats keep the layer within the tolerance."""
import numpy as np
import pytest
import torch

import oracle.act_study as A
import synth
from oracle.run import reference


def test_representable_values_are_fixed_points():
    for fmt in ("e2m1", "e4m3"):
        mags = A._magnitudes(fmt)
        v = np.concatenate([mags, -mags])
        np.testing.assert_array_equal(A.round_to_format(v, fmt), v)
    assert A._magnitudes("e2m1").tolist() == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert A._magnitudes("e4m3")[-1] == 448 and A._magnitudes("e4m3")[1] == 2.0 ** -9


def test_e2m1_midpoints_round_to_even_codes_and_saturate():
    # midpoints between neighbours: the even code (even mantissa) wins
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    want = [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]
    np.testing.assert_array_equal(A.round_to_format(np.array(mids), "e2m1"), want)
    np.testing.assert_array_equal(A.round_to_format(-np.array(mids), "e2m1"), -np.array(want))
    np.testing.assert_array_equal(A.round_to_format(np.array([7.0, 100.0, -9.0]), "e2m1"),
                                  [6.0, 6.0, -6.0])


def test_e4m3_rounding_matches_torch():
    """torch's float8_e4m3fn conversion rounds to nearest even; inside the
    finite range the two must agree everywhere."""
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.normal(0, 1, 20000) * 2.0 ** rng.integers(-12, 9, 20000),
                        A._magnitudes("e4m3")[1:] * 1.0625,     # off-grid points
                        (A._magnitudes("e4m3")[1:] + A._magnitudes("e4m3")[:-1]) / 2])  # ties
    v = v[np.abs(v) <= 448]
    ref = torch.from_numpy(v).to(torch.float32).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(A.round_to_format(v, "e4m3"), ref)


def test_scale_rule():
    # amax in [4, 8): X = 1 for e2m1 (emax 2) and 2^-6 for e4m3 (emax 8)
    v = np.zeros(32)
    v[0] = 5.9
    v[1] = 0.4
    q = A.mx_quantise(v, "e2m1")
    assert q[0] == 6.0 and q[1] == 0.5
    v[0] = 8.0                       # amax 8: X = 2, 0.4 / 2 = 0.2 -> 0
    q = A.mx_quantise(v, "e2m1")
    assert q[0] == 8.0 and q[1] == 0.0
    # a block already on the grid of its own scale is unchanged
    rng = np.random.default_rng(1)
    codes = rng.integers(0, 8, 32)
    vals = A._magnitudes("e2m1")[codes] * rng.choice([-1, 1], 32)
    vals[3] = 6.0
    for s in (-5, 0, 3):
        np.testing.assert_array_equal(A.mx_quantise(vals * 2.0 ** s, "e2m1"), vals * 2.0 ** s)
    np.testing.assert_array_equal(A.mx_quantise(np.zeros(64), "e4m3"), np.zeros(64))


def test_two_term_is_far_closer_than_one_term():
    v = np.random.default_rng(2).normal(0, 1, 4096)
    e1 = np.max(np.abs(A.mx_quantise(v, "e4m3") - v))
    e2 = np.max(np.abs(A.two_term(v, "e4m3") - v))
    assert e2 < e1 / 8


def _x64(x_bf16):
    return (x_bf16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_exact_treatment_is_the_oracle_ffn():
    w = synth.WORKLOADS["tiny"]
    x, lg = synth.make_x(w), synth.make_logits(w)

    def expert(e):
        return A.decoded(synth.expert_weights(w.seed, e, w.D, w.F))

    got = A.ffn(_x64(x), lg.astype(np.float64), w.k, expert, ["exact"])["exact"]
    ref = reference(w, x, lg)["out"]
    assert np.max(np.abs(got - ref)) <= 1e-10 * np.max(np.abs(ref))


def test_activation_formats_against_the_tolerance(capsys):
    """K3 shape, two tokens of the decode workload (32 experts): bf16 h and the
    two-term E4M3 split stay inside max_rel 2e-2 / mae_rel 1e-3; one E4M3
    term and MXFP4 activations (an FP4 x FP4 mode) do not."""
    base = synth.WORKLOADS["decode1"]
    w = synth.Workload("k3t2", T=2, D=base.D, F=base.F, E=base.E, k=base.k, seed=base.seed)
    x, lg = synth.make_x(w, 5), synth.make_logits(w, 5)

    def expert(e):
        return A.decoded(synth.expert_weights(w.seed, e, w.D, w.F))

    treats = ["exact", "bf16_h", "two_term_e4m3", "one_term_e4m3", "mxfp4"]
    ys = A.ffn(_x64(x), lg.astype(np.float64), w.k, expert, treats)
    errs = {tr: A.errors(ys[tr], ys["exact"]) for tr in treats[1:]}
    with capsys.disabled():
        for tr, e in errs.items():
            print(f"\n{tr:15s} max_rel {e['max_rel']:.2e}  mae_rel {e['mae_rel']:.2e}", end="")
        print()
    ok = {tr: e["max_rel"] <= 2e-2 and e["mae_rel"] <= 1e-3 for tr, e in errs.items()}
    assert ok == {"bf16_h": True, "two_term_e4m3": True, "one_term_e4m3": False, "mxfp4": False}
