"""GPU decode path (moe_plan + moe_decode) against the CPU oracle."""
import numpy as np
import pytest
import torch

import synth
from harness import (assert_close, bf16_dev_to_f64, device_layer_weights, errors,
                     host_layer_weights, to_dev_bf16)
from oracle.run import reference

pytestmark = pytest.mark.gpu

# The decode path dequantises exactly and accumulates in fp32; beyond the
# stated tolerance its error should stay near bf16 output rounding.
DECODE_MAX_REL = 6e-3
DECODE_MAE_REL = 6e-4


def _decode(w, weights, x_np, lg_np):
    from mxfp4_routed_expert_03_gb300 import check
    from mxfp4_routed_expert_03_gb300.layer import Layer, Plan
    T = x_np.shape[0]
    layer = Layer(w.D, w.F, w.E, w.k, weights)
    plan = Plan(T, w.E, w.k)
    x = to_dev_bf16(x_np)
    check(layer.plan(T, torch.from_numpy(lg_np).cuda(), None, plan), "plan")
    out = torch.empty((T, w.D), dtype=torch.int16, device="cuda")
    check(layer.decode(T, x, plan, out), "decode")
    assert layer.status() == 0
    layer.close()
    return bf16_dev_to_f64(out), plan


@pytest.fixture(scope="module")
def tiny_weights():
    return host_layer_weights(synth.WORKLOADS["tiny"])


def test_tiny_layer_all_tokens(tiny_weights):
    w = synth.WORKLOADS["tiny"]
    x, lg = synth.make_x(w), synth.make_logits(w)
    got, _ = _decode(w, tiny_weights, x, lg)
    ref = reference(w, x, lg)
    e = assert_close(got, ref["out"], DECODE_MAX_REL, DECODE_MAE_REL)
    print("tiny decode", e)


@pytest.mark.parametrize("T", [1, 3, 5, 37, 130])
def test_tiny_shapes_ragged_token_counts(tiny_weights, T):
    w = synth.WORKLOADS["tiny"]
    x, lg = synth.make_x(w, 7, T=T), synth.make_logits(w, 7, T=T)
    got, _ = _decode(w, tiny_weights, x, lg)
    assert_close(got, reference(w, x, lg)["out"], DECODE_MAX_REL, DECODE_MAE_REL)


def test_tiny_one_expert_holds_all_rows(tiny_weights):
    w = synth.WORKLOADS["tiny"]
    T = 24
    x, lg = synth.make_x(w, 3, T=T), synth.make_logits(w, 3, T=T)
    lg[:, 5] = 50.0
    got, plan = _decode(w, tiny_weights, x, lg)
    assert plan.counts.cpu().numpy()[5] == T
    assert_close(got, reference(w, x, lg)["out"], DECODE_MAX_REL, DECODE_MAE_REL)


@pytest.mark.parametrize("dist", [synth.CODES_UNIFORM, synth.CODES_PEAKED])
def test_device_generator_matches_host(dist):
    w = synth.WORKLOADS["decode1"]
    from mxfp4_routed_expert_03_gb300.layer import alloc_weights
    E = 3
    wts = alloc_weights(E, w.D, w.F)
    synth.dev_fill_layer(w.seed, E, w.D, w.F, {k: v.data_ptr() for k, v in wts.items()}, dist=dist)
    torch.cuda.synchronize()
    for e in range(E):
        host = synth.expert_weights(w.seed, e, w.D, w.F, dist=dist)
        for name, arr in host.items():
            np.testing.assert_array_equal(wts[name][e].cpu().numpy(), arr, err_msg=name)


@pytest.mark.parametrize("name", ["decode1", "decode4", "decode16"])
def test_k3_layer_decode_all_tokens(k3_layer, name):
    w = synth.WORKLOADS[name]
    x, lg = synth.make_x(w), synth.make_logits(w)
    got, plan = _decode(w, k3_layer, x, lg)
    ref = reference(w, x, lg)
    np.testing.assert_array_equal(plan.perm.cpu().numpy(), ref["plan"]["perm"])
    e = assert_close(got, ref["out"], DECODE_MAX_REL, DECODE_MAE_REL)
    print(name, e)
