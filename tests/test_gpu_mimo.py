"""The MiMo-shaped layer (256 experts, top-8; d_model 4096, d_ff 2048) through
both entry points and the compressed store, against the oracle: a second
workload of the same MXFP4 expert FFN."""
import numpy as np
import pytest
import torch

import synth
from harness import assert_close, bf16_dev_to_f64, device_layer_weights, to_dev_bf16
from oracle.run import reference

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mimo_layer():
    w = synth.WORKLOADS["mimo_decode"]
    weights = device_layer_weights(w)
    yield weights
    del weights
    torch.cuda.empty_cache()


def _run(w, weights, x_np, lg_np, path):
    from mxfp4_routed_expert_03_gb300 import check
    from mxfp4_routed_expert_03_gb300.layer import Layer, Plan
    T = x_np.shape[0]
    layer = Layer(w.D, w.F, w.E, w.k, weights)
    plan = Plan(T, w.E, w.k)
    check(layer.plan(T, torch.from_numpy(lg_np).cuda(), None, plan), "plan")
    out = torch.empty((T, w.D), dtype=torch.int16, device="cuda")
    fn = layer.forward if path == "forward" else layer.decode
    check(fn(T, to_dev_bf16(x_np), plan, out), path)
    st = layer.status()
    layer.close()
    assert st == 0, st
    return bf16_dev_to_f64(out), plan


@pytest.mark.parametrize("path", ["forward", "decode"])
@pytest.mark.parametrize("T", [1, 4, 16])
def test_mimo_decode_batches(mimo_layer, T, path):
    import dataclasses
    w = dataclasses.replace(synth.WORKLOADS["mimo_decode"], T=T)
    x, lg = synth.make_x(w, 3), synth.make_logits(w, 3)
    got, plan = _run(w, mimo_layer, x, lg, path)
    ref = reference(w, x, lg)
    np.testing.assert_array_equal(plan.perm.cpu().numpy(), ref["plan"]["perm"])
    e = assert_close(got, ref["out"])
    print("mimo", path, T, e)


def test_mimo_prefill_sampled_tokens(mimo_layer):
    w = synth.WORKLOADS["mimo_prefill4k"]
    x, lg = synth.make_x(w), synth.make_logits(w)
    got, plan = _run(w, mimo_layer, x, lg, "forward")
    tok = np.random.default_rng(2).choice(w.T, 48, replace=False)
    ref = reference(w, x, lg, tokens=tok)
    np.testing.assert_array_equal(plan.perm.cpu().numpy(), ref["plan"]["perm"])
    e = assert_close(got[tok], ref["out"])
    assert np.all(np.isfinite(got))
    print("mimo prefill4k", e)
