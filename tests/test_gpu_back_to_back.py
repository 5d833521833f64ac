"""Many small-batch calls queued back to back on one stream, with no host
synchronisation between them.

The small-batch chain (plan, fused quantise/gather, the two grouped GEMMs,
finalize) is launched with programmatic dependent launch: a kernel may start
while its predecessor is still running and waits for it only where it reads
its output. The reuse of the same plan, workspace and accumulator by
consecutive calls is where a missing wait would show: every queued call must
still give its own inputs' answer (checked against the oracle, within the
parity tolerance) and no device-side error may be recorded.
"""
import numpy as np
import pytest
import torch

import synth
from harness import assert_close, bf16_dev_to_f64, host_layer_weights, to_dev_bf16
from oracle.run import reference

pytestmark = pytest.mark.gpu


def _queue(w, weights, T, n_calls, path):
    from mxfp4_routed_expert_03_gb300 import check
    from mxfp4_routed_expert_03_gb300.layer import Layer, Plan
    sets = [(synth.make_x(w, 200 + i, T=T), synth.make_logits(w, 200 + i, T=T)) for i in range(3)]
    xs = [to_dev_bf16(x) for x, _ in sets]
    lgs = [torch.from_numpy(lg).cuda() for _, lg in sets]
    layer = Layer(w.D, w.F, w.E, w.k, weights)
    layer.prepare()
    plan = Plan(T, w.E, w.k)
    outs = [torch.empty((T, w.D), dtype=torch.int16, device="cuda") for _ in range(n_calls)]
    torch.cuda.synchronize()
    run = layer.forward if path == "forward" else layer.decode
    for i in range(n_calls):   # one plan buffer and one workspace for every call
        s = i % len(sets)
        check(layer.plan(T, lgs[s], None, plan), "plan")
        check(run(T, xs[s], plan, outs[i]), path)
    assert layer.status() == 0
    layer.close()
    refs = [reference(w, x, lg)["out"] for x, lg in sets]
    for i in range(n_calls):
        assert_close(bf16_dev_to_f64(outs[i]), refs[i % len(sets)])


@pytest.fixture(scope="module")
def tiny_weights():
    return host_layer_weights(synth.WORKLOADS["tiny"])


@pytest.mark.parametrize("T", [1, 4, 16])
def test_tiny_layer_queued_forwards(tiny_weights, T):
    _queue(synth.WORKLOADS["tiny"], tiny_weights, T, 48, "forward")


@pytest.mark.parametrize("T", [1, 16])
def test_k3_layer_queued_forwards(k3_layer, T):
    _queue(synth.WORKLOADS["decode16"], k3_layer, T, 12, "forward")


def test_tiny_layer_queued_decodes_then_forwards(tiny_weights):
    """Decode (ordinary launches) and forward (dependent launches) interleaved."""
    from mxfp4_routed_expert_03_gb300 import check
    from mxfp4_routed_expert_03_gb300.layer import Layer, Plan
    w = synth.WORKLOADS["tiny"]
    T = 8
    x_np, lg_np = synth.make_x(w, 210, T=T), synth.make_logits(w, 210, T=T)
    layer = Layer(w.D, w.F, w.E, w.k, tiny_weights)
    layer.prepare()
    plan = Plan(T, w.E, w.k)
    x, lg = to_dev_bf16(x_np), torch.from_numpy(lg_np).cuda()
    outs = []
    for i in range(16):
        out = torch.empty((T, w.D), dtype=torch.int16, device="cuda")
        check(layer.plan(T, lg, None, plan), "plan")
        check((layer.decode if i % 2 else layer.forward)(T, x, plan, out), "call")
        outs.append(out)
    assert layer.status() == 0
    layer.close()
    ref = reference(w, x_np, lg_np)["out"]
    for o in outs:
        assert_close(bf16_dev_to_f64(o), ref)
