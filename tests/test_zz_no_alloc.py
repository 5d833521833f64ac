"""moe_decode_noalloc: decode with the library's fixed scratch, for callers
that cannot allocate device memory.

It must give the oracle's answer (within the decode path's tolerance) and
the same answer as moe_decode (within the normwise tolerance the other parity
tests use, and in practice bit for bit, since the kernels are the same) on
consecutive calls that reuse the shared scratch, and refuse calls that do not
fit the scratch. Collected last on purpose.
"""
import numpy as np
import pytest
import torch

import synth
from harness import assert_close, bf16_dev_to_f64, host_layer_weights, to_dev_bf16
from oracle.run import reference

pytestmark = pytest.mark.gpu


# the decode path's bound in its other parity tests
DECODE_MAX_REL = 6e-3
DECODE_MAE_REL = 6e-4


def _both(layer, w, T, it):
    from mxfp4_routed_expert_03_gb300 import check, moe_decode_noalloc
    from mxfp4_routed_expert_03_gb300.layer import Plan
    x_np, lg_np = synth.make_x(w, it, T=T), synth.make_logits(w, it, T=T)
    x = to_dev_bf16(x_np)
    lg = torch.from_numpy(lg_np).cuda()
    plan = Plan(T, w.E, w.k)
    check(layer.plan(T, lg, None, plan), "moe_plan")
    ref = torch.empty((T, w.D), dtype=torch.int16, device="cuda")
    got = torch.empty_like(ref)
    check(layer.decode(T, x, plan, ref), "moe_decode")
    check(moe_decode_noalloc(layer.h, T, x, plan.buf, got), "moe_decode_noalloc")
    assert layer.status() == 0
    oracle_out = reference(w, x_np, lg_np)["out"]
    return bf16_dev_to_f64(got), bf16_dev_to_f64(ref), oracle_out


@pytest.mark.parametrize("name,T", [("tiny", 8), ("decode16", 16)])
def test_noalloc_matches_decode_on_two_calls(name, T):
    from mxfp4_routed_expert_03_gb300.layer import Layer
    w = synth.WORKLOADS[name]
    if name == "tiny":
        weights = host_layer_weights(w)
    else:
        from harness import device_layer_weights
        weights = device_layer_weights(w)
    layer = Layer(w.D, w.F, w.E, w.k, weights)
    for it in (3, 4):   # the second call finds the first call's data in the scratch
        got, ref, oracle_out = _both(layer, w, T, it)
        assert_close(got, oracle_out, DECODE_MAX_REL, DECODE_MAE_REL)
        assert_close(got, ref)
        assert np.array_equal(got, ref)
    layer.close()
    del weights
    torch.cuda.empty_cache()


def test_noalloc_rejects_calls_beyond_the_scratch():
    from mxfp4_routed_expert_03_gb300 import MOE_ERR_WORKSPACE, moe_decode_noalloc
    from mxfp4_routed_expert_03_gb300.layer import Layer, Plan
    w = synth.WORKLOADS["tiny"]
    layer = Layer(w.D, w.F, w.E, w.k, host_layer_weights(w))
    T = 65   # 65 * 4 = 260 routed rows > 256
    x = torch.zeros((T, w.D), dtype=torch.int16, device="cuda")
    out = torch.empty_like(x)
    assert moe_decode_noalloc(layer.h, T, x, Plan(T, w.E, w.k).buf, out) == MOE_ERR_WORKSPACE
    layer.close()
