"""The device-side timeout path of the grouped GEMMs, driven on purpose.

With the test hook MOE_INJECT_GEMM_STALL the gate/up GEMM's first MMA issuer
waits on a barrier that nothing signals, under a short wait limit (2e6 SM
cycles, about a millisecond). That wait runs out while the CTA's producers
have operand copies in flight; the kernel must record
MOE_ERR_DEVICE_TIMEOUT, wind down (drain its MMAs, wait for every copy it
issued, free its tensor memory) and return, leaving the context usable. The
next call on the same handle, with the hook off, must match the oracle.

No GPU fault is involved: the wait that runs out is an ordinary bounded
mbarrier wait, and nothing traps.
"""
import numpy as np
import pytest
import torch

import synth
from harness import assert_close, bf16_dev_to_f64, host_layer_weights, to_dev_bf16
from oracle.run import reference

pytestmark = pytest.mark.gpu

SHORT_LIMIT = 2_000_000


def _stall_then_recover(w, weights, T, seed):
    from mxfp4_routed_expert_03_gb300 import (MOE_ERR_DEVICE_TIMEOUT, MOE_INJECT_GEMM_STALL,
                                              MOE_INJECT_NONE, check, moe_set_fault_injection)
    from mxfp4_routed_expert_03_gb300.layer import Layer, Plan
    x_np, lg_np = synth.make_x(w, seed, T=T), synth.make_logits(w, seed, T=T)
    layer = Layer(w.D, w.F, w.E, w.k, weights)
    plan = Plan(T, w.E, w.k)
    x = to_dev_bf16(x_np)
    check(layer.plan(T, torch.from_numpy(lg_np).cuda(), None, plan), "plan")
    out = torch.empty((T, w.D), dtype=torch.int16, device="cuda")
    layer.prepare()
    assert layer.status() == 0
    check(moe_set_fault_injection(layer.h, MOE_INJECT_GEMM_STALL, SHORT_LIMIT), "inject")
    check(layer.forward(T, x, plan, out), "forward (stalled)")
    assert layer.status() == MOE_ERR_DEVICE_TIMEOUT
    check(moe_set_fault_injection(layer.h, MOE_INJECT_NONE, 0), "inject off")
    # the status word was cleared by the read; the next call runs normally
    check(layer.forward(T, x, plan, out), "forward")
    assert layer.status() == 0
    got = bf16_dev_to_f64(out)
    tok = np.arange(T) if T <= 64 else np.random.default_rng(seed).choice(T, 24, replace=False)
    e = assert_close(got[tok], reference(w, x_np, lg_np, tokens=tok)["out"])
    layer.close()
    return e


@pytest.fixture(scope="module")
def tiny_weights():
    return host_layer_weights(synth.WORKLOADS["tiny"])


@pytest.mark.parametrize("T", [8, 500])
def test_tiny_layer_stall_times_out_then_recovers(tiny_weights, T):
    """T = 8: narrow tiles (two issuers); T = 500: wide tiles."""
    print(_stall_then_recover(synth.WORKLOADS["tiny"], tiny_weights, T, 60 + T))


@pytest.mark.parametrize("T", [4, 200])
def test_k3_layer_stall_with_full_rings_then_recovers(k3_layer, T):
    """K3 tiles run 28 stages, so every ring is full (5 narrow / 2 wide
    stages in flight) when the issuer gives up."""
    print(_stall_then_recover(synth.WORKLOADS["decode4"], k3_layer, T, 70 + T))


def test_injection_arguments_are_checked(tiny_weights):
    from mxfp4_routed_expert_03_gb300 import (MOE_ERR_INVALID_ARG, MOE_INJECT_NONE,
                                              moe_set_fault_injection)
    from mxfp4_routed_expert_03_gb300.layer import Layer
    w = synth.WORKLOADS["tiny"]
    layer = Layer(w.D, w.F, w.E, w.k, tiny_weights)
    assert moe_set_fault_injection(layer.h, 7, 0) == MOE_ERR_INVALID_ARG
    assert moe_set_fault_injection(layer.h, MOE_INJECT_NONE, 1000) == MOE_ERR_INVALID_ARG
    assert moe_set_fault_injection(layer.h, MOE_INJECT_NONE, 0) == 0
    layer.close()
