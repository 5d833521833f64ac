"""Expert streaming (HBM slot cache over pinned host memory) vs the oracle and
the replacement rule's reference."""
import numpy as np
import pytest
import torch

import synth
from harness import assert_close, bf16_dev_to_f64, host_layer_weights, to_dev_bf16
from oracle.run import reference
from stream_lru import LruModel

pytestmark = pytest.mark.gpu


def _host_copy(weights: dict) -> dict:
    return {k: v.cpu().pin_memory() for k, v in weights.items()}


def _run(layer, w, x_np, lg_np):
    from mxfp4_routed_expert_03_gb300 import check
    from mxfp4_routed_expert_03_gb300.layer import Plan
    T = x_np.shape[0]
    plan = Plan(T, w.E, w.k)
    check(layer.plan(T, torch.from_numpy(lg_np).cuda(), None, plan), "plan")
    out = torch.empty((T, w.D), dtype=torch.int16, device="cuda")
    check(layer.forward(T, to_dev_bf16(x_np), plan, out), "forward")
    a = plan.active.cpu().numpy()
    return bf16_dev_to_f64(out), [int(e) for e in a[1:1 + a[0]]]


def test_tiny_streaming_layer_matches_oracle_and_rule():
    from mxfp4_routed_expert_03_gb300.layer import StreamingLayer
    w = synth.WORKLOADS["tiny"]
    S = 12
    layer = StreamingLayer(w.D, w.F, w.E, w.k, _host_copy(host_layer_weights(w)), S)
    model = LruModel(w.E, S)
    for i, T in enumerate([1, 3, 2, 3, 1, 3, 3, 2]):
        x, lg = synth.make_x(w, 60 + i, T=T), synth.make_logits(w, 60 + i, T=T)
        got, active = _run(layer, w, x, lg)
        assert layer.status() == 0
        e = assert_close(got, reference(w, x, lg)["out"])
        misses = model.call(active)
        st = layer.cache_state()
        np.testing.assert_array_equal(st["slot_of"], model.slot_of)
        np.testing.assert_array_equal(st["expert_of"], model.expert_of)
        np.testing.assert_array_equal(st["stamp"], model.stamp)
        hits, total_misses, last = layer.stats()
        assert (hits, total_misses, last) == (model.hits, model.misses, len(misses))
        print("call %d T=%d misses %d" % (i, T, len(misses)), e)
    assert model.hits > 0 and model.misses > S   # the sequence both hits and evicts
    layer.close()


def test_streaming_rejections():
    import mxfp4_routed_expert_03_gb300 as m
    from mxfp4_routed_expert_03_gb300.layer import Plan, StreamingLayer
    w = synth.WORKLOADS["tiny"]
    layer = StreamingLayer(w.D, w.F, w.E, w.k, _host_copy(host_layer_weights(w)), 8)
    T = 3   # 3 * 4 = 12 > 8 slots < 32 experts
    plan = Plan(T, w.E, w.k)
    x = to_dev_bf16(synth.make_x(w, 1, T=T))
    m.check(layer.plan(T, torch.from_numpy(synth.make_logits(w, 1, T=T)).cuda(), None, plan))
    out = torch.empty((T, w.D), dtype=torch.int16, device="cuda")
    assert layer.forward(T, x, plan, out) == m.MOE_ERR_UNSUPPORTED
    assert layer.decode(T, x, plan, out) == m.MOE_ERR_UNSUPPORTED
    assert m.moe_create_streaming(layer.desc, layer.hdesc, layer.wdesc, 8, layer.state) != 0
    layer.close()


def test_streaming_rejects_bad_arguments():
    import mxfp4_routed_expert_03_gb300 as m
    from mxfp4_routed_expert_03_gb300.layer import StreamingLayer
    w = synth.WORKLOADS["tiny"]
    layer = StreamingLayer(w.D, w.F, w.E, w.k, _host_copy(host_layer_weights(w)), 4)
    for n_slots in (0, 33, 2000):
        with pytest.raises(m.MoeError):
            m.moe_create_streaming(layer.desc, layer.hdesc, layer.wdesc, n_slots, layer.state)
    with pytest.raises(m.MoeError):
        m.moe_create_streaming(layer.desc, layer.hdesc, layer.wdesc, 4, None)
    assert m.moe_stream_state_bytes(32, 0) == 0
    layer.close()


def test_k3_shaped_streaming_sampled_tokens():
    """K3 shapes (d_model 7168, d_ff 1536, top-16) over 64 experts held in host
    memory, 32 slots: T = 2 fills the cache, later calls hit and evict."""
    from mxfp4_routed_expert_03_gb300.layer import StreamingLayer
    from harness import device_layer_weights
    base = synth.WORKLOADS["decode1"]
    w = synth.Workload("k3s", T=2, D=base.D, F=base.F, E=64, k=16, seed=base.seed)
    dev = device_layer_weights(w)
    host = _host_copy(dev)
    del dev
    torch.cuda.empty_cache()
    S = 32
    layer = StreamingLayer(w.D, w.F, w.E, w.k, host, S)
    model = LruModel(w.E, S)
    for i in range(4):
        T = 2
        x, lg = synth.make_x(w, 80 + i, T=T), synth.make_logits(w, 80 + i, T=T)
        got, active = _run(layer, w, x, lg)
        assert layer.status() == 0
        e = assert_close(got, reference(w, x, lg)["out"])
        model.call(active)
        st = layer.cache_state()
        np.testing.assert_array_equal(st["expert_of"], model.expert_of)
        print("k3 streaming call %d" % i, e, layer.stats())
    layer.close()


def test_streaming_wide_tiles_and_full_cache():
    """T = 100 takes the wide (112-row, clustered) GEMM variant through the
    slot index; 32 slots for 32 experts, so every expert is resident after
    the first call and the second call is all hits."""
    from mxfp4_routed_expert_03_gb300.layer import StreamingLayer
    w = synth.WORKLOADS["tiny"]
    layer = StreamingLayer(w.D, w.F, w.E, w.k, _host_copy(host_layer_weights(w)), w.E)
    for i, T in enumerate([100, 130]):
        x, lg = synth.make_x(w, 90 + i, T=T), synth.make_logits(w, 90 + i, T=T)
        got, active = _run(layer, w, x, lg)
        assert layer.status() == 0
        tok = np.arange(0, T, 7)
        e = assert_close(got[tok], reference(w, x, lg, tokens=tok)["out"])
        print("wide streaming T=%d" % T, e, layer.stats())
    hits, misses, last = layer.stats()
    assert misses <= w.E   # with a slot per expert each expert is copied at most once
    layer.close()


def test_streaming_with_router_and_shared_expert():
    from mxfp4_routed_expert_03_gb300 import MOE_ROUTER_XWR, check
    from mxfp4_routed_expert_03_gb300.layer import Plan, StreamingLayer
    from harness import router_and_shared
    w = synth.Workload("tiny_xwr", T=5, D=256, F=128, E=32, k=4, seed=0, router="xwr",
                       shared=True)
    wr, sh = router_and_shared(w)
    layer = StreamingLayer(w.D, w.F, w.E, w.k, _host_copy(host_layer_weights(w)), 20,
                           MOE_ROUTER_XWR, wr, sh)
    for T in (5, 1):   # inputs with no near-tie in the router logits (as in the router tests)
        x_np = synth.make_x(w, 7, T=T)
        plan = Plan(T, w.E, w.k)
        x = to_dev_bf16(x_np)
        check(layer.plan(T, None, x, plan), "plan")
        out = torch.empty((T, w.D), dtype=torch.int16, device="cuda")
        check(layer.forward(T, x, plan, out), "forward")
        assert layer.status() == 0
        ref = reference(w, x_np, None)
        np.testing.assert_array_equal(plan.topk_idx.cpu().numpy(), ref["idx"])
        e = assert_close(bf16_dev_to_f64(out), ref["out"])
        print("streaming router+shared T=%d" % T, e)
    layer.close()
