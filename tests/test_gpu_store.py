"""GPU decode of the compressed expert store (moe_store_decode and streaming
from a store) against the oracle: decoded slots byte for byte equal to the
oracle's canonical arrays, forwards equal to the oracle's FFN, corrupted
tiles reported, not faulted on."""
import numpy as np
import pytest
import torch

import oracle.store as S
import synth
from harness import assert_close, bf16_dev_to_f64, host_layer_weights, to_dev_bf16
from oracle.run import reference
from stream_lru import LruModel

pytestmark = pytest.mark.gpu


def _host_weights(E, D, F, codes, seed=3):
    return {nm: np.ascontiguousarray(np.stack(
        [synth.expert_weights(seed, e, D, F, dist=codes)[nm].ravel() for e in range(E)]))
        for nm in S.NAMES}


class _DevStore:
    """An oracle-built store made readable by the device: blob pinned, records
    and tables on the GPU."""

    def __init__(self, st: dict, blob=None):
        import mxfp4_routed_expert_03_gb300 as m
        b = st["blob"] if blob is None else blob
        self.blob = torch.from_numpy(b.copy()).pin_memory()
        self.tiles = torch.from_numpy(st["records"].view(np.int32).copy()).cuda()
        self.tables = torch.from_numpy(st["tables"].view(np.int16).copy()).cuda()
        self.desc = m.moe_store(self.blob.data_ptr(), b.size, self.tiles.data_ptr(),
                                self.tables.data_ptr())


def _decode(E, D, F, store, experts, slots, n_slots):
    import mxfp4_routed_expert_03_gb300 as m
    from mxfp4_routed_expert_03_gb300.layer import WEIGHT_NAMES, alloc_weights
    dst = alloc_weights(n_slots, D, F)
    for v in dst.values():
        v.fill_(0xA5)
    wd = m.moe_weights(*[dst[n].data_ptr() for n in WEIGHT_NAMES], None, None, None, None)
    ex = torch.tensor(experts, dtype=torch.int32, device="cuda")
    sl = torch.tensor(slots, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = m.moe_store_decode(E, D, F, store.desc, ex, sl, len(experts), wd, n_slots, status)
    assert rc == 0
    torch.cuda.synchronize()
    return {k: v.cpu().numpy().reshape(n_slots, -1) for k, v in dst.items()}, int(status.item())


def _expect(w, e, a, nm):
    return S.canonical(w[nm][e]) if a % 2 == 0 else w[nm][e]


@pytest.mark.parametrize("codes", [synth.CODES_UNIFORM, synth.CODES_PEAKED])
@pytest.mark.parametrize("shape", [(5, 256, 160), (4, 512, 256)])
def test_decode_matches_oracle(codes, shape):
    E, D, F = shape
    w = _host_weights(E, D, F, codes)
    st = S.build_store(w, E, D, F)
    store = _DevStore(st)
    experts, slots = [E - 1, 0, E // 2], [0, 2, 1]
    got, status = _decode(E, D, F, store, experts, slots, 3)
    assert status == 0
    for e, s in zip(experts, slots):
        for a, nm in enumerate(S.NAMES):
            np.testing.assert_array_equal(got[nm][s], _expect(w, e, a, nm), err_msg=f"{e} {nm}")


def test_decode_raw_tiles():
    E, D, F = 3, 256, 256
    w = _host_weights(E, D, F, synth.CODES_UNIFORM)
    w["down_s"] = np.random.default_rng(7).integers(0, 256, w["down_s"].shape).astype(np.uint8)
    st = S.build_store(w, E, D, F)
    assert np.any(st["records"][:, :, 5] & 1)
    got, status = _decode(E, D, F, _DevStore(st), [2, 1, 0], [0, 1, 2], 3)
    assert status == 0
    for e, s in zip([2, 1, 0], [0, 1, 2]):
        for a, nm in enumerate(S.NAMES):
            np.testing.assert_array_equal(got[nm][s], _expect(w, e, a, nm))


def test_decode_k3_experts():
    """Four K3-shaped experts (1071 tiles each, 16 KiB tiles throughout) with
    the peaked code distribution."""
    E, D, F = 4, 7168, 1536
    w = _host_weights(E, D, F, synth.CODES_PEAKED)
    st = S.build_store(w, E, D, F)
    raw = sum(w[nm].size for nm in S.NAMES)
    print("K3 store: %.4f of raw" % (st["blob"].size / raw))
    got, status = _decode(E, D, F, _DevStore(st), [1, 3, 0, 2], [0, 1, 2, 3], 4)
    assert status == 0
    for e, s in zip([1, 3, 0, 2], [0, 1, 2, 3]):
        for a, nm in enumerate(S.NAMES):
            np.testing.assert_array_equal(got[nm][s], _expect(w, e, a, nm))


def test_corrupt_tiles_are_reported_and_contained():
    """Host-made damage: a flipped bit inside a coded tile, a record whose
    offset points past the blob, a table that does not sum to 4096, an expert
    index out of range. The kernel reports each and never leaves a tile's
    bytes or its slot; undamaged experts still decode exactly."""
    import mxfp4_routed_expert_03_gb300 as m
    E, D, F = 4, 256, 160
    w = _host_weights(E, D, F, synth.CODES_PEAKED)
    st = S.build_store(w, E, D, F)
    tpe = S.tiles_per_expert(D, F)
    # 1. one bit of expert 1's first tile (coded: its words follow the 128-byte header)
    r = st["records"][1, 0]
    assert not (r[5] & 1)
    blob = st["blob"].copy()
    blob[int(r[0]) + 128 + 40] ^= 0x10
    got, status = _decode(E, D, F, _DevStore(st, blob), [0, 1, 2], [0, 1, 2], 3)
    assert status == m.MOE_ERR_CORRUPT_TILE
    for e in (0, 2):
        for a, nm in enumerate(S.NAMES):
            np.testing.assert_array_equal(got[nm][e], _expect(w, e, a, nm))
    # 2. an offset past the end of the blob
    bad = dict(st, records=st["records"].copy())
    bad["records"][2, tpe - 1, 0] = np.uint32(st["blob"].size + 4096)
    got, status = _decode(E, D, F, _DevStore(bad), [2, 3], [0, 1], 2)
    assert status == m.MOE_ERR_CORRUPT_TILE
    for a, nm in enumerate(S.NAMES):
        np.testing.assert_array_equal(got[nm][1], _expect(w, 3, a, nm))
    # 3. a table whose entries do not sum to 4096
    bad = dict(st, tables=st["tables"].copy())
    bad["tables"][0, 0, int(np.argmax(bad["tables"][0, 0]))] += 5
    _, status = _decode(E, D, F, _DevStore(bad), [0], [0], 1)
    assert status == m.MOE_ERR_CORRUPT_TILE
    # 4. an expert out of range, and a slot out of range
    _, status = _decode(E, D, F, _DevStore(st), [E], [0], 1)
    assert status == m.MOE_ERR_BAD_INDEX
    _, status = _decode(E, D, F, _DevStore(st), [0], [5], 1)
    assert status == m.MOE_ERR_BAD_INDEX


def test_decode_rejects_bad_arguments():
    import mxfp4_routed_expert_03_gb300 as m
    from mxfp4_routed_expert_03_gb300.layer import WEIGHT_NAMES, alloc_weights
    E, D, F = 2, 256, 128
    st = S.build_store(_host_weights(E, D, F, 0), E, D, F)
    store = _DevStore(st)
    dst = alloc_weights(1, D, F)
    wd = m.moe_weights(*[dst[n].data_ptr() for n in WEIGHT_NAMES], None, None, None, None)
    ex = torch.zeros(1, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert m.moe_store_decode(E, D, F, store.desc, ex, ex, 1, wd, 1, None) == m.MOE_ERR_INVALID_ARG
    assert m.moe_store_decode(E, D, 100, store.desc, ex, ex, 1, wd, 1, status) == m.MOE_ERR_INVALID_ARG
    assert m.moe_store_decode(E, D, F, store.desc, ex, ex, -1, wd, 1, status) == m.MOE_ERR_INVALID_ARG
    assert m.moe_store_decode(E, D, F, store.desc, ex, ex, 0, wd, 1, status) == 0
    # a blob the device cannot read (pageable memory) is refused at creation
    desc = m.moe_desc(D, F, E, 2, 0, 0)
    state = torch.empty(m.moe_stream_state_bytes(E, 1), dtype=torch.uint8, device="cuda")
    pageable = np.zeros(st["blob"].size + 16, np.uint8)
    off = (-pageable.ctypes.data) % 16
    bad = m.moe_store(pageable.ctypes.data + off, st["blob"].size, store.tiles.data_ptr(),
                      store.tables.data_ptr())
    with pytest.raises(m.MoeError):
        m.moe_create_streaming_store(desc, bad, wd, 1, state)


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


@pytest.mark.parametrize("codes", [synth.CODES_UNIFORM, synth.CODES_PEAKED])
def test_streaming_from_store_matches_oracle_and_rule(codes):
    """The tiny layer streamed from a store built by the library's encoder:
    outputs equal the oracle's, the cache follows the replacement rule, and
    the slots hold the canonical bytes of their experts."""
    from mxfp4_routed_expert_03_gb300.layer import ExpertStore, StreamingLayer
    import dataclasses
    w = dataclasses.replace(synth.WORKLOADS["tiny"], codes=codes)
    host = {k: v.cpu() for k, v in host_layer_weights(w).items()}
    store = ExpertStore(w.E, w.D, w.F, host)
    ref_st = S.build_store({k: v.numpy().reshape(w.E, -1) for k, v in host.items()}, w.E, w.D, w.F)
    assert store.blob_bytes == ref_st["blob"].size
    np.testing.assert_array_equal(store.blob[:store.blob_bytes].numpy(), ref_st["blob"])
    S_ = 12
    layer = StreamingLayer(w.D, w.F, w.E, w.k, None, S_, store=store)
    model = LruModel(w.E, S_)
    for i, T in enumerate([1, 3, 2, 3, 1, 3]):
        x, lg = synth.make_x(w, 60 + i, T=T), synth.make_logits(w, 60 + i, T=T)
        got, active = _run(layer, w, x, lg)
        assert layer.status() == 0
        e = assert_close(got, reference(w, x, lg)["out"])
        model.call(active)
        st = layer.cache_state()
        np.testing.assert_array_equal(st["expert_of"], model.expert_of)
        print("store call %d T=%d" % (i, T), e)
    st = layer.cache_state()
    for s, ex in enumerate(st["expert_of"]):
        if ex < 0:
            continue
        for a, nm in enumerate(S.NAMES):
            want = host[nm][ex].numpy().ravel()
            want = S.canonical(want) if a % 2 == 0 else want
            np.testing.assert_array_equal(layer.weights[nm][s].cpu().numpy().ravel(), want)
    layer.close()


def test_k3_shaped_streaming_from_store():
    """K3 shapes over 64 experts with peaked codes behind 32 slots."""
    from mxfp4_routed_expert_03_gb300.layer import ExpertStore, StreamingLayer
    from harness import device_layer_weights
    base = synth.WORKLOADS["decode1"]
    w = synth.Workload("k3s", T=2, D=base.D, F=base.F, E=64, k=16, seed=base.seed,
                       codes=synth.CODES_PEAKED)
    dev = device_layer_weights(w)
    host = {k: v.cpu() for k, v in dev.items()}
    del dev
    torch.cuda.empty_cache()
    store = ExpertStore(w.E, w.D, w.F, host)
    print("K3 store over 64 experts: %.4f of raw" % (store.blob_bytes / store.raw_bytes))
    layer = StreamingLayer(w.D, w.F, w.E, w.k, None, 32, store=store)
    model = LruModel(w.E, 32)
    for i in range(4):
        x, lg = synth.make_x(w, 80 + i, T=2), synth.make_logits(w, 80 + i, T=2)
        got, active = _run(layer, w, x, lg)
        assert layer.status() == 0
        e = assert_close(got, reference(w, x, lg)["out"])
        model.call(active)
        np.testing.assert_array_equal(layer.cache_state()["expert_of"], model.expert_of)
        print("k3 store streaming call %d" % i, e, layer.stats())
    layer.close()
