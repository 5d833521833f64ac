"""The library's host encoder of the compressed expert store against the
oracle's (byte for byte: blob, tile records, tables), and its argument
checks. Host code only: no GPU needed."""
import ctypes

import numpy as np
import pytest

import oracle.store as S
import synth


def _weights(E, D, F, codes, seed=9):
    return {nm: np.ascontiguousarray(np.stack(
        [synth.expert_weights(seed, e, D, F, dist=codes)[nm].ravel() for e in range(E)]))
        for nm in S.NAMES}


def _encode(m, w, E, D, F, threads=3):
    tpe = m.moe_store_tiles_per_expert(D, F)
    cap = m.moe_store_blob_bound(E, D, F)
    blob = np.zeros(cap, np.uint8)
    tiles = np.zeros((E, tpe, 8), np.uint32)
    tabs = np.zeros((E, 6, 256), np.uint16)
    hw = m.moe_weights(*[w[nm].ctypes.data for nm in S.NAMES], None, None, None, None)
    n = m.moe_store_encode(E, D, F, hw, blob.ctypes.data, cap, tiles.ctypes.data,
                           tabs.ctypes.data, threads)
    return {"blob": blob[:n], "records": tiles, "tables": tabs}


@pytest.mark.parametrize("shape", [(3, 256, 160), (2, 256, 128), (5, 512, 256)])
@pytest.mark.parametrize("codes", [synth.CODES_UNIFORM, synth.CODES_PEAKED])
def test_library_encoder_matches_oracle(shape, codes):
    import mxfp4_routed_expert_03_gb300 as m
    E, D, F = shape
    w = _weights(E, D, F, codes)
    ref = S.build_store(w, E, D, F)
    got = _encode(m, w, E, D, F)
    assert m.moe_store_tiles_per_expert(D, F) == S.tiles_per_expert(D, F)
    np.testing.assert_array_equal(got["tables"], ref["tables"])
    np.testing.assert_array_equal(got["records"], ref["records"])
    np.testing.assert_array_equal(got["blob"], ref["blob"])


def test_library_encoder_raw_tiles_and_thread_count():
    """Random bytes in a scale array (kept as they are) do not compress: raw
    tiles, same bytes as the oracle, whatever the number of threads."""
    import mxfp4_routed_expert_03_gb300 as m
    E, D, F = 4, 256, 256
    rng = np.random.default_rng(11)
    w = _weights(E, D, F, synth.CODES_UNIFORM)
    w["gate_s"] = rng.integers(0, 256, w["gate_s"].shape).astype(np.uint8)
    ref = S.build_store(w, E, D, F)
    assert np.any(ref["records"][:, :, 5] & 1)
    for threads in (1, 2, 7, 0):
        got = _encode(m, w, E, D, F, threads)
        np.testing.assert_array_equal(got["blob"], ref["blob"])
        np.testing.assert_array_equal(got["records"], ref["records"])


def test_store_sizes():
    import mxfp4_routed_expert_03_gb300 as m
    assert m.moe_store_tiles_per_expert(7168, 1536) == 3 * (336 + 21) == 1071
    assert m.moe_store_blob_bound(896, 7168, 1536) == 896 * m.moe_expert_bytes(7168, 1536)
    assert m.moe_store_tiles_per_expert(256, 160) == 9
    assert m.moe_store_blob_bound(2, 256, 160) == 2 * 3 * (16384 + 4096 + 1280)
    assert m.moe_store_tiles_per_expert(0, 128) == -1
    assert m.moe_store_blob_bound(0, 256, 128) == -1


def test_encoder_rejects_bad_arguments():
    import mxfp4_routed_expert_03_gb300 as m
    E, D, F = 2, 256, 128
    w = _weights(E, D, F, synth.CODES_UNIFORM)
    hw = m.moe_weights(*[w[nm].ctypes.data for nm in S.NAMES], None, None, None, None)
    cap = m.moe_store_blob_bound(E, D, F)
    blob = np.zeros(cap, np.uint8)
    tiles = np.zeros((E, m.moe_store_tiles_per_expert(D, F), 8), np.uint32)
    tabs = np.zeros((E, 6, 256), np.uint16)
    with pytest.raises(m.MoeError):   # capacity below the bound
        m.moe_store_encode(E, D, F, hw, blob.ctypes.data, cap - 16, tiles.ctypes.data,
                           tabs.ctypes.data)
    with pytest.raises(m.MoeError):   # missing array
        bad = m.moe_weights(None, *[w[nm].ctypes.data for nm in S.NAMES[1:]], None, None, None,
                            None)
        m.moe_store_encode(E, D, F, bad, blob.ctypes.data, cap, tiles.ctypes.data,
                           tabs.ctypes.data)
    with pytest.raises(m.MoeError):   # shape
        m.moe_store_encode(E, D, 100, hw, blob.ctypes.data, cap, tiles.ctypes.data,
                           tabs.ctypes.data)


@pytest.mark.parametrize("D,F", [(32, 32), (96, 64), (32, 1024), (2048, 96), (288, 160)])
def test_library_encoder_matches_oracle_on_irregular_shapes(D, F):
    """Multiples of 32 that are not multiples of 128: arrays far below one
    tile, scale arrays of a few dozen bytes, ragged last tiles."""
    import mxfp4_routed_expert_03_gb300 as m
    E = 3
    w = _weights(E, D, F, synth.CODES_PEAKED, seed=21)
    ref = S.build_store(w, E, D, F)
    got = _encode(m, w, E, D, F, threads=2)
    np.testing.assert_array_equal(got["tables"], ref["tables"])
    np.testing.assert_array_equal(got["records"], ref["records"])
    np.testing.assert_array_equal(got["blob"], ref["blob"])
    back = S.decode_store(ref, E, D, F)
    for a, nm in enumerate(S.NAMES):
        want = S.canonical(w[nm]) if a % 2 == 0 else w[nm]
        np.testing.assert_array_equal(back[nm], want.reshape(back[nm].shape))
