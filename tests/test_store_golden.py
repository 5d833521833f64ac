"""The store format, frozen: the tiny layer's store in tests/golden/store_tiny.txt
(written by tests/golden/make_store_golden.py from the oracle) is rebuilt
byte for byte by the oracle and by the library's encoder, and decodes back
to the layer's canonical bytes."""
import os

import numpy as np

import oracle.store as S
import synth
from conftest import golden_path

E, D, F, SEED = 2, 64, 64, 13


def _read():
    rec, tab, blob, sec = [], [], [], None
    for line in open(golden_path("store_tiny.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line in ("records", "tables", "blob"):
            sec = line
            continue
        if sec == "records":
            rec.append([int(v) for v in line.split()])
        elif sec == "tables":
            t = np.zeros(256, np.uint16)
            for item in line.split():
                b, f = item.split(":")
                t[int(b)] = int(f)
            tab.append(t)
        else:
            blob.append(bytes.fromhex(line))
    tpe = S.tiles_per_expert(D, F)
    return {"records": np.array(rec, np.uint32).reshape(E, tpe, 8),
            "tables": np.stack(tab).reshape(E, 6, 256),
            "blob": np.frombuffer(b"".join(blob), np.uint8)}


def _weights():
    return {nm: np.ascontiguousarray(np.stack(
        [synth.expert_weights(SEED, e, D, F, dist=synth.CODES_PEAKED)[nm].ravel()
         for e in range(E)])) for nm in S.NAMES}


def test_golden_store_is_rebuilt_by_both_encoders_and_decodes():
    import mxfp4_routed_expert_03_gb300 as m
    gold, w = _read(), _weights()
    ref = S.build_store(w, E, D, F)
    for k in ("records", "tables", "blob"):
        np.testing.assert_array_equal(ref[k], gold[k], err_msg=k)
    cap = m.moe_store_blob_bound(E, D, F)
    blob = np.zeros(cap, np.uint8)
    tiles = np.zeros_like(gold["records"])
    tabs = np.zeros_like(gold["tables"])
    hw = m.moe_weights(*[w[nm].ctypes.data for nm in S.NAMES], None, None, None, None)
    n = m.moe_store_encode(E, D, F, hw, blob.ctypes.data, cap, tiles.ctypes.data,
                           tabs.ctypes.data, 2)
    np.testing.assert_array_equal(blob[:n], gold["blob"])
    np.testing.assert_array_equal(tiles, gold["records"])
    np.testing.assert_array_equal(tabs, gold["tables"])
    back = S.decode_store(gold, E, D, F)
    for a, nm in enumerate(S.NAMES):
        want = S.canonical(w[nm]) if a % 2 == 0 else w[nm]
        np.testing.assert_array_equal(back[nm], want)
