"""CPU oracle of the compressed expert store (test infrastructure only).

Wraps ``libstore_oracle.so`` built from ``store_oracle.c``, which defines the
store's format (canonical negative zeros, per-array frequency tables, 16 KiB
tiles coded by 32 interleaved rANS coders, Adler-32 per tile). Only
``tests/`` may import it. Pinned by ``tests/test_oracle_store.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libstore_oracle.so")
_SRC = os.path.join(_HERE, "store_oracle.c")
_lib = None

TILE = 16384
NAMES = ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s")


def build(force: bool = False) -> None:
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-o", _SO, _SRC])


def _L():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        i32, i64, u32, p = ctypes.c_int, ctypes.c_int64, ctypes.c_uint32, ctypes.c_void_p
        L.oracle_store_canonical.argtypes = [p, i64, p]
        L.oracle_adler32.argtypes = [p, i64]
        L.oracle_adler32.restype = u32
        L.oracle_store_freq.argtypes = [p, i64, p]
        L.oracle_store_freq.restype = i32
        L.oracle_store_encode_tile.argtypes = [p, i64, p, p, p, p]
        L.oracle_store_encode_tile.restype = i64
        L.oracle_store_decode_tile.argtypes = [p, i64, u32, i32, p, p]
        L.oracle_store_decode_tile.restype = i32
        L.oracle_store_tiles_per_expert.argtypes = [i64, i64]
        L.oracle_store_tiles_per_expert.restype = i64
        L.oracle_store_build.argtypes = [i64, i64, i64, p, p, i64, p, p]
        L.oracle_store_build.restype = i64
        _lib = L
    return _lib


def _u8(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.uint8)


def _p(a: np.ndarray) -> int:
    return a.ctypes.data


def canonical(b) -> np.ndarray:
    b = _u8(b)
    out = np.empty_like(b)
    _L().oracle_store_canonical(_p(b), b.size, _p(out))
    return out


def adler32(b) -> int:
    b = _u8(b)
    return int(_L().oracle_adler32(_p(b), b.size))


def freq(canon) -> np.ndarray:
    c = _u8(canon)
    f = np.zeros(256, np.uint16)
    if _L().oracle_store_freq(_p(c), c.size, _p(f)) != 0:
        raise ValueError("empty array")
    return f


def encode_tile(d, f) -> tuple[np.ndarray, int, bool]:
    """(stored bytes, n_words, raw) of one tile of canonical bytes d."""
    d = _u8(d)
    f = np.ascontiguousarray(f, dtype=np.uint16)
    out = np.zeros(128 + 2 * max(1, d.size), np.uint8)
    nw = ctypes.c_uint32(0)
    raw = ctypes.c_int(0)
    sz = _L().oracle_store_encode_tile(_p(d), d.size, _p(f), _p(out), ctypes.addressof(nw),
                                       ctypes.addressof(raw))
    if sz < 0:
        raise ValueError("a byte of the tile has frequency 0")
    return out[:sz].copy(), int(nw.value), bool(raw.value)


def decode_tile(stored, n: int, n_words: int, raw: bool, f) -> tuple[np.ndarray, bool]:
    """(n decoded bytes, sound) of one stored tile."""
    s = np.zeros(max(int(np.asarray(stored).size), 128 + 2 * n_words), np.uint8)
    s[:np.asarray(stored).size] = _u8(stored)
    f = np.ascontiguousarray(f, dtype=np.uint16)
    d = np.zeros(max(n, 1), np.uint8)
    bad = _L().oracle_store_decode_tile(_p(s), n, n_words, int(raw), _p(f), _p(d))
    return d[:n].copy(), bad == 0


def tiles_per_expert(D: int, F: int) -> int:
    return int(_L().oracle_store_tiles_per_expert(D, F))


def build_store(weights: dict, E: int, D: int, F: int) -> dict:
    """The store of experts 0..E-1 from host arrays weights[name] ([E][...] uint8).

    Returns blob (uint8), records ([E][tiles][8] uint32) and tables
    ([E][6][256] uint16)."""
    arrs = [_u8(weights[nm]).reshape(-1) for nm in NAMES]
    tpe = tiles_per_expert(D, F)
    cap = sum(a.size for a in arrs) + 16 * E * tpe
    blob = np.zeros(cap, np.uint8)
    rec = np.zeros((E, tpe, 8), np.uint32)
    tab = np.zeros((E, 6, 256), np.uint16)
    ptrs = (ctypes.c_void_p * 6)(*[_p(a) for a in arrs])
    n = _L().oracle_store_build(E, D, F, ptrs, _p(blob), cap, _p(rec), _p(tab))
    if n < 0:
        raise ValueError("store build failed")
    return {"blob": blob[:n].copy(), "records": rec, "tables": tab}


def decode_store(store: dict, E: int, D: int, F: int) -> dict:
    """Every expert's six canonical arrays back from a store, checking each
    tile's soundness and Adler-32 (raises on a bad tile)."""
    n = D * F
    nb = [n // 2 if a % 2 == 0 else n // 32 for a in range(6)]
    out = {nm: np.zeros((E, nb[a]), np.uint8) for a, nm in enumerate(NAMES)}
    blob, rec, tab = store["blob"], store["records"], store["tables"]
    for e in range(E):
        t = 0
        for a, nm in enumerate(NAMES):
            for p in range(0, nb[a], TILE):
                r = rec[e, t]
                off = int(r[0]) | (int(r[1]) << 32)
                nbytes, nw, raw = int(r[2]), int(r[3]), bool(r[5] & 1)
                size = nbytes if raw else 128 + 2 * nw
                d, ok = decode_tile(blob[off:off + size], nbytes, nw, raw, tab[e, a])
                if not ok or adler32(d) != int(r[4]):
                    raise ValueError(f"bad tile: expert {e} array {nm} tile {t}")
                out[nm][e, p:p + nbytes] = d
                t += 1
    return out
