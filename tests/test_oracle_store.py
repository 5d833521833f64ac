"""Pins of the compressed-store oracle (oracle/store_oracle.c) against what
the mathematics and a library routine fix: zlib's Adler-32, the E2M1 values
the canonicalisation must keep, closed forms of the frequency table, exact
round trips, the rANS code length against the entropy of the bytes under the
table, and detection of corrupted tiles."""
import math
import zlib

import numpy as np
import pytest

import oracle
import oracle.store as S
import synth


def test_adler32_matches_zlib():
    rng = np.random.default_rng(1)
    for n in (0, 1, 2, 5551, 5552, 5553, 16384, 100_000):
        d = rng.integers(0, 256, n).astype(np.uint8)
        assert S.adler32(d) == zlib.adler32(d.tobytes())
    ff = np.full(70_000, 255, np.uint8)  # sums that wrap the modulus many times
    assert S.adler32(ff) == zlib.adler32(ff.tobytes())


def test_canonical_keeps_every_e2m1_value():
    b = np.arange(256, dtype=np.uint8)
    c = S.canonical(b)
    for x, y in zip(b.tolist(), c.tolist()):
        for sh in (0, 4):
            vx, vy = oracle.e2m1((x >> sh) & 15), oracle.e2m1((y >> sh) & 15)
            assert vx == vy                       # same value (-0 == +0)
            assert ((y >> sh) & 15) != 8          # no negative zero left
            if ((x >> sh) & 15) != 8:
                assert ((x >> sh) & 15) == ((y >> sh) & 15)  # nothing else moves
    assert len(set(c.tolist())) == 15 * 15
    assert np.array_equal(S.canonical(c), c)  # idempotent


def test_freq_closed_forms():
    f = S.freq(np.repeat(np.arange(256, dtype=np.uint8), 7))
    assert np.all(f == 16)
    f = S.freq(np.full(1000, 42, np.uint8))
    assert f[42] == 4096 and f.sum() == 4096
    f = S.freq(np.array([3] * 250 + [9] * 750, np.uint8))
    assert f[3] == 1024 and f[9] == 3072
    # 128 rare bytes (each bumped up to 1) beside 128 common ones: the
    # overshoot is taken from the largest entries, never below 1
    d = np.concatenate([np.arange(128, dtype=np.uint8),
                        np.repeat(np.arange(128, 256).astype(np.uint8), 400)])
    f = S.freq(d)
    assert f.sum() == 4096 and np.all(f[:128] == 1) and np.all(f[128:] >= 1)
    rng = np.random.default_rng(2)
    for _ in range(20):
        k = int(rng.integers(1, 257))
        p = rng.dirichlet(np.full(k, 0.3))
        d = rng.choice(rng.permutation(256)[:k], size=int(rng.integers(1, 30000)), p=p).astype(np.uint8)
        f = S.freq(d)
        cnt = np.bincount(d, minlength=256)
        assert f.sum() == 4096
        assert np.all((f > 0) == (cnt > 0))
        # every entry within the adjustment budget of its proportional share
        share = cnt * 4096 / d.size
        assert np.all(np.abs(f - share) <= 1 + (cnt > 0).sum())


def _sources():
    rng = np.random.default_rng(3)
    peaked = S.canonical(synth.mx_codes(5, 1, 0, 128, 1024, dist=synth.CODES_PEAKED).ravel())
    uniform = S.canonical(synth.mx_codes(5, 2, 0, 128, 1024).ravel())
    scales = synth.mx_scales(5, 4, 0, 512, 1024).ravel()
    return {
        "peaked": peaked, "uniform_codes": uniform, "scales": scales,
        "one_byte": np.full(40000, 7, np.uint8),
        "two_bytes": rng.choice([0, 255], 40000, p=[0.9, 0.1]).astype(np.uint8),
        "random": rng.integers(0, 256, 40000).astype(np.uint8),
    }


@pytest.mark.parametrize("n", [1, 31, 32, 33, 1000, 16383, 16384])
def test_tile_round_trip(n):
    for name, src in _sources().items():
        d = src[:n]
        f = S.freq(src)  # table of the whole array, as the store builds it
        if np.any(f[d] == 0):
            continue
        st, nw, raw = S.encode_tile(d, f)
        assert len(st) == (n if raw else 128 + 2 * nw)
        if not raw:
            assert 128 + 2 * nw < n
        out, ok = S.decode_tile(st, n, nw, raw, f)
        assert ok and np.array_equal(out, d), name


def test_code_length_is_the_entropy_under_the_table():
    """16 bits per word plus what the final states hold beyond 2^16 equals
    sum(log2(4096 / f[b])) over the tile's bytes, up to rANS's small loss."""
    for name, src in _sources().items():
        d = src[:16384]
        f = S.freq(src)
        st, nw, raw = S.encode_tile(d, f)
        if raw:
            continue
        x = st[:128].view("<u4").astype(np.float64)
        stored_bits = 16 * nw + float(np.sum(np.log2(x) - 16))
        info = float(np.sum(np.log2(4096.0 / f[d].astype(np.float64))))
        assert abs(stored_bits - info) <= 0.002 * d.size + 64, (name, stored_bits, info)


def test_incompressible_tile_is_stored_raw():
    d = np.random.default_rng(4).integers(0, 256, 16384).astype(np.uint8)
    st, nw, raw = S.encode_tile(d, S.freq(d))
    assert raw and nw == 0 and np.array_equal(st, d)


def test_corrupt_tiles_are_detected():
    src = _sources()["peaked"][:16384]
    f = S.freq(src)
    st, nw, raw = S.encode_tile(src, f)
    assert not raw
    rng = np.random.default_rng(5)
    for _ in range(40):
        bad = st.copy()
        pos = int(rng.integers(0, len(bad)))
        bad[pos] ^= np.uint8(1 << int(rng.integers(0, 8)))
        out, ok = S.decode_tile(bad, 16384, nw, raw, f)
        assert (not ok) or S.adler32(out) != S.adler32(src)
    # a truncated word stream is never sound
    out, ok = S.decode_tile(st[:128 + 2 * (nw - 3)], 16384, nw - 3, False, f)
    assert not ok


@pytest.mark.parametrize("codes", [synth.CODES_UNIFORM, synth.CODES_PEAKED])
def test_store_round_trip_and_layout(codes):
    E, D, F = 3, 256, 160  # codes 20480 B = 2 tiles (the second ragged), scales 1280 B
    w = {nm: np.stack([synth.expert_weights(9, e, D, F, dist=codes)[nm].ravel() for e in range(E)])
         for nm in S.NAMES}
    st = S.build_store(w, E, D, F)
    tpe = S.tiles_per_expert(D, F)
    assert tpe == 3 * (2 + 1)
    back = S.decode_store(st, E, D, F)
    for a, nm in enumerate(S.NAMES):
        ref = S.canonical(w[nm]) if a % 2 == 0 else w[nm]
        assert np.array_equal(back[nm], ref.reshape(back[nm].shape)), nm
    rec = st["records"].reshape(-1, 8).astype(np.int64)
    off = rec[:, 0] | (rec[:, 1] << 32)
    size = np.where(rec[:, 5] & 1, rec[:, 2], 128 + 2 * rec[:, 3])
    pad = (size + 15) // 16 * 16
    assert np.all(off % 16 == 0) and off[0] == 0
    assert np.array_equal(off[1:], off[:-1] + pad[:-1])
    assert off[-1] + pad[-1] == st["blob"].size
    assert np.all(rec[:, 6:] == 0)
    assert np.all(st["tables"].sum(axis=2) == 4096)
    if codes == synth.CODES_PEAKED:
        raw_bytes = sum(w[nm].size for nm in S.NAMES)
        assert st["blob"].size < 0.95 * raw_bytes
