"""Pins of the oracle's MXFP4 decode (E2M1 elements, E8M0 scales, nibble order)."""
import math

import numpy as np
import torch

import oracle
from bruteforce import decode as np_decode, e8m0_torch, ocp_e2m1_table
from conftest import golden_path


def _same(a, b):
    return (a == b and math.copysign(1, a) == math.copysign(1, b)) or (math.isnan(a) and math.isnan(b))


def test_e2m1_matches_ocp_table():
    tab = ocp_e2m1_table()
    for code in range(16):
        assert _same(oracle.e2m1(code), float(tab[code])), code


def test_e2m1_embeds_in_e4m3_through_torch():
    # Every E2M1 value is exact in E4M3 (bias 7): a normal E2M1 number with
    # exponent field e and mantissa m is E4M3 with exponent field e+6 and the
    # mantissa bit at the top of its 3 mantissa bits; 0.5 is 2^-1 (field 6).
    bits = []
    for code in range(16):
        s, e, m = code >> 3, (code >> 1) & 3, code & 1
        if e == 0:
            b = 0 if m == 0 else (6 << 3)
        else:
            b = ((e + 6) << 3) | (m << 2)
        bits.append((s << 7) | b)
    dec = torch.tensor(bits, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    for code in range(16):
        assert _same(oracle.e2m1(code), float(dec[code])), code


def test_e8m0_matches_torch_all_256():
    ref = e8m0_torch(np.arange(256, dtype=np.uint8))
    for b in range(256):
        assert _same(oracle.e8m0(b), float(ref[b])), b


def test_dequant_exhaustive_codes_by_scales():
    # One row per scale byte (0..254); each 32-wide block repeats all 16 codes.
    codes = np.arange(32) % 16
    row_q = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)
    q = np.tile(row_q, (255, 1))
    s = np.arange(255, dtype=np.uint8)[:, None]
    W = oracle.dequant(q, s)
    tab = ocp_e2m1_table()
    sc = e8m0_torch(np.arange(255, dtype=np.uint8))
    expect = tab[codes][None, :] * sc[:, None]
    assert W.shape == (255, 32)
    np.testing.assert_array_equal(W, expect)
    np.testing.assert_array_equal(np.signbit(W), np.signbit(expect))


def test_dequant_matches_numpy_decoder_random():
    rng = np.random.default_rng(5)
    q = rng.integers(0, 256, size=(37, 96), dtype=np.uint8)
    s = rng.integers(100, 140, size=(37, 6), dtype=np.uint8)
    np.testing.assert_array_equal(oracle.dequant(q, s), np_decode(q, s))


def test_hand_worked_examples():
    rows = []
    with open(golden_path("mxfp4_worked_examples.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    assert len(rows) >= 4
    for b, sb, e0, e1 in rows:
        q = np.zeros((1, 16), dtype=np.uint8)
        q[0, 0] = int(b, 16)
        s = np.full((1, 1), int(sb, 16), dtype=np.uint8)
        W = oracle.dequant(q, s)
        assert _same(W[0, 0], float(e0)), (b, sb)
        assert _same(W[0, 1], float(e1)), (b, sb)


def test_scale_block_boundary():
    # Element 31 uses scale 0, element 32 uses scale 1.
    q = np.full((1, 32), 0x22, dtype=np.uint8)   # all elements 1.0
    s = np.array([[127, 130]], dtype=np.uint8)
    W = oracle.dequant(q, s)
    assert W[0, 31] == 1.0 and W[0, 32] == 8.0
