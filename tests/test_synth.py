"""The seeded input generator: Philox known answers and the workload recipes."""
import numpy as np

import synth


def test_philox4x32_10_known_answers():
    # Known-answer vectors published with the Random123 library (Salmon et al.,
    # SC'11) for philox4x32 with 10 rounds.
    kat = [
        ([0, 0, 0, 0], [0, 0], [0x6627e8d5, 0xe169c58d, 0xbc57ac4c, 0x9b00dbd8]),
        ([0xffffffff] * 4, [0xffffffff] * 2, [0x408f276d, 0x41c83b0e, 0xa20bc7c6, 0x6d5451fd]),
        ([0x243f6a88, 0x85a308d3, 0x13198a2e, 0x03707344], [0xa4093822, 0x299f31d0],
         [0xd16cfe09, 0x94fdcceb, 0x5001e420, 0x24126ea1]),
    ]
    for ctr, key, out in kat:
        assert synth.philox(ctr, key) == out


def test_weight_distributions():
    q = synth.mx_codes(0, synth.GATE_Q, 3, 256, 512)
    codes = np.concatenate([q & 15, q >> 4]).ravel()
    cnt = np.bincount(codes, minlength=16)
    assert cnt.min() > 0.9 * codes.size / 16 and cnt.max() < 1.1 * codes.size / 16
    s = synth.mx_scales(0, synth.GATE_S, 3, 256, 512)
    assert set(np.unique(s).tolist()) == {123, 124, 125, 126, 127}


def test_streams_are_keyed_by_expert_and_tensor():
    a = synth.mx_codes(0, synth.GATE_Q, 0, 4, 64)
    assert not np.array_equal(a, synth.mx_codes(0, synth.GATE_Q, 1, 4, 64))
    assert not np.array_equal(a, synth.mx_codes(0, synth.UP_Q, 0, 4, 64))
    np.testing.assert_array_equal(a, synth.mx_codes(0, synth.GATE_Q, 0, 4, 64))
    # rows are independent of how many rows are drawn
    np.testing.assert_array_equal(a[:2], synth.mx_codes(0, synth.GATE_Q, 0, 2, 64))


def test_normals():
    x = synth.normal_f32(1, synth.X, 200, 1000)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01
    b = synth.normal_bf16(1, synth.X, 200, 1000)
    xf = (b.astype(np.uint32) << 16).view(np.float32)
    assert np.max(np.abs(xf - x)) <= np.max(np.abs(x)) * 2.0 ** -8


def test_peaked_code_distribution():
    """Magnitudes follow the stated table (parts of 2^15) and the sign bit is
    uniform, so half of the zero codes are negative zeros."""
    q = synth.mx_codes(0, synth.GATE_Q, 3, 512, 1024, dist=synth.CODES_PEAKED)
    codes = np.concatenate([q & 15, q >> 4]).ravel()
    table = np.array([3260, 6318, 5757, 4928, 5580, 4299, 2218, 408]) / 32768.0
    mag = np.bincount(codes & 7, minlength=8) / codes.size
    assert np.all(np.abs(mag - table) < 4 * np.sqrt(table / codes.size) + 1e-4)
    neg = (codes >> 3).mean()
    assert abs(neg - 0.5) < 0.005
    z = codes[(codes & 7) == 0]
    assert abs((z == 8).mean() - 0.5) < 0.01
    # the uniform distribution is unchanged by the new entry point
    np.testing.assert_array_equal(synth.mx_codes(0, synth.GATE_Q, 3, 8, 64),
                                  synth.mx_codes(0, synth.GATE_Q, 3, 8, 64, dist=synth.CODES_UNIFORM))


def test_fp8_expert_draws():
    """FP8 lane: each code byte comes from one Philox byte b as
    (b & 0x80) | (0x20 + (b & 0x3F)), each block scale from one word w as the
    fp32 2^-7 (1 + (w >> 9) 2^-23); recomputed here from the raw stream."""
    import oracle.fp8 as F8
    seed, e, D, F = 5, 3, 256, 128
    w = synth.fp8_expert_weights(seed, e, D, F)
    assert w["gate_q"].shape == (F, D) and w["down_q"].shape == (D, F)
    assert w["gate_s"].shape == (1, 2) and w["down_s"].shape == (2, 1)
    # code bytes of gate row 1, block 2 from the raw Philox block
    words = synth.philox([2, 1, e, seed >> 32], [seed & 0xFFFFFFFF, synth.F8_GATE_Q])
    raw = [(wd >> (8 * j)) & 0xFF for wd in words for j in range(4)]
    want = [(b & 0x80) | (0x20 + (b & 0x3F)) for b in raw]
    assert w["gate_q"][1, 32:48].tolist() == want
    # scale (0, 1) of up from word 1 of block (0, 0)
    wd = synth.philox([0, 0, e, seed >> 32], [seed & 0xFFFFFFFF, synth.F8_UP_S])[1]
    assert w["up_s"][0, 1] == np.float32(2.0 ** -7 * (1 + (wd >> 9) * 2.0 ** -23))
    vals = F8.TABLE[w["up_q"]]
    assert np.all(np.isfinite(vals))
    assert np.abs(vals).min() == 0.125 and np.abs(vals).max() <= 30.0
    assert np.all((w["down_s"] >= 2.0 ** -7) & (w["down_s"] < 2.0 ** -6))
