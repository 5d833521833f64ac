"""Pins of the FP8 expert oracle (oracle/fp8.py)."""
import math

import numpy as np
import torch

import oracle
import oracle.fp8 as F8
import synth
from oracle.run import reference


def test_all_codes_against_torch_and_the_ocp_special_values():
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    ref = ref.to(torch.float64).numpy()
    for c in range(256):
        a, b = F8.TABLE[c], ref[c]
        assert (math.isnan(a) and math.isnan(b)) or a == b, (c, a, b)
    assert np.isnan(F8.TABLE[0x7F]) and np.isnan(F8.TABLE[0xFF])
    assert int(np.isnan(F8.TABLE).sum()) == 2            # no infinities, two NaNs
    assert F8.TABLE[0x7E] == 448.0 and F8.TABLE[0xFE] == -448.0
    assert F8.TABLE[0x08] == 2.0 ** -6                   # smallest normal
    assert F8.TABLE[0x07] == 0.875 * 2.0 ** -6           # largest subnormal
    assert F8.TABLE[0x01] == 2.0 ** -9                   # smallest subnormal
    assert F8.TABLE[0x00] == 0.0 and math.copysign(1, F8.TABLE[0x80]) == -1.0
    assert F8.TABLE[0x38] == 1.0                         # exponent bias 7


def test_block_scales():
    N, K = 200, 300   # ragged last blocks in both directions
    codes = np.full((N, K), 0x38, np.uint8)                 # all 1.0
    scales = np.arange(1, 1 + 2 * 3, dtype=np.float32).reshape(2, 3)
    d = F8.dequant(codes, scales)
    assert d[0, 0] == 1 and d[127, 127] == 1 and d[127, 128] == 2 and d[128, 0] == 4
    assert d[199, 299] == 6 and d[199, 255] == 5 and d[199, 256] == 6
    np.testing.assert_array_equal(F8.dequant(F8.encode_exact(np.array([[0.5, -3.0]])),
                                             np.ones((1, 1))), [[0.5, -3.0]])


def test_ffn_equals_the_mxfp4_oracle_on_exactly_reencoded_experts():
    """MXFP4 values of the synthetic experts (E2M1 x 2^-4..2^0) are exact in
    E4M3FN: re-encoded with unit block scales, the FP8 FFN must reproduce the
    MXFP4 oracle's output to rounding."""
    w = synth.WORKLOADS["tiny"]
    x, lg = synth.make_x(w), synth.make_logits(w)

    def expert(e):
        ew = synth.expert_weights(w.seed, e, w.D, w.F)
        out = []
        for q, s in (("gate_q", "gate_s"), ("up_q", "up_s"), ("down_q", "down_s")):
            v = oracle.dequant(ew[q], ew[s])
            n, kk = v.shape
            out += [F8.encode_exact(v), np.ones(((n + 127) // 128, (kk + 127) // 128), np.float32)]
        return out

    x64 = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    got = F8.ffn(x64, lg.astype(np.float64), w.k, expert)
    ref = reference(w, x, lg)["out"]
    assert np.max(np.abs(got - ref)) <= 1e-10 * np.max(np.abs(ref))
