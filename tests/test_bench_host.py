"""bench.py's host-side helpers: workload shapes, the generator workload each
bench workload draws from, and the traffic lookup's source-hash guard."""
import hashlib
import os

import bench
import synth


def test_every_workload_has_a_shape_and_a_generator_workload():
    for name, wl in bench.BENCH_WORKLOADS.items():
        bench.use_shape(wl)
        base = bench.base_workload(name)
        assert (bench.D_MODEL, bench.D_FF, bench.N_EXPERTS, bench.TOP_K) == \
            (base.D, base.F, base.E, base.k), name
        assert bench.EXPERT_BYTES == 3 * (base.D * base.F // 2 + base.D * base.F // 32)
        assert wl["Ts"] and all(T > 0 for T in wl["Ts"])
    bench.use_shape({})
    assert bench.EXPERT_BYTES == 17547264           # the K3 expert, codes + scales
    assert bench.GATEUP_BYTES + bench.DOWN_BYTES == bench.EXPERT_BYTES


def test_mimo_shape_reading():
    bench.use_shape(bench.BENCH_WORKLOADS["mimo_decode"])
    # routed experts alone account for the stated 310B total over 48 layers
    total = 3 * bench.D_MODEL * bench.D_FF * bench.N_EXPERTS * 48
    assert 300e9 < total < 310e9 and bench.TOP_K == 8 and bench.N_EXPERTS == 256
    bench.use_shape({})


def test_store_workload_uses_peaked_codes():
    wl = bench.BENCH_WORKLOADS["decode_stream_store"]
    assert wl["store"] and wl["codes"] == synth.CODES_PEAKED and wl["stream_slots"] > 0


def test_traffic_lookup_requires_the_current_kernel_source():
    lines = [l.split() for l in open(os.path.join(bench.ROOT, "profiles", "traffic.txt"))
             if l.strip() and not l.startswith("#")]
    for name, h, wl, nbytes in lines:
        source = "decode.cu" if name.startswith("moe_decode") else "grouped_gemm.cu"
        src = os.path.join(bench.ROOT, "mxfp4_routed_expert_03_gb300", "csrc", source)
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        got = bench.kernel_traffic(name, source, wl)
        assert got == (float(nbytes) if h == sha else None)
    assert bench.kernel_traffic("moe_grouped_gemm_kernel<0>", "grouped_gemm.cu", "no-such") is None


def test_default_run_records_and_their_roofline_arithmetic():
    bench.use_shape({})
    assert set(bench.RECORDS) <= set(bench.BENCH_WORKLOADS)
    for name in bench.RECORDS:
        assert bench.base_workload(name).D == 7168
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0}
    # a one-token forward: 16 experts' gate/up weights, far below the tensor roof
    nbytes, flop = bench.kernel_work("forward", 1, 16)
    assert nbytes == 16 * bench.GATEUP_BYTES + 16 * (2 * 7168 + 2 * 1536)
    assert flop == 2.0 * 16 * 2 * 7168 * 1536
    r = bench.roofline("forward", nbytes, flop, nbytes / 6000e9 * 1e3 * 2, peaks, "x")
    assert r["bound"] == "hbm" and abs(r["frac"] - 0.5) < 1e-12
    assert abs(r["frac_of_binding_roof"] - 0.5) < 1e-12
    # 16384 tokens over every expert: two MMAs per algorithmic one at the FP8 rate bind
    nbytes, flop = bench.kernel_work("forward", 16384, 896)
    tensor_ms = 2 * flop / 4000e12 * 1e3
    r = bench.roofline("forward", nbytes, flop, 4 * tensor_ms, peaks, "x")
    assert r["bound"] == "tensor" and abs(r["frac_of_binding_roof"] - 0.25) < 1e-12
    assert abs(r["frac"] - 0.125) < 1e-12   # of the FP8 peak, two-term work counted once


def test_arithmetic_types_follow_the_workload():
    w = bench.BENCH_WORKLOADS
    assert bench.dtype_of(w["decode"], w["decode"]["path"]) == "mxfp4 x 2-term e4m3 -> f32"
    assert bench.dtype_of(w["prefill4k"], "forward") == "mxfp4 x 2-term e4m3 -> f32"
    assert bench.dtype_of(w["prefill4k_fp4"], "forward") == "mxfp4 x mxfp4 -> f32"
    assert bench.dtype_of(w["router16k_fp4"], "forward") == "mxfp4 x mxfp4 -> f32"
    assert bench.dtype_of(w["decode_fp8"], "decode") == "e4m3fn x f16 -> f32"
    assert bench.dtype_of(w["prefill4k_fp8"], "forward") == "bf16 (from e4m3fn) x bf16 -> f32"
    assert bench.dtype_of(w["decode"], "decode") == "mxfp4 x f16 -> f32"


def test_end_to_end_inputs_keep_every_piece_256_byte_aligned():
    import numpy as np
    for n in (0, 1, 15, 16, 255, 256, 257, 14336, 3584):
        a = np.arange(n, dtype=np.int64).astype(np.uint8)
        p = bench.pad256(a)
        assert len(p) % 256 == 0 and len(p) - n < 256
        assert np.array_equal(p[:n], a) and not p[n:].any()
