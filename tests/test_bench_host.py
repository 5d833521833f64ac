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
    src = os.path.join(bench.ROOT, "mxfp4_routed_expert_03_gb300", "csrc", "grouped_gemm.cu")
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    lines = [l.split() for l in open(os.path.join(bench.ROOT, "profiles", "traffic.txt"))
             if l.strip() and not l.startswith("#")]
    for name, h, wl, nbytes in lines:
        got = bench.kernel_traffic(name, "grouped_gemm.cu", wl)
        assert got == (float(nbytes) if h == sha else None)
    assert bench.kernel_traffic("moe_grouped_gemm_kernel<0>", "grouped_gemm.cu", "no-such") is None
