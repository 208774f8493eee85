"""The benchmark's JSON contract, checked on the CPU: the reference arm (the oracle on the host
cores) prints one line with the contract's keys, and the algorithmic byte counts follow their
definitions."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in rec, key
    assert rec["impl"] == "reference" and rec["n_gpus"] == 1 and rec["steps"] == 1
    assert rec["value"] > 0 and rec["unit"] == "GB/s" and rec["higher_is_better"] is True
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["cores"] >= 1
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["e2e"]["d2h_bytes_per_step"] == 0
    assert "workload" in rec["config"]


def test_algorithmic_byte_counts():
    import bench
    M, K, N, G = 3, 256, 64, 128
    # packed int4 weights, fp16 scales, packed zero points, fp16 x and y
    assert bench.w4a16_bytes(M, K, N, G) == K * N // 2 + (K // G) * N * 2 + (K // G) * N // 2 + 2 * M * K + 2 * M * N
    # int8 weights, fp32 channel scales, int8 codes, fp32 token scales, fp16 y
    assert bench.w8a8_bytes(M, K, N) == N * K + 4 * N + M * K + 4 * M + 2 * M * N
    # fp16 x and gamma in, int8 codes and fp32 scales out; with the residual: r in and h out as well
    assert bench.qrmsnorm_bytes(M, K) == 2 * M * K + 2 * K + M * K + 4 * M
    assert bench.add_qrmsnorm_bytes(M, K) == bench.qrmsnorm_bytes(M, K) + 4 * M * K
    assert bench.gemm_flops(M, K, N) == 2 * M * K * N


def test_phase_trace_summary_on_synthetic_stamps():
    # Six launches of four CTAs of the decode kernel, 10 us apart.  Launch l resolves its
    # dependency at 10 l + 1 us; its CTAs end at 10 l + 3.5, 3.6, 3.7 and 4 us, so the flush
    # (dependency resolution after the preceding launch's last CTA end) is 7 us.  Phase k of CTA c
    # is stamped 0.1 k + 0.02 c us after the dependency; slot 31 holds the SM id.
    import numpy as np
    import bench
    L, C = 6, 4
    t = np.zeros((L, C, 32), dtype=np.int64)
    names = bench.TRACE_PHASES[0]
    end = bench.TRACE_END[0]
    dep = names.index("dependency resolved")
    for l in range(L):
        for c in range(C):
            base = 10_000 * l + 1_000
            for k in range(len(names)):
                t[l, c, k] = base + 100 * k + 20 * c
            t[l, c, dep] = base
            t[l, c, 0] = base - 500 + 20 * c  # start, before the dependency resolves
            t[l, c, end] = 10_000 * l + [3_500, 3_600, 3_700, 4_000][c]
            t[l, c, 31] = 7 + c
    out = bench.trace_summary(t, 0)
    assert out["ctas_per_launch"] == C and out["distinct_sms"] == C
    assert out["launch_period_us"] == 10.0
    assert out["flush_us"] == 7.0
    ph = out["phases_us_from_dependency"]
    assert ph["dependency resolved"] == [0.0, 0.0, 0.0]
    assert ph["start"] == [-0.47, -0.5, -0.44]
    k = names.index("lanes folded")
    assert ph["lanes folded"] == [round(0.1 * k + 0.03, 2), round(0.1 * k, 2), round(0.1 * k + 0.06, 2)]
    assert ph["end"] == [2.65, 2.5, 3.0]
