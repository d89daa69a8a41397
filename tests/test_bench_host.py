"""The bench's algorithmic work counts, checked on the host against closed forms
for the T = 65536 step (one causal sequence, top-2048, H = 128, 576 / 512
channels, indexer with 64 heads of 128)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_step_flops_match_closed_forms():
    T, k = 65536, 2048
    pairs = T * (T + 1) // 2                      # causal (query, key) pairs, self included
    valid = k * (k + 1) // 2 + (T - k) * k        # sum over t of min(t + 1, k)
    assert valid == sum(min(t + 1, k) for t in range(T))
    f_idx, f_fwd, f_bwd, f_kl, f_ibwd = bench.flops_of(valid, pairs)
    # indexer: one multiply-add per head and channel for every causal pair
    assert f_idx == pairs * 64 * 128 * 2 == 35_184_908_959_744
    # forward: QK^T over 576 channels and PV over 512, per head and valid pair
    assert f_fwd == valid * 128 * 2 * (576 + 512) == 36_799_565_004_800
    # backward: S and dQ, dK over 576; dP and dV over 512
    assert f_bwd == valid * 128 * 2 * (3 * 576 + 2 * 512) == 93_081_252_659_200
    # indexer KL: the student scores of every valid slot (64 heads x 128 channels)
    assert f_kl == valid * 64 * 128 * 2 == 2_164_680_294_400
    # indexer backward: the scores again, dq_I and dk_I
    assert f_ibwd == 3 * f_kl


def test_job_rate_is_ranks_times_work_over_slowest_time():
    assert bench.job_tflops(1, 1e12, 1000.0) == 1.0
    assert bench.job_tflops(8, 2e12, 500.0) == 32.0


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` (the CPU oracle on a bounded row sample of the
    same workload) prints one JSON line with the GPU arm's metric and unit."""
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--ref-rows", "2"], capture_output=True, text=True, timeout=600,
                       env={**os.environ, "RANK": "0", "WORLD_SIZE": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC
    assert line["unit"] == "TFLOP/s" and line["higher_is_better"] is True and line["value"] > 0
    assert line["config"]["workload"] == bench.WORKLOAD
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["value"] == line["value"] and cpu["cores"] >= 1
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
