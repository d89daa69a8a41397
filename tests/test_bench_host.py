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
    f_idx, f_fwd, f_bwd = bench.flops_of(valid, pairs)
    # indexer: one multiply-add per head and channel for every causal pair
    assert f_idx == pairs * 64 * 128 * 2 == 35_184_908_959_744
    # forward: QK^T over 576 channels and PV over 512, per head and valid pair
    assert f_fwd == valid * 128 * 2 * (576 + 512) == 36_799_565_004_800
    # backward: S and dQ, dK over 576; dP and dV over 512
    assert f_bwd == valid * 128 * 2 * (3 * 576 + 2 * 512) == 93_081_252_659_200


def test_job_rate_is_ranks_times_work_over_slowest_time():
    assert bench.job_tflops(1, 1e12, 1000.0) == 1.0
    assert bench.job_tflops(8, 2e12, 500.0) == 32.0
