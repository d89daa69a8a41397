"""Host-side logic of the N-rank bench on CPU: world_size-2 gloo ranks run the
same rank plumbing that torchrun ranks run on GPUs (process group, barrier,
max over ranks of the timed region, whole-job rate, rank-0-only output of the
reference arm).  No GPU and no kernel is involved."""
import argparse
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, outdir: str, times_ms):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import torch.distributed as dist
    r, w, local = bench.dist_setup(world, backend="gloo")
    bench.barrier(w)
    ms = bench.allmax(times_ms[r], w)
    rate = bench.job_tflops(w, 1e12, ms)
    bench.barrier(w)
    dist.destroy_process_group()
    with open(os.path.join(outdir, f"rank{r}.json"), "w") as f:
        json.dump({"rank": r, "world": w, "local": local, "ms": ms, "rate": rate}, f)


def test_two_gloo_ranks_take_the_slowest_rank(tmp_path):
    """Each rank reports its own time; both see the maximum, and the job rate is
    (ranks x work per rank) / slowest time."""
    world, times = 2, [40.0, 50.0]
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path), times), nprocs=world,
                       join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    assert [x["rank"] for x in res] == [0, 1] and all(x["world"] == 2 for x in res)
    assert all(x["ms"] == 50.0 for x in res)
    # 2 ranks x 1e12 flops in 50 ms = 40 TFLOP/s
    assert all(x["rate"] == pytest.approx(40.0) for x in res)


def test_single_rank_needs_no_process_group(monkeypatch):
    for k in ("RANK", "LOCAL_RANK", "WORLD_SIZE"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_setup(1, backend="gloo") == (0, 1, 0)
    assert bench.allmax(3.25, 1) == 3.25
    assert bench.job_tflops(1, 2e12, 1000.0) == pytest.approx(2.0)


def test_world_size_must_match_gpus(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "0")
    with pytest.raises(SystemExit):
        bench.dist_setup(1, backend="gloo")


def test_reference_arm_prints_on_rank_zero_only(monkeypatch):
    """Under torchrun the CPU reference arm runs on rank 0 alone; other ranks
    exit 0 at once without touching the oracle."""
    monkeypatch.setenv("RANK", "1")
    args = argparse.Namespace(gpus=2, steps=1, warmup=1, ref_rows=1)
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.run_reference(args) == 0
    assert buf.getvalue() == ""
