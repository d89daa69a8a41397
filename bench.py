"""Benchmark of the trainable sparse-attention hot path on GB300.

Workload: long-context absorbed sparse MLA, one sequence of T = 65536 tokens,
H = 128 heads, q/kv bf16 with 576 channels (values = first 512), top-2048,
softmax scale 1/sqrt(192); streaming indexer with 64 heads, d_I = 128,
w ~ U(0,1).  One step = the whole trainable path over one batch:

    qsa_topk (indexer score + exact top-k, streamed)  ->  sparse_mla_fwd
    ->  sparse_mla_bwd (Dlt preprocess, dQ/dKV, dKV conversion, and the
        indexer's teacher: the head mean of P at the selected slots)
    ->  qsa_indexer_kl (student scores at the slots, KL loss, dI = p - a)
    ->  qsa_indexer_bwd (dq_I, dk_I, dw)

value = algorithmic TFLOP/s of the step (indexer GEMM, attention fwd + bwd,
the indexer's KL and backward GEMMs over the selected slots, all counted from
the actual indices) with inputs resident in HBM; per-stage times, indexer
queries/s and roofline fractions are reported alongside.  Inputs (~20 GB)
exceed the 129 MB L2, so no flush is needed between steps.

`secondary.qsa_gqa` times the block Sparse-GQA workload on its own after the
main step (packed THD of four sequences 4096/8192/12288/8192, Hq = 32,
Hkv = 4, d = 128, block 64, top-32 blocks per query and kv group, indexer with
8 heads in 4 groups): block indexer + top-k, GQA forward and backward.  It is
not part of `value`.

`--impl reference` times the CPU oracle on a bounded sample of the same
workload on the host cores (the reference arm: the pages ship no runnable
reference implementation).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

T_TOK = 65536
H = 128
D = 576
DV = 512
TOPK = 2048
# DRAM bytes (read + write) of one forward launch per query, from an ncu capture
# of the current forward kernel on the same workload at T=4096 (scaled by the
# number of queries); None when the kernel changed since the capture.
FWD_TRAFFIC_BYTES_PER_QUERY = 277630  # (0.642460 + 0.494712) GB / 4096 queries; re-captured for each forward kernel change
SCALE = 1.0 / math.sqrt(192)
H_I = 64
D_I = 128
WORKLOAD = "mla_t65536_h128_topk2048"
METRIC = "sparse-attn fwd/bwd + indexer/top-k algorithmic TFLOP/s"  # both arms report this metric


def set_T(t: int):
    """Shrink the sequence (profiling captures only); the workload name says so."""
    global T_TOK, WORKLOAD
    T_TOK = int(t)
    WORKLOAD = f"mla_t{T_TOK}_h128_topk2048"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def flops_of(valid_per_row_total: int, causal_pairs: int):
    """Algorithmic FLOPs: indexer GEMM over causal pairs; attention per valid
    (query, key) pair and head: fwd 2*(576+512), bwd 2*(3*576+2*512); the
    indexer's training per valid pair and indexer head: KL 2*d_I (the student
    scores), backward 3*2*d_I (the scores again, dq_I, dk_I)."""
    f_idx = causal_pairs * H_I * D_I * 2
    f_fwd = valid_per_row_total * H * 2 * (D + DV)
    f_bwd = valid_per_row_total * H * 2 * (3 * D + 2 * DV)
    f_kl = valid_per_row_total * H_I * D_I * 2
    f_ibwd = valid_per_row_total * H_I * D_I * 2 * 3
    return f_idx, f_fwd, f_bwd, f_kl, f_ibwd


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(n_gpus: int, backend: str = "nccl"):
    """Rank, world size and local rank from the torchrun environment; with more
    than one rank, joins the process group (NCCL on GPUs, one rank per GPU;
    gloo for the host-side logic on CPU, where no device is selected)."""
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != n_gpus:
        raise SystemExit(f"--gpus {n_gpus} but WORLD_SIZE={world}: launch one process per GPU with torchrun")
    if world > 1:
        import torch.distributed as dist
        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)
    elif backend == "nccl":
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def allmax(x: float, world) -> float:
    """Maximum of x over the ranks (the timed region of the slowest rank)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world: int, flops_per_rank: float, ms: float) -> float:
    """Whole-job rate: every rank runs the same work on its own replica, and the
    job takes as long as its slowest rank (ms, already the max over ranks)."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


# ---------------------------------------------------------------- oracle timing

def oracle_sample(n_rows: int, seed: int = 123):
    """Run the CPU oracle on n_rows query rows of the workload (indexer + top-k,
    attention fwd and bwd per row) and return (seconds, algorithmic flops)."""
    import numpy as np
    import torch
    import oracle as O
    import synth

    cu = [0, T_TOK]
    rng = np.random.default_rng(seed)
    rows = sorted(rng.choice(T_TOK, size=n_rows, replace=False).tolist())
    # inputs for the sampled rows only (the oracle widens rows lazily); keys/kv in full
    g = synth.gen(seed, "cpu")
    k_idx = synth.randn_bf16((T_TOK, D_I), g, "cpu")
    kv = synth.randn_bf16((T_TOK, D), g, "cpu")
    q_rows = synth.randn_bf16((n_rows, H_I, D_I), g, "cpu")
    w_rows = synth.uniform_f32((n_rows, H_I), g, "cpu")
    q_att = synth.randn_bf16((n_rows, H, D), g, "cpu")
    do_rows = synth.randn_bf16((n_rows, H, DV), g, "cpu")

    class Rows:
        """Row accessor: row t of the full tensor is the i-th sampled row."""
        def __init__(self, data, shape):
            self.data, self.shape, self.pos = data, shape, {t: i for i, t in enumerate(rows)}

        def __getitem__(self, t):
            return self.data[self.pos[t]]

    qI = Rows(q_rows, (T_TOK, H_I, D_I))
    W = Rows(w_rows, (T_TOK, H_I))
    Q = Rows(q_att, (T_TOK, H, D))
    dO = Rows(do_rows, (T_TOK, H, DV))
    t0 = time.perf_counter()
    sc = O.indexer_token_scores(qI, k_idx, W, cu, rows)
    idx_rows = O.topk_rows(sc, TOPK)[:, 0, :]
    I = Rows(torch.from_numpy(idx_rows), (T_TOK, TOPK))
    O.sparse_mla_fwd(Q, kv, I, cu, SCALE, rows=rows)
    O.sparse_mla_bwd(Q, kv, I, cu, SCALE, dO, rows=rows)
    tea = O.mla_teacher(Q, kv, I, cu, SCALE, rows=rows)
    I3 = Rows(torch.from_numpy(idx_rows[:, None, :]), (T_TOK, 1, TOPK))
    sc_sel = O.indexer_scores_at(qI, k_idx, W, cu, I3, rows=rows)[:, 0, :]
    _, dI = O.sparse_kl(sc_sel, tea)
    G3 = Rows(torch.from_numpy(dI[:, None, :]), (T_TOK, 1, TOPK))
    O.indexer_bwd(qI, k_idx, W, cu, I3, G3, rows=rows)
    dt = time.perf_counter() - t0
    valid = int((idx_rows >= 0).sum())
    pairs = sum(t + 1 for t in rows)
    f = sum(flops_of(valid, pairs))
    return dt, f, rows


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    n_rows = args.ref_rows
    times, fl = [], 0.0
    for i in range(args.warmup + args.steps):
        dt, f, _ = oracle_sample(n_rows, seed=1000 + i)
        if i >= args.warmup:
            times.append(dt)
            fl = f
    mean = sum(times) / len(times)
    value = fl / mean / 1e12
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC,
        "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": mean * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "T": T_TOK, "H": H, "d_qk": D, "topk": TOPK, "H_I": H_I, "d_I": D_I,
                   "sample_rows_per_step": n_rows},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n_rows} random query rows of the T=65536 workload per step "
                                   "(indexer+top-k, fwd, bwd, teacher, indexer KL and backward), numpy fp64"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU arm

def run_gpu(args):
    import torch
    import synth
    import trainable_sparse_attention_gb300 as tsa

    rank, world, local = dist_setup(args.gpus)
    tsa.build() if rank == 0 else None
    barrier(world)
    tsa.load_library()
    dev = torch.device("cuda", local)
    cu = [0, T_TOK]
    peaks = load_peaks()

    # inputs resident in HBM (seeded per rank: independent replicas)
    x = synth.indexer_inputs(T_TOK, H_I, D_I, seed=5 + rank, device=dev)
    m = synth.mla_inputs(T_TOK, H, D, seed=7 + rank, device=dev, with_grad_out=True)
    q_i, k_i, w = x["q_idx"], x["k_idx"], x["w"]
    q, kv, dout = m["q"], m["kv"], m["dout"]
    del x, m
    ws_topk = torch.empty(tsa.qsa_topk_workspace_size(cu), dtype=torch.uint8, device=dev)
    ws_bwd = torch.empty(tsa.sparse_mla_bwd_workspace_size(T_TOK, H, D, TOPK), dtype=torch.uint8, device=dev)
    idx = torch.empty((T_TOK, 1, TOPK), dtype=torch.int32, device=dev)
    out = torch.empty((T_TOK, H, DV), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T_TOK, H), dtype=torch.float32, device=dev)
    dq = torch.empty_like(q)
    dkv = torch.empty_like(kv)
    teacher = torch.empty((T_TOK, TOPK), dtype=torch.float32, device=dev)
    loss = torch.empty((T_TOK,), dtype=torch.float32, device=dev)
    dscore = torch.empty((T_TOK, TOPK), dtype=torch.float32, device=dev)
    dq_i, dk_i, dw = torch.empty_like(q_i), torch.empty_like(k_i), torch.empty_like(w)
    ws_ibwd = torch.empty(tsa.qsa_indexer_bwd_workspace_size(T_TOK, D_I), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        i2 = idx.view(T_TOK, TOPK)
        if ev:
            ev[0].record(stream)
        tsa.qsa_topk(q_i, k_i, w, cu, TOPK, workspace=ws_topk, out=idx)
        if ev:
            ev[1].record(stream)
        tsa.sparse_mla_fwd(q, kv, i2, cu, SCALE, out=out, lse=lse)
        if ev:
            ev[2].record(stream)
        tsa.sparse_mla_bwd(q, kv, i2, out, lse, dout, cu, SCALE, workspace=ws_bwd, dq=dq, dkv=dkv, teacher=teacher)
        if ev:
            ev[3].record(stream)
        tsa.qsa_indexer_kl(q_i, k_i, w, cu, i2, teacher, loss=loss, dscore=dscore)
        if ev:
            ev[4].record(stream)
        tsa.qsa_indexer_bwd(q_i, k_i, w, cu, i2, dscore, workspace=ws_ibwd, dq=dq_i, dk=dk_i, dw=dw)
        if ev:
            ev[5].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    valid = int((idx >= 0).sum().item())
    pairs = T_TOK * (T_TOK + 1) // 2
    f_idx, f_fwd, f_bwd, f_kl, f_ibwd = flops_of(valid, pairs)
    f_step = f_idx + f_fwd + f_bwd + f_kl + f_ibwd

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    launches0 = tsa.kernel_launches()
    barrier(world)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    launches = (tsa.kernel_launches() - launches0) // args.steps
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    total_ms = allmax(total_ms, world)
    ms_step = total_ms / args.steps
    st_idx = sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps
    st_fwd = sum(e[1].elapsed_time(e[2]) for e in evs) / args.steps
    st_bwd = sum(e[2].elapsed_time(e[3]) for e in evs) / args.steps
    st_kl = sum(e[3].elapsed_time(e[4]) for e in evs) / args.steps
    st_ibwd = sum(e[4].elapsed_time(e[5]) for e in evs) / args.steps
    value = job_tflops(world, f_step, ms_step)
    psus = peaks["bf16_tflops_sustained"]
    stages = {
        "indexer_topk": {"ms": st_idx, "tflops": f_idx / (st_idx * 1e-3) / 1e12,
                         "queries_per_s": T_TOK / (st_idx * 1e-3),
                         "frac_of_measured_bf16_sustained": f_idx / (st_idx * 1e-3) / 1e12 / psus},
        "mla_fwd": {"ms": st_fwd, "tflops": f_fwd / (st_fwd * 1e-3) / 1e12,
                    "frac_of_measured_bf16_sustained": f_fwd / (st_fwd * 1e-3) / 1e12 / psus},
        "mla_bwd": {"ms": st_bwd, "tflops": f_bwd / (st_bwd * 1e-3) / 1e12,
                    "frac_of_measured_bf16_sustained": f_bwd / (st_bwd * 1e-3) / 1e12 / psus,
                    "note": "includes the indexer teacher (head mean of P, from the dKV GEMM of the 576-channel rows)"},
        "indexer_kl": {"ms": st_kl, "tflops": f_kl / (st_kl * 1e-3) / 1e12,
                       "frac_of_measured_bf16_sustained": f_kl / (st_kl * 1e-3) / 1e12 / psus},
        "indexer_bwd": {"ms": st_ibwd, "tflops": f_ibwd / (st_ibwd * 1e-3) / 1e12,
                        "frac_of_measured_bf16_sustained": f_ibwd / (st_ibwd * 1e-3) / 1e12 / psus,
                        "dk_reduction_gbs": valid * D_I * 4 / (st_ibwd * 1e-3) / 1e9},
    }
    # Roofline of the dominant kernel: the forward is one launch (mla_fwd_tc_kernel)
    # whose stage events bracket exactly that launch, and it is the longest single
    # launch of the step (the backward is five kernels per query chunk).
    achieved = f_fwd / (st_fwd * 1e-3) / 1e12
    roofline = {"bound": "tensor", "kernel": "mla_fwd_tc_kernel", "achieved": achieved, "peak": psus,
                "unit": "TFLOP/s", "frac": achieved / psus,
                "traffic": FWD_TRAFFIC_BYTES_PER_QUERY * T_TOK if FWD_TRAFFIC_BYTES_PER_QUERY else None,
                "traffic_unit": "bytes per launch (DRAM read + write)",
                "peak_source": f"{peaks['source']} bf16 sustained (MEASURED_PEAKS.json)"}

    # end to end through the public API with host buffers (pinned), copies inside the timed region
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, tsa, dev, cu, {"q_idx": q_i, "k_idx": k_i, "w": w, "q": q, "kv": kv, "dout": dout},
                      f_step, world)

    gqa = None if args.no_gqa else run_gqa(args, tsa, dev, world)

    cpu = None
    if rank == 0 and world >= 1 and not args.no_cpu_baseline:
        dt, f, _ = oracle_sample(args.ref_rows)
        cpu = {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{args.ref_rows} random query rows of the same workload (indexer+top-k, fwd, bwd, "
                         f"teacher, indexer KL and backward), numpy fp64, {dt:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value,
            "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "T": T_TOK, "H": H, "d_qk": D, "d_v": DV, "topk": TOPK,
                       "softmax_scale": "1/sqrt(192)", "H_I": H_I, "d_I": D_I, "parallelism": f"replicas{world}",
                       "l2": "inputs (~20 GB) exceed L2; no flush"},
            "stages": stages,
            "indexer_topk_queries_per_s": world * T_TOK / (stages["indexer_topk"]["ms"] * 1e-3),
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": int(launches),
            "clocks": clk,
            "flops_per_step": {"indexer": f_idx, "fwd": f_fwd, "bwd": f_bwd, "indexer_kl": f_kl,
                               "indexer_bwd": f_ibwd, "valid_pairs": valid},
            "secondary": {"qsa_gqa": gqa},
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


GQA_LENGTHS = [4096, 8192, 12288, 8192]  # packed THD of four sequences
GQA_HQ, GQA_HKV, GQA_D, GQA_BS, GQA_NSEL = 32, 4, 128, 64, 32
GQA_HI, GQA_DI = 8, 128


def run_gqa(args, tsa, dev, world):
    """QSA block Sparse-GQA workload, timed on its own after the main step:
    block indexer + exact top-32 blocks per (query, kv group), GQA forward and
    backward.  Algorithmic FLOPs per attended (query, group, token) triple:
    forward 4 d G (QK^T and PV for the G = Hq / Hkv heads of the group),
    backward 10 d G (S recompute, dP, dQ, dK, dV); gathered K + V rows
    2 d bf16 per triple."""
    import torch
    import synth
    lengths = GQA_LENGTHS if args.gqa_lengths is None else [int(v) for v in args.gqa_lengths.split(",")]
    cu = synth.cu_seqlens_thd(lengths)
    T = cu[-1]
    g = synth.gqa_inputs(T, GQA_HQ, GQA_HKV, GQA_D, seed=8, device=dev, with_grad_out=True)
    x = synth.indexer_inputs(T, GQA_HI, GQA_DI, seed=6, device=dev)
    scale = 1.0 / math.sqrt(GQA_D)
    ws = torch.empty(max(1, tsa.qsa_topk_workspace_size(cu, GQA_HKV, GQA_BS)), dtype=torch.uint8, device=dev)
    ws_f = torch.empty(tsa.sparse_gqa_fwd_workspace_size(T, GQA_HQ, GQA_HKV, GQA_D, GQA_NSEL), dtype=torch.uint8,
                       device=dev)
    ws_b = torch.empty(tsa.sparse_gqa_bwd_workspace_size(T, GQA_HQ, GQA_HKV, GQA_D, GQA_NSEL), dtype=torch.uint8,
                       device=dev)
    blk = torch.empty((T, GQA_HKV, GQA_NSEL), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        tsa.qsa_topk(x["q_idx"], x["k_idx"], x["w"], cu, GQA_NSEL, groups=GQA_HKV, block_size=GQA_BS,
                     workspace=ws, out=blk)
        if ev:
            ev[1].record(stream)
        out, lse = tsa.sparse_gqa_fwd(g["q"], g["k"], g["v"], blk, cu, GQA_BS, scale, workspace=ws_f)
        if ev:
            ev[2].record(stream)
        tsa.sparse_gqa_bwd(g["q"], g["k"], g["v"], blk, out, lse, g["dout"], cu, GQA_BS, scale, workspace=ws_b)
        if ev:
            ev[3].record(stream)

    for _ in range(max(3, min(args.warmup, 3))):
        step()
    torch.cuda.synchronize()
    # attended (query, group, token) triples: the causal tokens s <= t of each selected block
    cuT = torch.tensor(cu, device=dev)
    t = torch.arange(T, device=dev)
    p = t - cuT[torch.searchsorted(cuT, t, right=True) - 1]
    b = blk.long()
    ntok = torch.where(b >= 0, torch.clamp(p[:, None, None] - b * GQA_BS + 1, 0, GQA_BS), torch.zeros_like(b))
    triples = int(ntok.sum().item())
    pairs = sum(n * (n + 1) // 2 for n in lengths)
    G = GQA_HQ // GQA_HKV
    f_idx = pairs * GQA_HI * GQA_DI * 2
    f_fwd = triples * 4 * GQA_D * G
    f_bwd = triples * 10 * GQA_D * G
    steps = max(1, min(args.steps, 5))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        step(evs[i])
    torch.cuda.synchronize()
    ms = [sum(e[k].elapsed_time(e[k + 1]) for e in evs) / steps for k in range(3)]
    ms = [allmax(v, world) for v in ms]
    del g, x, ws, ws_f, ws_b, blk
    torch.cuda.empty_cache()
    return {
        "workload": f"qsa_gqa_thd{T}_hq32_hkv4_bs64_top32",
        "lengths": lengths, "Hq": GQA_HQ, "Hkv": GQA_HKV, "d": GQA_D, "block_size": GQA_BS,
        "blocks_selected": GQA_NSEL, "indexer_heads": GQA_HI, "d_I": GQA_DI, "steps": steps,
        "note": "timed separately after the main step; not part of value",
        "block_indexer_topk": {"ms": ms[0], "tflops": job_tflops(world, f_idx, ms[0]),
                               "queries_per_s": world * T / (ms[0] * 1e-3)},
        "gqa_fwd": {"ms": ms[1], "tflops": job_tflops(world, f_fwd, ms[1]),
                    "gather_gbs": world * triples * 2 * GQA_D * 2 / (ms[1] * 1e-3) / 1e9},
        "gqa_bwd": {"ms": ms[2], "tflops": job_tflops(world, f_bwd, ms[2])},
        "attended_triples": triples,
    }


def gpu_local_cpus(local: int):
    """The allowed CPUs that sysfs lists as local to the GPU, or None.  Pinned
    host pages are placed on the NUMA node of the allocating thread, so the
    end-to-end leg allocates them from these CPUs: on a two-socket host, pages
    on the far socket cross the inter-socket link on every copy."""
    try:
        import torch
        p = torch.cuda.get_device_properties(local)
        path = (f"/sys/bus/pci/devices/{p.pci_domain_id:04x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
                "/local_cpulist")
        cpus = set()
        for part in open(path).read().strip().split(","):
            if "-" in part:
                lo, hi = part.split("-")
                cpus.update(range(int(lo), int(hi) + 1))
            elif part:
                cpus.add(int(part))
        cpus &= os.sched_getaffinity(0)
        return sorted(cpus) if cpus else None
    except Exception:
        return None


def run_e2e(args, tsa, dev, cu, dev_inputs, f_step, world):
    """Same step through the public API from pinned host buffers: every step
    copies its inputs host -> device and reads its results device -> host
    inside the timed region.  The copies are pipelined with the compute: the
    inputs of step i+1 are copied (H2D stream, second device buffer set) and
    the results of step i read back (D2H stream) while step i+1 computes.
    Dependencies are per tensor: the inputs are copied in the order the step
    uses them and each call waits only for its own, and each result is read
    back as soon as the call that produces it has finished, so the first
    step's indexer starts after ~1 GB of inputs rather than all 19 GB and the
    last step's results overlap its remaining calls."""
    import torch
    saved_affinity = os.sched_getaffinity(0)
    local_cpus = gpu_local_cpus(dev.index if dev.index is not None else 0)
    if local_cpus:
        os.sched_setaffinity(0, local_cpus)
    host_in = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in dev_inputs.items()}
    for k, v in dev_inputs.items():
        host_in[k].copy_(v)
    outs_shape = {"idx": ((T_TOK, 1, TOPK), torch.int32), "out": ((T_TOK, H, DV), torch.bfloat16),
                  "lse": ((T_TOK, H), torch.float32), "dq": ((T_TOK, H, D), torch.bfloat16),
                  "dkv": ((T_TOK, D), torch.bfloat16), "loss": ((T_TOK,), torch.float32),
                  "dq_i": ((T_TOK, H_I, D_I), torch.bfloat16), "dk_i": ((T_TOK, D_I), torch.bfloat16),
                  "dw": ((T_TOK, H_I), torch.float32)}
    host_out = [{k: torch.empty(s, dtype=d, pin_memory=True) for k, (s, d) in outs_shape.items()} for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out[0].values())
    comp = torch.cuda.current_stream()
    s_in = torch.cuda.Stream()
    s_out = torch.cuda.Stream()
    ws_topk = torch.empty(tsa.qsa_topk_workspace_size(cu), dtype=torch.uint8, device=dev)
    ws_bwd = torch.empty(tsa.sparse_mla_bwd_workspace_size(T_TOK, H, D, TOPK), dtype=torch.uint8, device=dev)
    ws_ibwd = torch.empty(tsa.qsa_indexer_bwd_workspace_size(T_TOK, D_I), dtype=torch.uint8, device=dev)
    d_in = [dict(dev_inputs), {k: torch.empty_like(v, device=dev) for k, v in host_in.items()}]

    order = [k for k in ("q_idx", "k_idx", "w", "q", "kv", "dout") if k in host_in]
    order += [k for k in host_in if k not in order]

    def copy_in(i, after):
        # inputs of step i into buffer set i % 2, once the step that last read it
        # has finished, in the order the step uses them; one event per tensor
        evs = {}
        with torch.cuda.stream(s_in):
            if after is not None:
                s_in.wait_event(after)
            for k in order:
                d_in[i % 2][k].copy_(host_in[k], non_blocking=True)
                evs[k] = torch.cuda.Event()
                evs[k].record(s_in)
        return evs

    def compute(i, ready, out_host):
        x = d_in[i % 2]

        def need(*keys):
            for k in keys:
                comp.wait_event(ready[k])

        def give(**res):
            # each result goes back as soon as the call that made it is done
            ev = torch.cuda.Event()
            ev.record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev)
                for k, t in res.items():
                    out_host[k].copy_(t, non_blocking=True)
                    t.record_stream(s_out)

        need("q_idx", "k_idx", "w")
        idx = tsa.qsa_topk(x["q_idx"], x["k_idx"], x["w"], cu, TOPK, workspace=ws_topk)
        give(idx=idx)
        i2 = idx.view(T_TOK, TOPK)
        need("q", "kv")
        out, lse = tsa.sparse_mla_fwd(x["q"], x["kv"], i2, cu, SCALE)
        give(out=out, lse=lse)
        need("dout")
        dq, dkv, tea = tsa.sparse_mla_bwd(x["q"], x["kv"], i2, out, lse, x["dout"], cu, SCALE, workspace=ws_bwd,
                                          want_teacher=True)
        give(dq=dq, dkv=dkv)
        loss, dscore = tsa.qsa_indexer_kl(x["q_idx"], x["k_idx"], x["w"], cu, i2, tea)
        give(loss=loss)
        dq_i, dk_i, dw = tsa.qsa_indexer_bwd(x["q_idx"], x["k_idx"], x["w"], cu, i2, dscore, workspace=ws_ibwd)
        give(dq_i=dq_i, dk_i=dk_i, dw=dw)
        done = torch.cuda.Event()
        done.record(comp)
        return done

    def run(nsteps, start=None):
        ready = copy_in(0, start)  # the first copy belongs to the timed region
        prev_done = None
        for i in range(nsteps):
            done = compute(i, ready, host_out[i % 2])
            if i + 1 < nsteps:
                ready = copy_in(i + 1, prev_done)  # buffer set (i+1) % 2 was last read by step i-1
            prev_done = done

    run(1)
    torch.cuda.synchronize()
    steps = max(1, min(args.steps, 5))
    barrier(world)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(comp)
    run(steps, a)
    s_out_done = torch.cuda.Event()
    s_out_done.record(s_out)
    comp.wait_event(s_out_done)
    b.record(comp)
    torch.cuda.synchronize()
    ms = allmax(a.elapsed_time(b) / steps, world)
    del d_in, host_in, host_out
    torch.cuda.empty_cache()
    os.sched_setaffinity(0, saved_affinity)
    return {"value": job_tflops(world, f_step, ms), "unit": "TFLOP/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "pipelined": ("per tensor: inputs copied in the order the step uses them, each result read back "
                          "once its call is done; H2D of step i+1 and D2H of step i overlap the compute"),
            "host_cpus": f"{len(local_cpus)} GPU-local CPUs" if local_cpus else "unrestricted (no sysfs locality)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--ref-rows", type=int, default=192, help="oracle rows per CPU sample")
    ap.add_argument("--T", type=int, default=T_TOK, help="sequence length (smaller only for profiling captures)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-gqa", action="store_true", help="skip the separately timed block Sparse-GQA workload")
    ap.add_argument("--gqa-lengths", default=None,
                    help="profiling aid: comma-separated sequence lengths of the GQA workload (default 4096,8192,12288,8192)")
    ap.add_argument("--gqa-only", action="store_true",
                    help="profiling aid: time only the block Sparse-GQA workload and print its object")
    args = ap.parse_args()
    if args.T != T_TOK:
        set_T(args.T)
    if args.impl == "reference":
        return run_reference(args)
    if args.gqa_only:
        import torch
        import trainable_sparse_attention_gb300 as tsa
        tsa.build()
        tsa.load_library()
        print(json.dumps(run_gqa(args, tsa, torch.device("cuda", 0), 1)), flush=True)
        return 0
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
