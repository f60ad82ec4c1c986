"""Host-side logic of bench.py across ranks, on CPU with gloo (world size 2).

Each rank draws its own problem of the same shape (weak scaling, no collective
on the data path); the reported time is the maximum over ranks.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, lr, ws = bench.dist_env()
        times = [3.5, 1.25]
        mx = bench.max_over_ranks(times[rank], ws)
        bench.barrier(ws)
        out[rank] = (r, lr, ws, mx, bench.rank_seed(1001, r))
    finally:
        dist.destroy_process_group()


def test_two_ranks_max_time_and_distinct_problems():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    assert [res[r][:3] for r in range(world)] == [(0, 0, 2), (1, 1, 2)]
    assert res[0][3] == res[1][3] == 3.5          # max over ranks
    assert res[0][4] != res[1][4]                 # independent problems per rank


def test_single_rank_defaults(monkeypatch):
    for k in ("RANK", "LOCAL_RANK", "WORLD_SIZE"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 0, 1)
    assert bench.max_over_ranks(2.5, 1) == 2.5


def test_visible_rows_match_flop_count():
    from exact_attention_forward_sm_gb300 import workloads as wl
    for case in (wl.make_case(2, 3, 1, 300, 300, 64, "bf16", True, seed=1),
                 wl.make_case(0, 2, 2, 0, 0, 64, "fp16", True, seed=2,
                              seqlens_q=[5, 130, 64], seqlens_k=[9, 130, 70]),
                 wl.make_case(1, 4, 4, 100, 50, 128, "bf16", False, seed=3),
                 wl.make_case(2, 2, 2, 90, 300, 64, "bf16", False, seed=4, window=(17, 5)),
                 wl.make_case(0, 2, 1, 0, 0, 64, "fp16", True, seed=5, window=(40, -1),
                              seqlens_q=[70, 1, 200], seqlens_k=[30, 9, 260])):
        vis = bench._visible_per_row(case)
        assert vis.shape[0] == case.lse_rows()
        assert 4 * case.D * int(vis.sum()) == wl.attention_flops(case)


def test_backward_workloads_and_oracle_sample():
    """Every forward workload with head dim 64 / 128 has a backward twin, and
    the backward CPU baseline times the oracle's gradients on a sub-problem
    (batch 0, every head, a prefix of the positions) with 2.5x its forward
    FLOPs."""
    from exact_attention_forward_sm_gb300 import workloads as wl
    names = {w.name for w in wl.WORKLOADS if w.D in (64, 128)}
    assert {n[len(bench.BWD_PREFIX):] for n in bench.BWD_WORKLOADS} == names
    case = wl.make_case(2, 4, 2, 300, 300, 64, "fp16", True, seed=3)
    dout = torch.randn(tuple(case.q.shape)).to(case.q.dtype)
    r = bench.oracle_sample_bwd(case, dout, seconds=0.05)
    sp = r["rows"] // case.Hq
    assert 1 <= sp <= 300 and r["rows_total"] == 2 * 4 * 300
    assert r["flops"] == 2.5 * 4.0 * 64 * 4 * sp * (sp + 1) / 2
    assert r["tflops"] > 0 and r["threads"] >= 1


def test_reference_arm_prints_one_json_line():
    """`bench.py --impl reference` times the oracle on bounded samples of the
    default workload and prints one JSON line: the shared keys, impl,
    cpu_baseline and an end-to-end object with no host-device copies."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "3", "--reference-budget-s", "2"],
                       cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["config"]["workload"] == "b4_h16_s2048_d128_bf16_causal"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
