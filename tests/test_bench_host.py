"""Host-side logic of bench.py (no GPU): the max-over-ranks timing and the
whole-job rate with two gloo ranks, the algorithmic work counts, and the
clock-sample parsing."""
import math
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from pyramid_top_block_mean_gb300 import workloads as W


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    t = [0.25, 0.5][rank]  # rank 1 is the slower one
    tmax = bench.reduce_max(t, ws)
    bench.barrier(ws)
    rate = bench.whole_job_rate(1000, ws, tmax)
    out[rank] = (tmax, rate)
    dist.destroy_process_group()


def test_two_rank_max_time_and_weak_scaling_rate():
    ws = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(ws, port, out), nprocs=ws, join=True)
    assert out[0] == out[1] == (0.5, 4000.0)


def test_single_rank_is_identity():
    assert bench.reduce_max(1.5, 1) == 1.5
    assert bench.whole_job_rate(10, 1, 2.0) == 5.0


def test_algorithmic_leaf_count_matches_brute_force():
    s = W.Shape(B=1, N=64 * 40 + 5, Hq=4, Hkv=2, d=16, K=3)
    rng = np.random.default_rng(0)
    kept2 = rng.integers(-1, 25, size=(s.B * s.Hkv * s.N * s.K,)).astype(np.int32)
    work = bench.algorithmic_work(s, kept2)
    n = 0
    kp = kept2.reshape(s.B * s.Hkv, s.N, s.K)
    for bh in range(s.B * s.Hkv):
        for t in range(s.N):
            qb = t // s.C
            for p in kp[bh, t]:
                if p < 0:
                    continue
                n += sum(1 <= leaf <= qb - 2 for leaf in (2 * p, 2 * p + 1))
    assert work["leaf_candidates"] == n
    assert work["leaf_flops"] == 2.0 * s.d * s.G * s.C * n
    assert work["bytes"] > 0 and work["route_flops"] > 0


def test_clock_sampler_parses_reasons():
    cs = bench.ClockSampler(0)
    cs.proc = type("P", (), {"terminate": lambda self: None, "wait": lambda self, timeout=None: 0,
                             "kill": lambda self: None})()
    cs.lines = ["0, 1800, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Active",
                "0, 1900, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active",
                "garbage"]
    r = cs.stop()
    assert r["sm_mhz"] == 1850 and r["sm_max_mhz"] == 2070 and r["reasons"] == ["sw_power_cap"]


def test_attention_work_counts_attended_keys_by_brute_force():
    s = W.Shape(B=1, N=64 * 9 + 21, Hq=8, Hkv=2, d=16, K=3)
    g = torch.Generator().manual_seed(2)
    idx = torch.randint(-2, 12, (s.B, s.Hkv, s.N, s.K + 3), generator=g, dtype=torch.int32)
    flops, bytes_, n_keys = bench.attention_work(s, idx)
    n = 0
    for h in range(s.Hkv):
        for t in range(s.N):
            for j in idx[0, h, t].tolist():
                n += sum(1 for i in range(j * s.C, (j + 1) * s.C) if 0 <= j and i <= t)
    assert n_keys == n
    assert flops == 4.0 * s.d * n * s.G
    assert bytes_ == 2 * (s.Hq * s.N * s.d * 2) + 2 * (s.Hkv * s.N * s.d * 2) + idx.numel() * 4
