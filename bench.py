"""Benchmark of the pyramid Top-K block selector on one GB300 (or N replicas).

Default workload: the long-prefill point of the sweep, 262144 tokens, B = 1,
16 query / 4 key heads, d = 128, bf16, C = 64, g = 2, K = 8, iid N(0, 1)
inputs.  One step = pyramid build + routing + leaf LSE + Top-K for every
query position (the whole prefill selector).  Inputs (1.3 GB) are larger
than L2, so no flush is needed between steps.

Prints one JSON line.  value = whole-job queries/s (query positions selected
per second, summed over ranks).  `--impl reference` times the fp64 CPU
oracle (the only reference this method has) on the host cores instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "PISA selection ms and queries/s at 64K/128K/256K; % of HBM/tensor roofline"
UNIT = "queries/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["pisa", "reference"], default="pisa")
    ap.add_argument("--N", type=int, default=262144)
    ap.add_argument("--no-extras", action="store_true", help="skip the sweep, flat and decode side measurements")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--profile-case", choices=["prefill64k", "decode8", "attend256k"], default=None,
                    help="run one small invocation of every kernel (for ncu captures) and exit")
    ap.add_argument("--configs", action="store_true",
                    help="time every listed workload (GPU and CPU oracle), one JSON line each, and exit")
    return ap.parse_args()


# ------------------------------------------------------------------ ranks
def dist_setup(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = os.environ.get("PISA_BENCH_BACKEND", "nccl")
        if backend == "nccl":
            import torch
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return ws, rank, local


def reduce_max(x: float, ws: int) -> float:
    """Max of a float over ranks (identity for one rank)."""
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def whole_job_rate(units_per_rank: float, ws: int, seconds_max: float) -> float:
    """Weak scaling: every rank processes its own batch of `units_per_rank`."""
    return units_per_rank * ws / seconds_max


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------- workloads
def workload(N: int, rank: int):
    from pyramid_top_block_mean_gb300 import workloads as W
    s = W.sweep(N)
    q, k = W.iid(s, 3 + 1000 * rank)
    return s, q, k


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d.get("bf16_tflops_sustained"),
                    sm_max_mhz=d.get("sm_max_mhz", 2070.0), source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, sm_max_mhz=2070.0, source="fallback")


def eligible_count(level, qb):
    if qb - 2 < 1:
        return 0
    if level == 1:
        return qb - 2
    return ((qb - 2) >> (level - 1)) + 1


def algorithmic_work(s, kept2):
    """Algorithmic work of one prefill step.  Leaf flops are exact, from the
    routing output: 2 d G C per eligible (query, leaf) candidate.  Routing
    flops are 2 d G per child summary scored, with at most 2 eligible
    children for each of at most 2K candidates per level below the start
    level.  Bytes: q and k read once, the fp32 pyramid written and read
    once, and the K + 3 outputs written."""
    import numpy as np
    K, C, d, G = s.K, s.C, s.d, s.G
    t = np.arange(s.N)
    qb = t // C
    kp = kept2.reshape(-1, s.N, K)  # [B*Hkv, N, K]
    p = kp.astype(np.int64)
    valid = p >= 0
    leaf0, leaf1 = 2 * p, 2 * p + 1
    e_hi = (qb - 2)[None, :, None]
    ncand = ((valid & (leaf0 >= 1) & (leaf0 <= e_hi)).sum() + (valid & (leaf1 >= 1) & (leaf1 <= e_hi)).sum())
    leaf_flops = 2.0 * d * G * C * float(ncand)
    # routing: child dot products of the walk; every scored level has at most
    # 2K candidates with at most 2 eligible children each
    nb = -(-s.N // C)
    L = 1
    n = nb
    while n > 1:
        n = -(-n // 2)
        L += 1
    dots = 0
    for qbv in range(nb):
        l0 = 0
        for level in range(L, 1, -1):
            if eligible_count(level, qbv) > K:
                l0 = level
                break
        if l0 == 0:
            continue
        per = eligible_count(l0 - 1, qbv) + sum(min(4 * K, 2 * eligible_count(lv - 1, qbv)) for lv in range(l0 - 1, 1, -1))
        nq = min(C, s.N - qbv * C)
        dots += per * nq
    route_flops = 2.0 * d * G * dots * s.B * s.Hkv
    P = 0
    n = nb
    while True:
        P += n
        if n == 1:
            break
        n = -(-n // 2)
    bytes_ = (s.B * s.Hq * s.N * d * 2 + s.B * s.Hkv * s.N * d * 2 + 2 * s.B * s.Hkv * P * d * 4
              + s.B * s.Hkv * s.N * (K + 3) * 8)
    q_bytes = s.B * s.Hq * s.N * d * 2
    k_bytes = s.B * s.Hkv * s.N * d * 2
    pyr_bytes = s.B * s.Hkv * P * d * 4
    kept_bytes = s.B * s.Hkv * s.N * K * 4
    out_bytes = s.B * s.Hkv * s.N * (K + 3) * 8
    return dict(leaf_candidates=int(ncand), leaf_flops=leaf_flops, route_flops=route_flops, bytes=bytes_,
                pyramid_bytes=k_bytes + pyr_bytes,
                # route: q read once, the pyramid read once, the kept level-2 nodes written
                route_bytes=q_bytes + pyr_bytes + kept_bytes,
                # leaves: q and k read once, the kept nodes read, the outputs written
                leaf_bytes=q_bytes + k_bytes + kept_bytes + out_bytes)


ROUTE_KERNEL = "route_haar_kernel"


def load_traffic(name):
    """dram bytes per launch of a kernel, from the committed ncu summary."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        return json.load(open(path)).get(name)
    except (OSError, ValueError):
        return None


def run_config(s, ws):
    """The `config` object of both arms' JSON lines (identical by design)."""
    return {"workload": f"prefill selection, B={s.B} N={s.N} Hq={s.Hq} Hkv={s.Hkv} d={s.d} C={s.C} "
                        f"g=2 K={s.K} bf16 (build + route + leaf LSE + Top-K)",
            "B": s.B, "N": s.N, "H_q": s.Hq, "H_kv": s.Hkv, "d": s.d, "C": s.C, "K": s.K,
            "l2": "inputs (1.3 GB at N=262144) larger than L2; no flush", "parallelism": f"replicas x{ws}"}


def stage_rooflines(s, work, stage_ms, pk):
    """Roofline of each prefill stage and of the whole selector, from the
    algorithmic work of one step (algorithmic_work) and the measured stage
    times.  Each stage's roofline time is the slower of its algorithmic bytes
    at the measured HBM copy bandwidth and its algorithmic flops at the
    measured bf16 burst peak (the step lasts milliseconds); `bound` names the
    slower term, `achieved` is that term's work divided by the stage time and
    frac = achieved / peak = roofline time / stage time."""
    def one(kernel, bytes_, flops, ms, traffic_name):
        t_hbm = bytes_ / (pk["hbm"] * 1e9) * 1e3
        t_tc = flops / (pk["bf16"] * 1e12) * 1e3
        if t_hbm >= t_tc:
            r = {"bound": "hbm", "achieved": bytes_ / (ms * 1e-3) / 1e9, "peak": pk["hbm"], "unit": "GB/s",
                 "peak_source": f"{pk['source']} HBM copy"}
        else:
            r = {"bound": "tensor", "achieved": flops / (ms * 1e-3) / 1e12, "peak": pk["bf16"], "unit": "TFLOP/s",
                 "peak_source": f"{pk['source']} bf16 burst"}
        r.update({"kernel": kernel, "frac": r["achieved"] / r["peak"], "t_roof_ms": max(t_hbm, t_tc),
                  "t_hbm_ms": t_hbm, "t_tensor_ms": t_tc, "measured_ms": ms, "algorithmic_bytes": bytes_,
                  "algorithmic_flops": flops,
                  "traffic": load_traffic(traffic_name) if traffic_name else None})
        return r
    out = {
        "build": one("build_lower_kernel + build_upper_smem_kernel", work["pyramid_bytes"], 0.0, stage_ms["build"],
                     "build_lower_kernel"),
        "route": one("route stage (pyramid split + routing kernel)", work["route_bytes"], work["route_flops"],
                     stage_ms["route"], ROUTE_KERNEL),
        "leaves": one("leaf stage (bucketing + leaf_tc_kernel + finalize)", work["leaf_bytes"], work["leaf_flops"],
                      stage_ms["leaves"], "leaf_tc_kernel"),
    }
    t_roof = max(work["bytes"] / (pk["hbm"] * 1e9), (work["leaf_flops"] + work["route_flops"]) /
                 (pk["bf16"] * 1e12)) * 1e3
    out["selector"] = {"t_roof_ms": t_roof}
    return out


# ------------------------------------------------------------- GPU arm
def run_pisa(args, ws, rank, local):
    import numpy as np
    import torch
    from pyramid_top_block_mean_gb300 import pisa

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    s, q_h, k_h = workload(args.N, rank)
    q_h = q_h.pin_memory()
    k_h = k_h.pin_memory()
    p = pisa.params_from_shape(s)
    sel = pisa.Selector(p, device=dev)
    q = q_h.to(dev, non_blocking=True)
    k = k_h.to(dev, non_blocking=True)
    st = torch.cuda.current_stream(dev)
    torch.cuda.synchronize(dev)

    def step():
        pisa.build_pyramid(p, k, sel.pyramid, None, st)
        pisa.prefill_route(p, q, sel.pyramid, sel.ws, None, st)
        pisa.prefill_leaves(p, q, k, sel.ws, sel.out_idx, sel.out_score, st)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    assert sel.device_status(st) == 0

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(ws)
    torch.cuda.synchronize(dev)
    t_all0 = torch.cuda.Event(enable_timing=True)
    t_all1 = torch.cuda.Event(enable_timing=True)
    launches0 = pisa.kernel_launches()
    t_all0.record(st)
    for i in range(args.steps):
        e = ev[i]
        e[0].record(st)
        pisa.build_pyramid(p, k, sel.pyramid, None, st)
        e[1].record(st)
        pisa.prefill_route(p, q, sel.pyramid, sel.ws, None, st)
        e[2].record(st)
        pisa.prefill_leaves(p, q, k, sel.ws, sel.out_idx, sel.out_score, st)
        e[3].record(st)
    t_all1.record(st)
    launches = pisa.kernel_launches() - launches0
    torch.cuda.synchronize(dev)
    barrier(ws)
    clk = clocks.stop()
    total_ms = t_all0.elapsed_time(t_all1)
    ms_step = total_ms / args.steps
    stage = {nm: statistics.mean(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(args.steps))
             for j, nm in enumerate(["build", "route", "leaves"])}
    ms_max = reduce_max(ms_step, ws)
    value = whole_job_rate(s.B * s.N, ws, ms_max / 1e3)

    # algorithmic work of this input (outside the timed region)
    kept2 = sel.ws[256:256 + s.B * s.Hkv * s.N * s.K * 4].view(torch.int32).cpu().numpy()
    work = algorithmic_work(s, kept2)
    pk = peaks()
    rl = stage_rooflines(s, work, stage, pk)
    t_roof_ms = rl["selector"]["t_roof_ms"]
    roof = rl[max(stage, key=stage.get)]

    # end to end through the public API with host buffers: every step copies
    # its q and k from pinned host memory and reads its indices back.  Steps
    # are pipelined over two buffer sets: the copy of step i+1's inputs and
    # the read-back of step i-1's indices overlap the selection of step i.
    del sel
    torch.cuda.empty_cache()
    sels = [pisa.Selector(p, device=dev) for _ in range(2)]
    qs = [q, torch.empty_like(q)]
    ks = [k, torch.empty_like(k)]
    out_h = [torch.empty(sels[0].out_idx.shape, dtype=torch.int32).pin_memory() for _ in range(2)]
    cs_in = torch.cuda.Stream(dev)
    cs_out = torch.cuda.Stream(dev)
    # the pipeline's first copy and last selection are not overlapped; 16 steps
    # keep that share small so the number reflects the steady state
    e2e_steps = max(8, min(2 * args.steps, 16))

    def e2e_run(n):
        ready = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]
        read = [torch.cuda.Event() for _ in range(2)]
        e_start = torch.cuda.Event(enable_timing=True)
        e_end = torch.cuda.Event(enable_timing=True)
        e_start.record(st)
        cs_in.wait_event(e_start)
        with torch.cuda.stream(cs_in):
            qs[0].copy_(q_h, non_blocking=True)
            ks[0].copy_(k_h, non_blocking=True)
        ready[0].record(cs_in)
        for i in range(n):
            b = i % 2
            if i + 1 < n:
                nb_ = (i + 1) % 2
                if i >= 1:
                    cs_in.wait_event(done[nb_])  # step i-1 has finished reading buffer nb_
                with torch.cuda.stream(cs_in):
                    qs[nb_].copy_(q_h, non_blocking=True)
                    ks[nb_].copy_(k_h, non_blocking=True)
                ready[nb_].record(cs_in)
            st.wait_event(ready[b])
            if i >= 2:
                st.wait_event(read[b])  # step i-2's indices have left selector b
            sels[b].prefill(qs[b], ks[b], stream=st)
            done[b].record(st)
            cs_out.wait_event(done[b])
            with torch.cuda.stream(cs_out):
                out_h[b].copy_(sels[b].out_idx, non_blocking=True)
            read[b].record(cs_out)
        st.wait_stream(cs_out)
        e_end.record(st)
        torch.cuda.synchronize(dev)
        return e_start.elapsed_time(e_end) / n

    e2e_run(2)
    barrier(ws)
    e2e_ms = reduce_max(e2e_run(e2e_steps), ws)
    e2e = {"value": whole_job_rate(s.B * s.N, ws, e2e_ms / 1e3), "unit": UNIT, "ms_per_step": e2e_ms,
           "h2d_bytes_per_step": q_h.numel() * 2 + k_h.numel() * 2,
           "d2h_bytes_per_step": out_h[0].numel() * 4, "steps": e2e_steps,
           "how": "pisa_select_prefill (build + select) per step; H2D of q, k from pinned memory and D2H of "
                  "the indices on two copy streams, double-buffered so they overlap the neighbouring steps"}
    del sels, qs, ks
    torch.cuda.empty_cache()

    extras = {}
    if not args.no_extras:
        extras = side_measurements(args, dev, st, rank)

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded iid N(0,1) q and k)",
            "config": run_config(s, ws),
            "stage_ms": stage, "selector_roofline": {
                "t_roof_ms": t_roof_ms, "frac": t_roof_ms / ms_max, "bytes": work["bytes"],
                "flops": work["leaf_flops"] + work["route_flops"], "leaf_candidates": work["leaf_candidates"],
                "rule": "max(bytes / HBM, flops / bf16 tensor burst peak), measured peaks"},
            "stage_rooflines": {k_: v for k_, v in rl.items() if k_ != "selector"},
            "roofline": roof, "e2e": e2e, "gpu_launches": launches, "clocks": clk}
    line.update(extras)
    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(s, q_h, k_h, budget_s=15.0)
    return line


def attention_work(s, idx):
    """Algorithmic work of attention over a selection: 4 d flops per (query
    head, attended key) (the q.k dot and the p v update); bytes = q, k, v and
    the output read or written once, plus the index rows.  Attended keys
    come from the selection: 64 per listed block before the query's own
    block, t mod 64 + 1 in its own block."""
    import torch
    t = torch.arange(s.N, device=idx.device)
    qb = (t // s.C).view(1, 1, -1, 1)
    own = (t % s.C + 1).view(1, 1, -1, 1)
    keys = torch.where((idx < 0) | (idx > qb), torch.zeros_like(idx),
                       torch.where(idx < qb, torch.full_like(idx, s.C), own))
    n_keys = int(keys.sum().item())  # per (sequence, key head, position): the G heads share it
    flops = 4.0 * s.d * n_keys * s.G
    bytes_ = (s.B * s.Hq * s.N * s.d * 2) * 2 + 2 * (s.B * s.Hkv * s.N * s.d * 2) + idx.numel() * 4
    return flops, bytes_, n_keys


def attention_measurements(dev, st, tm):
    """Block-sparse attention over the PISA selection at 64K-256K tokens
    (pisa_attend_prefill), the selection + attention total, and PyTorch's
    dense causal scaled_dot_product_attention (the full attention it
    replaces) on the same q, k, v; each timed with CUDA events."""
    import torch
    from pyramid_top_block_mean_gb300 import pisa
    from pyramid_top_block_mean_gb300 import workloads as W

    pk = peaks()
    res = {}
    for N in (65536, 131072, 262144):
        s = W.sweep(N)
        g = torch.Generator(device=dev)
        g.manual_seed(11 + N)
        q = torch.randn(s.B, s.Hq, s.N, s.d, device=dev, generator=g).to(torch.bfloat16)
        k = torch.randn(s.B, s.Hkv, s.N, s.d, device=dev, generator=g).to(torch.bfloat16)
        v = torch.randn(s.B, s.Hkv, s.N, s.d, device=dev, generator=g).to(torch.bfloat16)
        p = pisa.params_from_shape(s)
        sel = pisa.Selector(p, device=dev, with_scores=False)
        at = pisa.Attention(p, device=dev)
        with torch.cuda.stream(st):
            idx, _ = sel.prefill(q, k, stream=st)
        torch.cuda.synchronize(dev)
        t_at = tm(lambda: at(q, k, v, idx, stream=st), 5)
        t_both = tm(lambda: (sel.prefill(q, k, stream=st), at(q, k, v, idx, stream=st)), 5)
        flops, bytes_, n_keys = attention_work(s, idx)
        kk = k.repeat_interleave(s.G, 1)
        vv = v.repeat_interleave(s.G, 1)

        def dense():
            with torch.cuda.stream(st):
                torch.nn.functional.scaled_dot_product_attention(q, kk, vv, is_causal=True)
        t_dense = tm(dense, 2)
        t_roof = max(bytes_ / (pk["hbm"] * 1e9), flops / (pk["bf16"] * 1e12)) * 1e3
        res[str(N)] = {"attend_ms": t_at, "select_plus_attend_ms": t_both, "dense_sdpa_ms": t_dense,
                       "dense_over_sparse": t_dense / t_both, "attended_keys_per_query": n_keys / (s.B * s.Hkv * s.N),
                       "roofline": {"t_roof_ms": t_roof, "frac": t_roof / t_at, "flops": flops, "bytes": bytes_,
                                    "bound": "tensor" if flops / pk["bf16"] / 1e12 >
                                    bytes_ / pk["hbm"] / 1e9 else "hbm",
                                    "partial_bytes": 2 * s.B * s.Hq * s.N * (s.K + 3) * (s.d * 2 + 4)}}
        del q, k, v, kk, vv, sel, at, idx
        torch.cuda.empty_cache()
    res["workload"] = ("B=1, Hq=16 Hkv=4 d=128 K=8 bf16; v iid N(0,1); dense = torch SDPA causal "
                       "(flash) with k, v repeated over the GQA group")
    return res


def side_measurements(args, dev, st, rank):
    """Sweep points, the flat comparator and the decode step (not the
    headline; each timed with CUDA events after warm-up)."""
    import torch
    from pyramid_top_block_mean_gb300 import pisa
    from pyramid_top_block_mean_gb300 import workloads as W

    def tm(fn, reps):
        for _ in range(2):
            fn()
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(st)
        for _ in range(reps):
            fn()
        b.record(st)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / reps

    sweep = {}
    attention = attention_measurements(dev, st, tm)
    for N in (65536, 131072, 262144):
        s = W.sweep(N)
        g = torch.Generator(device=dev)
        g.manual_seed(3 + N)
        q = torch.randn(s.B, s.Hq, s.N, s.d, device=dev, generator=g).to(torch.bfloat16)
        k = torch.randn(s.B, s.Hkv, s.N, s.d, device=dev, generator=g).to(torch.bfloat16)
        p = pisa.params_from_shape(s)
        sel = pisa.Selector(p, device=dev)
        fs = pisa.Selector(p, device=dev, mode="flat")
        t_pisa = tm(lambda: sel.prefill(q, k, stream=st), 5)
        t_flat = tm(lambda: fs.flat(q, k, stream=st), 3)
        pp = pisa.params_from_shape(s, summaries=pisa.SUMMARIES_PREFIX)
        ps = pisa.Selector(pp, device=dev)
        t_prefix = tm(lambda: ps.prefill(q, k, stream=st), 5)
        sweep[str(N)] = {"pisa_ms": t_pisa, "pisa_queries_per_s": N / t_pisa * 1e3, "flat_ms": t_flat,
                         "pisa_over_flat_speedup": t_flat / t_pisa,
                         "pisa_prefix_summaries_ms": t_prefix}
        del q, k, sel, fs, ps
    torch.cuda.empty_cache()
    # decode: 64 sequences x 131072 cached keys, 32/8 heads, K = 32
    s = W.DECODE
    g = torch.Generator(device=dev)
    g.manual_seed(4)
    kc = torch.randn(s.B, s.Hkv, s.N, s.d, device=dev, generator=g, dtype=torch.bfloat16)
    qd = torch.randn(W.DECODE_STEPS, s.B, s.Hq, s.d, device=dev, generator=g, dtype=torch.bfloat16)
    p = pisa.params_from_shape(s)
    ds = pisa.Selector(p, device=dev, mode="decode")
    ds.build(kc, torch.full((s.B,), W.DECODE_CACHED, dtype=torch.int32, device=dev))
    lens = [torch.full((s.B,), W.DECODE_CACHED + 1 + i, dtype=torch.int32, device=dev)
            for i in range(W.DECODE_STEPS)]
    # warm-up: the first step twice (its in-place update is idempotent)
    for _ in range(2):
        ds.decode(qd[0], kc, lens[0], stream=st)
    torch.cuda.synchronize(dev)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(st)
    for i in range(W.DECODE_STEPS):
        ds.decode(qd[i], kc, lens[i], stream=st)
    b.record(st)
    torch.cuda.synchronize(dev)
    us = a.elapsed_time(b) / W.DECODE_STEPS * 1e3
    leaf_bytes = s.B * s.Hkv * 2 * s.K * s.C * s.d * 2
    # child summary rows the walk reads (fp32): all children of the start
    # level's candidates, then one child per candidate below it
    qb = (W.DECODE_CACHED + W.DECODE_STEPS // 2) // s.C
    rows = 0
    nb = qb + 1
    L = 1
    while nb > 1:
        nb = -(-nb // 2)
        L += 1
    l0 = next((lv for lv in range(L, 1, -1) if eligible_count(lv, qb) > s.K), 0)
    if l0:
        rows = 2 * eligible_count(l0, qb) + sum(min(2 * s.K, eligible_count(lv, qb)) for lv in range(l0 - 1, 1, -1))
    walk_bytes = s.B * s.Hkv * rows * s.d * 4
    step_bytes = leaf_bytes + walk_bytes + s.B * s.Hq * s.d * 2
    pk = peaks()
    # attention of the same decode steps over their selections (values iid N(0,1))
    vc = torch.randn(s.B, s.Hkv, s.N, s.d, device=dev, generator=g, dtype=torch.bfloat16)
    at = pisa.Attention(p, device=dev, mode="decode")
    idx_steps = []
    ds.build(kc, torch.full((s.B,), W.DECODE_CACHED, dtype=torch.int32, device=dev))
    for i in range(W.DECODE_STEPS):
        ds.decode(qd[i], kc, lens[i], stream=st)
        idx_steps.append(ds.out_idx.clone())
    torch.cuda.synchronize(dev)
    for _ in range(2):
        at.decode(qd[0], kc, vc, lens[0], idx_steps[0], stream=st)
    torch.cuda.synchronize(dev)
    a.record(st)
    for i in range(W.DECODE_STEPS):
        at.decode(qd[i], kc, vc, lens[i], idx_steps[i], stream=st)
    b.record(st)
    torch.cuda.synchronize(dev)
    at_us = a.elapsed_time(b) / W.DECODE_STEPS * 1e3
    # keys read: 64 per listed block before the query's own block, t mod 64 + 1 in it
    n_keys = 0
    for i in range(W.DECODE_STEPS):
        t_ = W.DECODE_CACHED + i
        ids = idx_steps[i]
        qb_ = t_ // s.C
        n_keys += int(((ids >= 0) & (ids < qb_)).sum().item()) * s.C + int((ids == qb_).sum().item()) * (t_ % s.C + 1)
    at_bytes = n_keys / W.DECODE_STEPS * s.d * 2 * 2 + 2 * s.B * s.Hq * s.d * 2
    attn = {"us_per_step": at_us, "selection_plus_attention_us": us + at_us,
            "roofline": {"bound": "hbm", "bytes_per_step": at_bytes, "achieved": at_bytes / (at_us * 1e-6) / 1e9,
                         "peak": pk["hbm"], "unit": "GB/s", "frac": at_bytes / (at_us * 1e-6) / 1e9 / pk["hbm"],
                         "bytes": "keys and values of the attended positions, q and the output"}}
    del kc, vc, at
    torch.cuda.empty_cache()
    return {"sweep": sweep, "attention": attention, "decode": {"us_per_step": us, "steps": W.DECODE_STEPS,
                                       "workload": "B=64, 131072 cached keys, Hq=32 Hkv=8 d=128 bf16 K=32",
                                       "leaf_key_bytes_per_step": leaf_bytes,
                                       "leaf_key_GBps": leaf_bytes / (us * 1e-6) / 1e9,
                                       "roofline": {"bound": "hbm", "bytes_per_step": step_bytes,
                                                    "achieved": step_bytes / (us * 1e-6) / 1e9,
                                                    "peak": pk["hbm"], "unit": "GB/s",
                                                    "frac": step_bytes / (us * 1e-6) / 1e9 / pk["hbm"],
                                                    "bytes": "leaf keys + walked child rows (fp32) + q"},
                                       "attention": attn}}


# ----------------------------------------------------------- CPU oracle
ORACLE_CHUNK = 64  # queries per OpenMP work item in the oracle's selection loop


def oracle_sample(s, q_h, nblocks, offset=0):
    """Every (query position, key head) pair of `nblocks` evenly spaced leaf
    blocks (counted from the last block), as one selection batch: the sel
    triples and the matching [n, G, d] fp64 head rows."""
    import numpy as np
    import torch
    nb = -(-s.N // s.C)
    stride = max(1, nb // max(1, nblocks))
    blocks = [blk for blk in range(nb - 1 - offset, -1, -stride)][:nblocks]
    ts = np.concatenate([np.arange(blk * s.C, min((blk + 1) * s.C, s.N)) for blk in blocks])
    hs = np.repeat(np.arange(s.Hkv), len(ts))
    tt = np.tile(ts, s.Hkv)
    sel = np.stack([np.zeros_like(hs), hs, tt], axis=1)
    qv = q_h[0].reshape(s.Hkv, s.G, s.N, s.d)
    rows = qv[torch.from_numpy(hs), :, torch.from_numpy(tt)].double().numpy()
    return sel, rows, len(blocks)


def oracle_rate(s, q_h, k_h, budget_s, threads=None, kn=None, pyr=None, t_pyr=None):
    """The fp64 oracle as it stands on `threads` host threads (all when None):
    the fp64 pyramid of all keys, then selection batches of whole leaf blocks
    (all key heads) until about `budget_s` seconds of selection work.  Every
    batch holds at least ORACLE_CHUNK pairs per thread, so every thread
    works.  Returns the throughput that implies for the whole workload
    (pyramid once, plus the measured cost per (query, key head) pair for all
    B N Hkv pairs) and what was timed."""
    import oracle
    o = oracle.Oracle.from_shape(s)
    prev = oracle.num_threads()
    if threads:
        oracle.set_num_threads(threads)
    try:
        nthr = oracle.num_threads()
        if kn is None:
            kn = k_h.double().numpy()
        if pyr is None:
            t0 = time.perf_counter()
            pyr = o.pyramid(kn)  # the oracle builds its pyramid on one thread
            t_pyr = time.perf_counter() - t0
        pyr_ = pyr
        # blocks per batch: >= ORACLE_CHUNK pairs per thread (a block gives C * Hkv pairs)
        per_batch = max(1, -(-ORACLE_CHUNK * nthr // (s.C * s.Hkv)))
        t_sel, n_sel, n_blocks, calls = 0.0, 0, 0, 0
        while t_sel < budget_s and n_blocks < -(-s.N // s.C):
            sel, rows, nbk = oracle_sample(s, q_h, per_batch, offset=calls)
            t0 = time.perf_counter()
            o.select(rows, kn, pyr_, sel=sel, qrows=True)
            t_sel += time.perf_counter() - t0
            n_sel += len(sel)
            n_blocks += nbk
            calls += 1
        per_pair = t_sel / n_sel
        total = t_pyr + per_pair * s.B * s.N * s.Hkv
        busy = min(nthr, -(-n_sel // calls // ORACLE_CHUNK))
        return dict(value=s.B * s.N / total, t_pyr=t_pyr, t_sel=t_sel, n_sel=n_sel, n_blocks=n_blocks,
                    calls=calls, threads=nthr, busy_threads=busy, per_pair_us=per_pair * 1e6,
                    kn=kn, pyr=pyr_)
    finally:
        oracle.set_num_threads(prev)


def cpu_baseline(s, q_h, k_h, budget_s=15.0, one_core_budget_s=6.0):
    """The fp64 oracle as it stands, on all host cores and on one core (see
    oracle_rate); `value` is the all-core figure."""
    import platform
    r = oracle_rate(s, q_h, k_h, budget_s)
    r1 = oracle_rate(s, q_h, k_h, one_core_budget_s, threads=1, kn=r["kn"], pyr=r["pyr"], t_pyr=r["t_pyr"])
    return {"value": r["value"], "unit": UNIT, "cores": r["busy_threads"], "kind": "oracle",
            "sample": f"fp64 pyramid of all {s.N} keys ({r['t_pyr']:.1f} s) + the selections of every "
                      f"(query, key head) pair of {r['n_blocks']} evenly spaced leaf blocks ({r['n_sel']} pairs, "
                      f"{r['t_sel']:.1f} s, {r['calls']} batches of >= {ORACLE_CHUNK} pairs per thread); "
                      f"value = B N / (pyramid s + s per pair x B N Hkv)",
            "per_pair_us": r["per_pair_us"], "threads": r["threads"],
            "one_core": {"value": r1["value"], "unit": UNIT, "cores": 1, "per_pair_us": r1["per_pair_us"],
                         "sample": f"{r1['n_sel']} pairs of {r1['n_blocks']} leaf blocks ({r1['t_sel']:.1f} s) "
                                   f"on one thread, plus the same single-threaded pyramid"},
            "host": f"{platform.machine()}, {os.cpu_count()} cpus",
            "seconds_measured": r["t_pyr"] + r["t_sel"] + r1["t_pyr"] + r1["t_sel"]}


def run_reference(args, ws, rank):
    """--impl reference: the fp64 CPU oracle on this config (rank 0 only).
    One step is real and timed as a whole: the fp64 pyramid of all keys plus
    the selections of a fixed sample of whole leaf blocks (all key heads),
    in one batch that keeps every thread busy.  ms_per_step is that measured
    step; value is the whole-workload throughput the step's own timings
    imply (pyramid once, plus its cost per pair for all B N Hkv pairs)."""
    if rank != 0:
        return None
    s, q_h, k_h = workload(args.N, 0)
    import oracle
    o = oracle.Oracle.from_shape(s)
    kn = k_h.double().numpy()
    nthr = oracle.num_threads()
    nblocks = max(1, -(-16 * ORACLE_CHUNK * nthr // (s.C * s.Hkv)))
    sel, rows, nbk = oracle_sample(s, q_h, nblocks)

    def step():
        t0 = time.perf_counter()
        pyr = o.pyramid(kn)
        t1 = time.perf_counter()
        o.select(rows, kn, pyr, sel=sel, qrows=True)
        t2 = time.perf_counter()
        return t2 - t0, (t1 - t0) + (t2 - t1) / len(sel) * s.B * s.N * s.Hkv

    for _ in range(args.warmup):
        step()
    meas = [step() for _ in range(args.steps)]
    step_s = statistics.mean(m[0] for m in meas)
    work_s = statistics.mean(m[1] for m in meas)
    val = s.B * s.N / work_s
    cfg = run_config(s, ws)
    return {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded iid N(0,1) q and k)",
            "config": cfg,
            "cpu_baseline": {"kind": "oracle", "cores": min(nthr, -(-len(sel) // ORACLE_CHUNK)), "value": val,
                             "unit": UNIT,
                             "sample": f"per step (timed whole, {step_s:.2f} s): fp64 pyramid of all {s.N} keys + "
                                       f"the selections of all {len(sel)} (query, key head) pairs of {nbk} evenly "
                                       f"spaced leaf blocks in one batch; value = B N / (pyramid s + s per pair x "
                                       f"{s.B * s.N * s.Hkv} pairs)"},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def profile_case(name: str):
    """One small invocation per kernel, sized for profiler captures: the 64K
    prefill point (build, route, leaves, flat, attention over the selection;
    inputs 400 MB > L2), one decode step of 8 sequences x 131073 keys (2.1 GB
    cache each for keys and values, with the attention over the selection),
    or the 256K selection followed by two attention calls (for the
    attention's launch list; 15 GB on the device, one-pass metrics only)."""
    import torch
    from pyramid_top_block_mean_gb300 import pisa
    from pyramid_top_block_mean_gb300 import workloads as W
    g = torch.Generator(device="cuda")
    if name == "prefill64k":
        s = W.sweep(65536)
        g.manual_seed(3)
        q = torch.randn(s.B, s.Hq, s.N, s.d, device="cuda", generator=g).to(torch.bfloat16)
        k = torch.randn(s.B, s.Hkv, s.N, s.d, device="cuda", generator=g).to(torch.bfloat16)
        p = pisa.params_from_shape(s)
        sel = pisa.Selector(p)
        sel.build(k)
        pisa.prefill_route(p, q, sel.pyramid, sel.ws)
        pisa.prefill_leaves(p, q, k, sel.ws, sel.out_idx, sel.out_score)
        fs = pisa.Selector(p, mode="flat")
        fs.build(k)
        pisa.select_flat(p, q, fs.pyramid, fs.ws, fs.out_idx, fs.out_score)
        v = torch.randn(s.B, s.Hkv, s.N, s.d, device="cuda", generator=g).to(torch.bfloat16)
        at = pisa.Attention(p)
        at(q, k, v, sel.out_idx)
        torch.cuda.synchronize()
        status = max(sel.device_status(), fs.device_status(), at.device_status())
    elif name == "attend256k":
        s = W.sweep(262144)
        g.manual_seed(11 + s.N)
        q = torch.randn(s.B, s.Hq, s.N, s.d, device="cuda", generator=g).to(torch.bfloat16)
        k = torch.randn(s.B, s.Hkv, s.N, s.d, device="cuda", generator=g).to(torch.bfloat16)
        v = torch.randn(s.B, s.Hkv, s.N, s.d, device="cuda", generator=g).to(torch.bfloat16)
        p = pisa.params_from_shape(s)
        sel = pisa.Selector(p, with_scores=False)
        idx, _ = sel.prefill(q, k)
        at = pisa.Attention(p)
        for _ in range(2):
            at(q, k, v, idx)
        torch.cuda.synchronize()
        status = max(sel.device_status(), at.device_status())
    else:
        s = W.Shape(B=8, N=W.DECODE_CACHED + 16, Hq=32, Hkv=8, d=128, K=32)
        g.manual_seed(4)
        kc = torch.randn(s.B, s.Hkv, s.N, s.d, device="cuda", generator=g, dtype=torch.bfloat16)
        qd = torch.randn(s.B, s.Hq, s.d, device="cuda", generator=g, dtype=torch.bfloat16)
        p = pisa.params_from_shape(s)
        ds = pisa.Selector(p, mode="decode")
        ds.build(kc, torch.full((s.B,), W.DECODE_CACHED, dtype=torch.int32, device="cuda"))
        ln = torch.full((s.B,), W.DECODE_CACHED + 1, dtype=torch.int32, device="cuda")
        ds.decode(qd, kc, ln)
        vc = torch.randn(s.B, s.Hkv, s.N, s.d, device="cuda", generator=g, dtype=torch.bfloat16)
        at = pisa.Attention(p, mode="decode")
        at.decode(qd, kc, vc, ln, ds.out_idx)
        torch.cuda.synchronize()
        status = max(ds.device_status(), at.device_status())
    print(json.dumps({"profile_case": name, "device_status": status}))
    if status != 0:
        sys.exit(1)


def _cuda_ms(fn, reps, st):
    import torch
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(st)
    for _ in range(reps):
        fn()
    b.record(st)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def configs_table():
    """Every listed workload: GPU prefill (build + select) and flat-comparator
    times with CUDA events, the CPU oracle on the host cores (in full where it
    takes seconds, else the sampled estimate of cpu_baseline), and the decode
    step.  Side table, not the headline line."""
    import time as _t
    import numpy as np
    import torch
    import oracle
    from pyramid_top_block_mean_gb300 import pisa
    from pyramid_top_block_mean_gb300 import workloads as W
    st = torch.cuda.current_stream()
    rows = []

    def prefill_row(name, s, q, k, cpu_full):
        p = pisa.params_from_shape(s)
        sel = pisa.Selector(p)
        qd, kd = q.cuda(), k.cuda()
        reps = 20 if s.N <= 65536 else 5
        t_pisa = _cuda_ms(lambda: sel.prefill(qd, kd, stream=st), reps, st)
        kept2 = sel.ws[256:256 + s.B * s.Hkv * s.N * s.K * 4].view(torch.int32).cpu().numpy()
        work = algorithmic_work(s, kept2)
        pk = peaks()
        t_roof = max(work["bytes"] / (pk["hbm"] * 1e9), (work["leaf_flops"] + work["route_flops"]) /
                     (pk["bf16"] * 1e12)) * 1e3
        roof = {"t_roof_ms": t_roof, "frac": t_roof / t_pisa, "bytes": work["bytes"],
                "flops": work["leaf_flops"] + work["route_flops"],
                "bound": "tensor" if t_roof > work["bytes"] / (pk["hbm"] * 1e9) * 1e3 else "hbm",
                "rule": "max(bytes / HBM copy, flops / bf16 burst), measured peaks; time = build + select"}
        t_flat = None
        if s.dtype == "bf16":
            fs = pisa.Selector(p, mode="flat")
            t_flat = _cuda_ms(lambda: fs.flat(qd, kd, stream=st), max(2, reps // 4), st)
            del fs
        del sel, qd, kd
        torch.cuda.empty_cache()
        if cpu_full:
            o = oracle.Oracle.from_shape(s)
            t0 = _t.perf_counter()
            pyr = o.pyramid(k.double().numpy())
            o.select(q.double().numpy(), k.double().numpy(), pyr)
            cpu_ms, cpu_how = (_t.perf_counter() - t0) * 1e3, "full"
        else:
            cb = oracle_rate(s, q, k, 5.0)
            cpu_ms = s.B * s.N / cb["value"] * 1e3
            cpu_how = (f"sampled: fp64 pyramid ({cb['t_pyr']:.1f} s) + {cb['n_sel']} (query, key head) pairs of "
                       f"{cb['n_blocks']} leaf blocks ({cb['t_sel']:.1f} s), {cb['busy_threads']} threads busy; "
                       f"ms = pyramid + per-pair cost x all pairs")
        rows.append({"config": name, "N": s.N, "K": s.K, "dtype": s.dtype, "pisa_ms": t_pisa,
                     "pisa_queries_per_s": s.B * s.N / t_pisa * 1e3, "roofline": roof, "flat_ms": t_flat,
                     "pisa_over_flat": (t_flat / t_pisa) if t_flat else None,
                     "cpu_oracle_ms": cpu_ms, "cpu_cores": (oracle.num_threads() if cpu_full else cb["busy_threads"]),
                     "cpu_how": cpu_how})
        print(json.dumps(rows[-1]), flush=True)

    q, k = W.iid(W.TINY, 0)
    prefill_row("tiny B=1 N=1024 H=1/1 d=64 fp32 K=4", W.TINY, q, k, True)
    q, k = W.planted(W.PRETRAIN, 1)
    prefill_row("pretrain B=2 N=4096 16/4 d=128 bf16 K=8 planted", W.PRETRAIN, q, k, True)
    q, k, _ = W.needles(W.CPT, 2)
    prefill_row("CPT B=1 N=16384 16/4 d=128 bf16 K=32 needles", W.CPT, q, k, True)
    for N in W.SWEEP_NS:
        s = W.sweep(N)
        q, k = W.iid(s, 3)
        prefill_row(f"sweep B=1 N={N} 16/4 d=128 bf16 K=8", s, q, k, N <= 16384)
        del q, k
    # decode: GPU step on the full workload; the oracle on one sequence, times 64
    s = W.DECODE
    g = torch.Generator(device="cuda")
    g.manual_seed(4)
    kc = torch.randn(s.B, s.Hkv, s.N, s.d, device="cuda", generator=g, dtype=torch.bfloat16)
    qd = torch.randn(W.DECODE_STEPS, s.B, s.Hq, s.d, device="cuda", generator=g, dtype=torch.bfloat16)
    p = pisa.params_from_shape(s)
    ds = pisa.Selector(p, mode="decode")
    ds.build(kc, torch.full((s.B,), W.DECODE_CACHED, dtype=torch.int32, device="cuda"))
    lens = [torch.full((s.B,), W.DECODE_CACHED + 1 + i, dtype=torch.int32, device="cuda")
            for i in range(W.DECODE_STEPS)]
    for _ in range(2):  # warm-up: the first step twice (its in-place update is idempotent)
        ds.decode(qd[0], kc, lens[0], stream=st)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(st)
    for i in range(W.DECODE_STEPS):
        ds.decode(qd[i], kc, lens[i], stream=st)
    b.record(st)
    torch.cuda.synchronize()
    us = a.elapsed_time(b) / W.DECODE_STEPS * 1e3
    del kc, ds
    torch.cuda.empty_cache()
    s1 = W.Shape(B=1, N=s.N, Hq=s.Hq, Hkv=s.Hkv, d=s.d, K=s.K)
    q1, k1 = W.decode_inputs(s1, 4, steps=1)
    o = oracle.Oracle.from_shape(s1)
    kn = k1.double().numpy()
    lens1 = [W.DECODE_CACHED + 1]
    t0 = _t.perf_counter()
    pyr = o.pyramid(kn, lens1)
    t1 = _t.perf_counter()
    o.select(q1[0].double().numpy(), kn, pyr, seq_lens=lens1, decode=True)
    t2 = _t.perf_counter()
    rows.append({"config": "decode B=64 x 131072 cached, 32/8 d=128 bf16 K=32", "pisa_us_per_step": us,
                 "cpu_oracle_ms_per_step": (t2 - t1) * 64 * 1e3,
                 "cpu_how": f"oracle select of one sequence (8 key heads: one OpenMP work item, so one "
                            f"thread) x 64; its fp64 pyramid rebuild ({(t1 - t0) * 1e3:.0f} ms per sequence) "
                            f"not included",
                 "cpu_cores": 1})
    print(json.dumps(rows[-1]), flush=True)


def main():
    args = parse()
    if args.profile_case:
        profile_case(args.profile_case)
        return
    if args.configs:
        configs_table()
        return
    ws, rank, local = dist_setup(args)
    if args.impl == "reference":
        line = run_reference(args, ws, rank)
    else:
        line = run_pisa(args, ws, rank, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
