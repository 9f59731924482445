"""GPU parity of the prefill path (pyramid build, routing, leaf LSE, Top-K)
against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from pyramid_top_block_mean_gb300 import workloads as W

from parity import Report, compare

pytestmark = pytest.mark.gpu

U = 2.0 ** -24  # fp32 unit roundoff


@pytest.fixture(scope="module")
def pisa():
    from pyramid_top_block_mean_gb300 import pisa as m
    return m


def run_prefill(pisa, s, q, k, trace=True):
    p = pisa.params_from_shape(s)
    sel = pisa.Selector(p)
    tr = None
    if trace:
        L = pisa.pyramid_levels(p)
        tr = torch.full((s.B, s.Hkv, s.N, L, s.K), -7, dtype=torch.int32, device="cuda")
    sel.prefill(q.cuda(), k.cuda(), trace=tr)
    torch.cuda.synchronize()
    assert sel.device_status() == 0
    W_ = s.K + 3
    return dict(pyr=sel.pyramid.cpu().double().numpy(),
                idx=sel.out_idx.reshape(-1, W_).cpu().numpy(),
                score=sel.out_score.reshape(-1, W_).cpu().double().numpy(),
                trace=None if tr is None else tr.reshape(s.B * s.Hkv * s.N, -1, s.K).cpu().numpy())


def full_parity(pisa, s, q, k):
    g = run_prefill(pisa, s, q, k)
    o = oracle.Oracle.from_shape(s)
    qn, kn = q.double().numpy(), k.double().numpy()
    pyr = o.pyramid(kn)
    ref = o.select(qn, kn, pyr)
    keys = [(b, h, t) for b in range(s.B) for h in range(s.Hkv) for t in range(s.N)]
    rep = compare(o, qn, kn, pyr, ref, g["idx"], g["score"], g["trace"], keys, Report())
    print(rep)
    assert rep.ok(), str(rep)
    return g, pyr, rep


def pyramid_tolerance(s, k):
    # leaf: sequential fp32 sum of C values then a division; each level adds
    # one rounded add and one rounded division (|error| <= 2u |value|).
    L = oracle.Oracle.from_shape(s).num_levels
    return (s.C + 2 * L + 2) * U * float(np.abs(k).max())


@pytest.mark.parametrize("N,d,dtype,G", [(1024, 64, "fp32", 1), (4096 + 37, 128, "bf16", 4),
                                         (3000, 64, "bf16", 2), (64 * 33 + 1, 128, "fp32", 8),
                                         (63, 128, "bf16", 4), (1, 64, "bf16", 1)])
def test_pyramid_matches_direct_means(pisa, N, d, dtype, G):
    s = W.Shape(B=2, N=N, Hq=2 * G, Hkv=2, d=d, K=4, dtype=dtype)
    q, k = W.iid(s, 5)
    p = pisa.params_from_shape(s)
    sel = pisa.Selector(p)
    sel.build(k.cuda())
    torch.cuda.synchronize()
    got = sel.pyramid.cpu().double().numpy()
    want = oracle.Oracle.from_shape(s).pyramid(k)
    kn = k.double().numpy()
    err = np.abs(got - want).max()
    assert err <= pyramid_tolerance(s, kn), err


def test_pyramid_long_sequence_matches_direct_means(pisa):
    """524,325 keys (ragged), d = 128: levels 5 and 6 exceed the shared-memory
    budget of the upper build, so the levels above 5 take the path through
    L2; every node against the oracle's direct means."""
    s = W.Shape(B=1, N=(1 << 19) + 37, Hq=1, Hkv=1, d=128, K=4, dtype="bf16")
    q, k = W.iid(s, 7)
    p = pisa.params_from_shape(s)
    sel = pisa.Selector(p)
    sel.build(k.cuda())
    torch.cuda.synchronize()
    got = sel.pyramid.cpu().double().numpy()
    want = oracle.Oracle.from_shape(s).pyramid(k)
    err = np.abs(got - want).max()
    assert err <= pyramid_tolerance(s, k.double().numpy()), err


def test_tiny_fp32_K4(pisa):
    s = W.TINY
    q, k = W.iid(s, 0)
    full_parity(pisa, s, q, k)


def test_tiny_fp32_K8_is_exhaustive(pisa):
    s = W.Shape(**{**W.TINY.__dict__, "K": 8})
    q, k = W.iid(s, 0)
    full_parity(pisa, s, q, k)


def test_pretrain_planted_bf16(pisa):
    s = W.PRETRAIN
    q, k = W.planted(s, 1)
    g, _, rep = full_parity(pisa, s, q, k)
    assert rep.exempt < 0.2 * rep.n


@pytest.mark.parametrize("N,Hq,Hkv,d,K,dtype", [
    (4096 + 37, 16, 4, 128, 8, "bf16"),   # ragged tail
    (2048 + 1, 8, 1, 64, 5, "bf16"),      # G = 8, d = 64
    (3333, 4, 2, 128, 3, "fp32"),         # G = 2, fp32 leaves on the CUDA cores
    (64 * 3 + 5, 4, 4, 128, 8, "bf16"),   # a few leaves only
    (5000, 2, 2, 64, 32, "bf16"),         # K = 32
    (3000, 8, 2, 64, 8, "bf16"),          # tensor-core routing with d = 64
    (2500, 8, 2, 128, 1, "bf16"),         # K = 1
    (2600, 16, 4, 128, 2, "bf16"),        # K = 2
    (2700, 16, 4, 128, 16, "bf16"),       # K = 16 on the tensor-core path
])
def test_prefill_shapes(pisa, N, Hq, Hkv, d, K, dtype):
    s = W.Shape(B=2, N=N, Hq=Hq, Hkv=Hkv, d=d, K=K, dtype=dtype)
    q, k = W.iid(s, N % 97)
    full_parity(pisa, s, q, k)


def test_cpt_needles_sampled(pisa):
    """N = 16384, K = 32, planted needle blocks; all queries of the last 3
    leaf blocks plus 3000 random positions per key head are checked, and
    every needle block must be selected by the last query."""
    s = W.CPT
    q, k, blocks = W.needles(s, 2)
    g = run_prefill(pisa, s, q, k)
    gen = np.random.default_rng(0)
    keys = []
    for h in range(s.Hkv):
        ts = set(range(s.N - 3 * 64, s.N)) | set(gen.integers(0, s.N, 3000).tolist())
        keys += [(0, h, t) for t in sorted(ts)]
    rows = [h * s.N + t for (_, h, t) in keys]
    o = oracle.Oracle.from_shape(s)
    qn, kn = q.double().numpy(), k.double().numpy()
    pyr = o.pyramid(kn)
    ref = o.select(qn, kn, pyr, sel=keys)
    rep = compare(o, qn, kn, pyr, ref, g["idx"][rows], g["score"][rows], g["trace"][rows], keys, Report())
    print(rep)
    assert rep.ok(), str(rep)
    for h in range(s.Hkv):
        last = g["idx"][h * s.N + s.N - 1]
        assert set(blocks[h]) <= set(last.tolist())


@pytest.mark.parametrize("N,Hq,Hkv,dtype", [
    (1, 4, 1, "bf16"),      # one query, only block 0
    (64, 8, 2, "bf16"),     # one full leaf block
    (65, 4, 1, "bf16"),     # the first query of block 1 forces blocks 0 and 1
    (191, 8, 2, "bf16"),    # block 2 is the last with no eligible block (E = [1, qb - 2] empty)
    (193, 4, 1, "fp32"),    # block 3: one eligible leaf
    (257, 16, 4, "bf16"),   # tensor-core routing path with a handful of leaves
])
def test_prefill_shortest_sequences(pisa, N, Hq, Hkv, dtype):
    """Sequences too short for any scored level: the output is the forced
    blocks plus the few eligible leaves, -1 padded."""
    s = W.Shape(B=2, N=N, Hq=Hq, Hkv=Hkv, d=128, K=4, dtype=dtype)
    q, k = W.iid(s, 11 + N)
    g, _, _ = full_parity(pisa, s, q, k)
    first = g["idx"][0]
    assert first[0] == 0 and (first[1:] == -1).all()


def test_prefill_262144_sampled(pisa):
    """The 262144-token long-prefill workload in the launch configuration the
    benchmark times (build, then the route and leaf stages): every query of
    the last two leaf blocks and 1500 random positions per key head against
    the oracle, which builds its own fp64 pyramid of all keys."""
    s = W.sweep(262144)
    q, k = W.iid(s, 3)
    p = pisa.params_from_shape(s)
    sel = pisa.Selector(p)
    L = pisa.pyramid_levels(p)
    qd, kd = q.cuda(), k.cuda()
    tr = torch.full((s.B, s.Hkv, s.N, L, s.K), -7, dtype=torch.int32, device="cuda")
    pisa.build_pyramid(p, kd, sel.pyramid)
    pisa.prefill_route(p, qd, sel.pyramid, sel.ws, tr)
    pisa.prefill_leaves(p, qd, kd, sel.ws, sel.out_idx, sel.out_score)
    torch.cuda.synchronize()
    assert sel.device_status() == 0
    gen = np.random.default_rng(5)
    keys = []
    for h in range(s.Hkv):
        ts = set(range(s.N - 2 * 64, s.N)) | set(gen.integers(0, s.N, 1500).tolist())
        keys += [(0, h, t) for t in sorted(ts)]
    rows = torch.tensor([h * s.N + t for (_, h, t) in keys], device="cuda")
    W_ = s.K + 3
    idx = sel.out_idx.reshape(-1, W_)[rows].cpu().numpy()
    score = sel.out_score.reshape(-1, W_)[rows].cpu().double().numpy()
    trace = tr.reshape(s.B * s.Hkv * s.N, L, s.K)[rows].cpu().numpy()
    del tr
    o = oracle.Oracle.from_shape(s)
    kn = k.double().numpy()
    pyr = o.pyramid(kn)
    qsel = np.stack([q[0, h * s.G:(h + 1) * s.G, t].double().numpy() for (_, h, t) in keys])
    ref = o.select(qsel, kn, pyr, sel=keys, qrows=True)
    rep = compare(o, qsel, kn, pyr, ref, idx, score, trace, keys, Report(), qmode="rows")
    print(rep)
    assert rep.ok(), str(rep)


@pytest.mark.parametrize("dtype,Hq,Hkv", [("bf16", 8, 2), ("fp32", 4, 2)])
def test_prefill_nonfinite_keys_stay_well_formed(pisa, dtype, Hq, Hkv):
    """Keys holding NaN and +-inf (whole leaf blocks and single entries):
    every ranking treats a NaN score as -inf, so each query still gets its
    forced blocks plus exactly min(K, |E|) causal blocks, ascending and -1
    padded, and the device status stays clear."""
    from parity import check_structure
    s = W.Shape(B=1, N=64 * 40 + 9, Hq=Hq, Hkv=Hkv, d=128, K=4, dtype=dtype)
    q, k = W.iid(s, 21)
    k = k.float()
    k[0, 0, 64 * 5:64 * 6] = float("nan")
    k[0, 0, 64 * 11 + 3, 7] = float("inf")
    k[0, Hkv - 1, 64 * 17:64 * 18, :4] = -float("inf")
    k[0, Hkv - 1, 64 * 23 + 1] = float("nan")
    k = k.to(s.torch_dtype)
    g = run_prefill(pisa, s, q, k, trace=False)
    rep = Report()
    for h in range(s.Hkv):
        for t in range(s.N):
            row = h * s.N + t
            ok = check_structure(g["idx"][row], None, t, s.C, s.K, rep, f"(h={h},t={t})")
            assert ok, rep.failures
