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
