"""GPU parity of the flat BSA-style comparator (tcgen05, bf16 leaf means)
against the fp64 flat oracle.

The GPU comparator multiplies the queries with the leaf means rounded to
bf16 (unit roundoff 2^-8), so a logit s q.mu moves by up to about
s |q| |mu| 2^-8 ~ 1e-3 relative to the block's probability; block scores
(sums of G probabilities) are therefore compared with a relative tolerance
REL = 5e-3, and a query whose K-th and (K+1)-th oracle scores are closer
than REL relative is tie-exempt: its GPU set must still be a valid Top-K of
the oracle's scores within REL."""
import math

import numpy as np
import pytest
import torch

import oracle
from pyramid_top_block_mean_gb300 import workloads as W

pytestmark = pytest.mark.gpu
REL = 5e-3


@pytest.fixture(scope="module")
def pisa():
    from pyramid_top_block_mean_gb300 import pisa as m
    return m


def flat_scores_np(qrows, mu, qb, s):
    """All block scores of one query (numpy, exact means)."""
    z = (mu[:qb] @ qrows.T) / math.sqrt(mu.shape[1])  # [qb, G]
    z = z - z.max(axis=0)
    p = np.exp(z) / np.exp(z).sum(axis=0)
    return p.sum(axis=1)


def check_flat(s, q, k, idx, score, keys):
    o = oracle.Oracle.from_shape(s)
    qn, kn = q.double().numpy(), k.double().numpy()
    pyr = o.pyramid(kn)
    ref = o.select_flat(qn, pyr, sel=keys)
    bad, exempt = [], 0
    for i, (b, h, t) in enumerate(keys):
        gi, gs = idx[i], score[i]
        ri, rs = ref["idx"][i], ref["score"][i]
        if (gi == ri).all():
            fin = np.isfinite(rs)
            if not (np.isinf(gs) == ~fin).all() or (np.abs(gs[fin] - rs[fin]) > REL * np.abs(rs[fin]) + 1e-7).any():
                bad.append((b, h, t, "score", gs, rs))
            continue
        qb = t // s.C
        kth = rs[np.isfinite(rs)].min() if np.isfinite(rs).any() else 0.0
        if ref["margin"][i] >= REL * kth:
            bad.append((b, h, t, "set", gi, ri))
            continue
        exempt += 1
        mu = pyr[b, h, :-(-s.N // s.C)]
        allsc = flat_scores_np(qn[b, h * s.G:(h + 1) * s.G, t], mu, qb, s)
        F = {0, qb - 1, qb}
        top = [j for j in gi if j >= 0 and j not in F]
        drop = [j for j in range(1, qb - 1) if j not in top]
        if top and drop and min(allsc[top]) < max(allsc[drop]) * (1 - REL):
            bad.append((b, h, t, "invalid top-k", gi, ri))
    assert not bad, bad[:5]
    return exempt


def run_flat(pisa, s, q, k):
    p = pisa.params_from_shape(s)
    sel = pisa.Selector(p, mode="flat")
    sel.flat(q.cuda(), k.cuda())
    torch.cuda.synchronize()
    assert sel.device_status() == 0
    W_ = s.K + 3
    return sel.out_idx.reshape(-1, W_).cpu().numpy(), sel.out_score.reshape(-1, W_).cpu().double().numpy()


# Top-K list paths of the kernel: per-lane register lists (G <= 4, K <= 8;
# G = 4, 1, 2 below), one register list per query (G = 8, K <= 8), lists in
# shared memory (K > 8, with G = 8 and G = 4)
@pytest.mark.parametrize("N,Hq,Hkv,d,K", [(4096, 16, 4, 128, 8), (4096 + 37, 4, 4, 128, 8),
                                          (3000, 8, 1, 64, 32), (2500, 4, 2, 128, 5), (700, 2, 1, 64, 3),
                                          (2048 + 5, 8, 1, 128, 6), (3000, 16, 4, 64, 12)])
def test_flat_matches_oracle(pisa, N, Hq, Hkv, d, K):
    s = W.Shape(B=2, N=N, Hq=Hq, Hkv=Hkv, d=d, K=K)
    q, k = W.iid(s, N % 89)
    idx, score = run_flat(pisa, s, q, k)
    keys = [(b, h, t) for b in range(s.B) for h in range(s.Hkv) for t in range(s.N)]
    ex = check_flat(s, q, k, idx, score, keys)
    assert ex < 0.2 * len(keys)


def test_flat_64k_sampled(pisa):
    s = W.sweep(65536)
    q, k = W.iid(s, 3)
    idx, score = run_flat(pisa, s, q, k)
    gen = np.random.default_rng(1)
    keys = [(0, h, int(t)) for h in range(s.Hkv) for t in gen.integers(0, s.N, 300)]
    rows = [h * s.N + t for (_, h, t) in keys]
    check_flat(s, q, k, idx[rows], score[rows], keys)


def test_flat_rejects_fp32(pisa):
    s = W.Shape(B=1, N=256, Hq=1, Hkv=1, d=64, K=4, dtype="fp32")
    p = pisa.params_from_shape(s)
    sel = pisa.Selector(p, mode="flat")
    q, k = W.iid(s, 0)
    with pytest.raises(pisa.PisaError):
        sel.flat(q.cuda(), k.cuda())
