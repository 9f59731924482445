"""Pins of the oracle's PISA-1 and PISA-2 block scorers (agihunt.info summary,
LSE paragraph: PISA-1 keeps only the mean, PISA-2 adds the variance term of
the LSE Taylor expansion; rcap.io post, "The scoring rule matters":
truncations at first and second order).  CPU only.

The scorers replace LSE(x) = log n + log mean exp(x_i) over the same summands
(child-summary dots above the leaves, raw-key dots at the leaves) by
log n + mean(x) (PISA-1) and log n + mean(x) + var(x)/2 (PISA-2).

What each pin catches:
  leaf closed forms       PISA-1 = sum_g (log C + s q_g . mu), mu the numpy mean
                          key (linearity of the mean); PISA-2 adds
                          s^2 q_g^T Cov q_g / 2 with numpy's population
                          covariance matrix -- wrong count, missing 1/2,
                          sample instead of population variance, wrong scale;
  intermediate levels     the same over the eligible children's direct means;
                          one eligible child gives its plain dot;
  Taylor orders           with the scale eps -> 0, LSE - PISA-1 shrinks as
                          eps^2 with coefficient var/2 and LSE - PISA-2 as
                          eps^3 with coefficient kappa_3/6 -- a dropped or
                          mis-signed term fails;
  Jensen                  PISA-1 <= LSE at every node;
  walk                    with K covering E every scorer returns all blocks.
"""
import math

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle
from pyramid_top_block_mean_gb300 import workloads as W


def np_inputs(shape, seed):
    q, k = W.iid(shape, seed)
    return q.double().numpy(), k.double().numpy()


def level_sizes(nb):
    sizes = [nb]
    while sizes[-1] > 1:
        sizes.append(-(-sizes[-1] // 2))
    return sizes


def span(level, j, C, n):
    w = 1 << (level - 1)
    return j * w * C, min((j + 1) * w * C, n)


S = W.Shape(B=1, N=64 * 40 + 17, Hq=4, Hkv=2, d=16, C=64, K=3, dtype="fp32")


@pytest.mark.parametrize("scorer", [1, 2])
def test_leaf_closed_forms(scorer):
    q, k = np_inputs(S, 5)
    o = oracle.Oracle.from_shape(S, scorer=scorer)
    pyr = o.pyramid(k)
    sc = 1.0 / math.sqrt(S.d)
    t = S.N - 1
    nb = -(-S.N // S.C)
    for h in range(S.Hkv):
        for j in range(1, t // S.C - 1):  # E = [1, qb - 2]: complete past blocks
            keys = k[0, h, j * S.C:(j + 1) * S.C]
            mu = keys.mean(axis=0)
            cov = np.cov(keys, rowvar=False, bias=True)
            want = 0.0
            for g in range(S.G):
                qg = q[0, h * S.G + g, t]
                want += math.log(S.C) + sc * qg @ mu
                if scorer == 2:
                    want += 0.5 * sc * sc * qg @ cov @ qg
            got = o.score_nodes(q, k, pyr, 0, h, t, 1, [j])[0]
            assert abs(got - want) < 1e-10 * max(1.0, abs(want)), (h, j, got, want)
    assert nb > 8


@pytest.mark.parametrize("scorer", [1, 2])
def test_intermediate_closed_forms(scorer):
    q, k = np_inputs(S, 6)
    o = oracle.Oracle.from_shape(S, scorer=scorer)
    pyr = o.pyramid(k)
    sizes = level_sizes(-(-S.N // S.C))
    sc = 1.0 / math.sqrt(S.d)
    checked = {1: 0, 2: 0}
    for t in (S.N - 1, 64 * 9 + 3, 64 * 23):
        for h in range(S.Hkv):
            for level in range(2, len(sizes) + 1):
                for j in range(sizes[level - 1]):
                    if not o.eligible(t, level, j):
                        continue
                    kids = [c for c in (2 * j, 2 * j + 1)
                            if c < sizes[level - 2] and o.eligible(t, level - 1, c)]
                    mus = [k[0, h, slice(*span(level - 1, c, S.C, S.N))].mean(axis=0) for c in kids]
                    want = 0.0
                    for g in range(S.G):
                        x = np.array([sc * q[0, h * S.G + g, t] @ m for m in mus])
                        want += math.log(len(x)) + x.mean()
                        if scorer == 2:
                            want += 0.5 * ((x - x.mean()) ** 2).mean()
                    got = o.score_nodes(q, k, pyr, 0, h, t, level, [j])[0]
                    assert abs(got - want) < 1e-10 * max(1.0, abs(want)), (level, j, got, want)
                    checked[len(kids)] += 1
    assert checked[1] > 0 and checked[2] > 0, checked


def test_taylor_orders_at_the_leaves():
    """As the scale eps -> 0 the truncation errors vanish at the orders the
    expansion fixes: LSE - PISA-1 ~ eps^2 var/2, LSE - PISA-2 ~ eps^3 k3/6,
    with var and k3 the central moments of the unscaled dots q . k_i."""
    s = W.Shape(B=1, N=64 * 12, Hq=1, Hkv=1, d=16, C=64, K=2, dtype="fp32")
    q, k = np_inputs(s, 9)
    t = s.N - 1
    j = 4
    x0 = k[0, 0, j * 64:(j + 1) * 64] @ q[0, 0, t]
    var = ((x0 - x0.mean()) ** 2).mean()
    k3 = ((x0 - x0.mean()) ** 3).mean()
    for eps in (1e-2, 5e-3):
        sc = {}
        for scorer in (0, 1, 2):
            o = oracle.Oracle.from_shape(s, scale=eps, scorer=scorer)
            sc[scorer] = o.score_nodes(q, k, o.pyramid(k), 0, 0, t, 1, [j])[0]
        assert sc[0] == pytest.approx(logsumexp(eps * x0), abs=1e-12)
        assert (sc[0] - sc[1]) / eps ** 2 == pytest.approx(var / 2, rel=5 * eps * abs(k3) / var + 1e-6)
        assert (sc[0] - sc[2]) / eps ** 3 == pytest.approx(k3 / 6, rel=0.05, abs=1e-3)


def test_jensen_mean_below_lse_and_full_walks():
    q, k = np_inputs(S, 7)
    o0 = oracle.Oracle.from_shape(S)
    o1 = oracle.Oracle.from_shape(S, scorer=1)
    pyr = o0.pyramid(k)
    sizes = level_sizes(-(-S.N // S.C))
    t = S.N - 1
    for level in range(1, len(sizes) + 1):
        nodes = [j for j in range(sizes[level - 1]) if o0.eligible(t, level, j)]
        a = o0.score_nodes(q, k, pyr, 0, 1, t, level, nodes)
        b = o1.score_nodes(q, k, pyr, 0, 1, t, level, nodes)
        assert (b <= a + 1e-12).all(), level
    # K covering E: every scorer returns every causal block
    big = W.Shape(B=1, N=64 * 12 + 5, Hq=2, Hkv=1, d=8, C=64, K=16, dtype="fp32")
    qb_, kb_ = np_inputs(big, 8)
    outs = [oracle.Oracle.from_shape(big, scorer=sc_).select(qb_, kb_)["idx"] for sc_ in (0, 1, 2)]
    assert (outs[0] == outs[1]).all() and (outs[0] == outs[2]).all()
    for t_ in range(big.N):
        want = list(range(t_ // 64 + 1))
        got = [x for x in outs[0][t_] if x >= 0]
        assert got == want, (t_, got)
