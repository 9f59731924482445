"""Pins of the fp64 CPU oracle against facts that do not come from the oracle
itself: hand-worked walks, closed forms, brute force on tiny inputs, library
routines (numpy means, scipy logsumexp/softmax), Jensen's inequality and
invariances.  CPU only.

What each pin catches:
  pyramid            wrong span, dropped/duplicated key, ragged-end or
                     seq_len handling, layout offsets;
  hand walks         level order, eligibility, child expansion, GQA sum,
                     tie rule, output format;
  closed form        forced set, causal range, leaf LSE value;
  exhaustive regime  leaf LSE, Top-K direction and tie rule;
  needle             argmax direction at every level, child indexing;
  scipy scores       intermediate LSE over eligible children (a dropped or
                     extra child, wrong level, wrong sign, wrong scale);
  Jensen chain       mean-vs-LSE ordering of the scoring rule;
  recursive ref.     the whole walk on many random tiny shapes;
  decode==prefill    the capacity layout and per-sequence lengths.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import logsumexp, softmax

import oracle
from pyramid_top_block_mean_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- helpers
def level_sizes(nb):
    sizes = [nb]
    while sizes[-1] > 1:
        sizes.append(-(-sizes[-1] // 2))
    return sizes


def np_inputs(shape, seed):
    q, k = W.iid(shape, seed)
    return q.double().numpy(), k.double().numpy()


def span_keys(level, j, C, length):
    w = 1 << (level - 1)
    return j * w * C, min((j + 1) * w * C, length)


class RecursiveRef:
    """An independent, recursive restatement of the walk (numpy means taken
    directly from the raw keys, scipy logsumexp).  Tiny inputs only."""

    def __init__(self, q, k, C, K, scale=None, prefix=False):
        self.q, self.k, self.C, self.K = q, k, C, K
        self.prefix = prefix  # summaries of the keys at positions <= t only
        self.d = q.shape[-1]
        self.s = scale if scale else 1.0 / math.sqrt(self.d)
        self.G = q.shape[1] // k.shape[1]

    def select(self, b, h, t, length=None, qrows=None):
        N = self.k.shape[2] if length is None else length
        C, K = self.C, self.K
        nb = -(-N // C)
        sizes = level_sizes(nb)
        qb = t // C
        E = set(range(1, qb - 1))
        F = sorted({0, qb - 1, qb} & set(range(0, qb + 1)))
        heads = [self.q[b, h * self.G + g, t] if qrows is None else qrows[g]
                 for g in range(self.G)]
        keys = self.k[b, h, :N]

        def leaves(level, j):
            w = 1 << (level - 1)
            return range(j * w, min((j + 1) * w, nb))

        def elig(level, j):
            return any(x in E for x in leaves(level, j))

        def mean(level, j):
            lo, hi = span_keys(level, j, C, N)
            if self.prefix:
                hi = min(hi, t + 1)
            return keys[lo:hi].mean(axis=0)

        def score(level, j):
            if level == 1:
                lo, hi = j * C, min((j + 1) * C, N)
                return sum(logsumexp(self.s * keys[lo:hi] @ qh) for qh in heads)
            kids = [c for c in (2 * j, 2 * j + 1) if c < sizes[level - 2] and elig(level - 1, c)]
            return sum(logsumexp([self.s * qh @ mean(level - 1, c) for c in kids]) for qh in heads)

        def descend(level, cands):
            if len(cands) > K:
                kept = sorted(cands, key=lambda j: (-score(level, j), j))[:K]
            else:
                kept = list(cands)
            if level == 1:
                return kept
            nxt = [c for j in kept for c in (2 * j, 2 * j + 1)
                   if c < sizes[level - 2] and elig(level - 1, c)]
            return descend(level - 1, nxt)

        top = descend(len(sizes), [0]) if E else []
        out = sorted(set(top) | set(F))
        sc = [math.inf if i in F else score(1, i) for i in out]
        return out, sc


def pad(idx, sc, width):
    idx = list(idx) + [-1] * (width - len(idx))
    sc = list(sc) + [-math.inf] * (width - len(sc))
    return np.array(idx, np.int32), np.array(sc)


# ------------------------------------------------------------------ pyramid
@pytest.mark.parametrize("seed", range(6))
def test_pyramid_nodes_are_direct_means(seed):
    gen = torch.Generator().manual_seed(100 + seed)
    s = W.random_shape(gen, max_blocks=37)
    q, k = np_inputs(s, seed)
    o = oracle.Oracle.from_shape(s)
    lens = None
    if seed % 2:
        lens = [int(torch.randint(0, s.N + 1, (1,), generator=gen)) for _ in range(s.B)]
    pyr = o.pyramid(k, lens)
    sizes = level_sizes(-(-s.N // s.C))
    for b in range(s.B):
        length = s.N if lens is None else lens[b]
        for h in range(s.Hkv):
            off = 0
            for level, n in enumerate(sizes, start=1):
                for j in range(n):
                    lo, hi = span_keys(level, j, s.C, length)
                    want = k[b, h, lo:hi].mean(axis=0) if hi > lo else np.zeros(s.d)
                    np.testing.assert_allclose(pyr[b, h, off + j], want, rtol=1e-12, atol=1e-12)
                off += n


def test_pyramid_parent_is_count_weighted_mean_of_children():
    s = W.Shape(B=1, N=1000, Hq=1, Hkv=1, d=8, C=16, K=2, dtype="fp32")
    _, k = np_inputs(s, 7)
    o = oracle.Oracle.from_shape(s)
    pyr = o.pyramid(k)[0, 0]
    sizes = level_sizes(-(-s.N // s.C))
    offs = np.cumsum([0] + sizes)
    for level in range(2, len(sizes) + 1):
        for j in range(sizes[level - 1]):
            num = np.zeros(s.d)
            cnt = 0
            for c in (2 * j, 2 * j + 1):
                if c < sizes[level - 2]:
                    lo, hi = span_keys(level - 1, c, s.C, s.N)
                    num += (hi - lo) * pyr[offs[level - 2] + c]
                    cnt += hi - lo
            np.testing.assert_allclose(pyr[offs[level - 1] + j], num / cnt, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(pyr[offs[-2]], k[0, 0].mean(axis=0), rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------- hand walks
@pytest.mark.parametrize("name", ["hand_walk_pruning.json", "hand_walk_gqa_tie.json"])
def test_hand_worked_walks(name):
    fx = json.load(open(os.path.join(GOLDEN, name)))
    sh = fx["shape"]
    N, d, Hq = sh["N"], sh["d"], sh["Hq"]
    q = np.zeros((1, Hq, N, d))
    for g, row in enumerate(fx["q_at_t"]):
        q[0, g, fx["t"]] = row
    k = np.array(fx["k"], np.float64).reshape(1, 1, N, d)
    o = oracle.Oracle(1, N, Hq, 1, d, sh["C"], sh["K"])
    r = o.select(q, k, sel=[(0, 0, fx["t"])], trace=True)
    assert r["idx"][0].tolist() == fx["expect_idx"]
    want = [float(x) for x in fx["expect_score"]]
    np.testing.assert_allclose(r["score"][0], want, rtol=0, atol=1e-12)
    for level, kept in fx["expect_trace"].items():
        got = [x for x in r["trace"][0, int(level) - 1] if x >= 0]
        assert got == kept, (level, got, kept)
    assert abs(r["margin"][0] - eval(fx["expect_margin"], {"math": math})) < 1e-12
    pyr = o.pyramid(k)
    for level, spec in fx.get("expect_level_scores", {}).items():
        got = o.score_nodes(q, k, pyr, 0, 0, fx["t"], int(level), spec["nodes"])
        want = [eval(e, {"math": math}) for e in spec["scores"]]
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)
    if "expect_exhaustive_top1" in fx:
        lse = {j: float(q[0, 0, fx["t"]] @ k[0, 0, j]) for j in range(1, fx["t"] // sh["C"] - 1)}
        assert max(lse, key=lse.get) == fx["expect_exhaustive_top1"]


# ----------------------------------------------------------- closed forms
@pytest.mark.parametrize("seed", range(3))
def test_K_at_least_E_returns_every_causal_block(seed):
    gen = torch.Generator().manual_seed(200 + seed)
    s = W.random_shape(gen, max_blocks=24)
    nb = -(-s.N // s.C)
    s.K = max(1, nb)  # K >= |E| for every query
    q, k = np_inputs(s, seed)
    o = oracle.Oracle.from_shape(s)
    r = o.select(q, k)
    sc = 1.0 / math.sqrt(s.d)
    W_ = s.K + 3
    for i, (b, h, t) in enumerate((b, h, t) for b in range(s.B) for h in range(s.Hkv) for t in range(s.N)):
        qb = t // s.C
        want_idx = list(range(qb + 1))
        F = {0, qb - 1, qb} & set(range(qb + 1))
        want_sc = []
        for j in want_idx:
            if j in F:
                want_sc.append(math.inf)
            else:
                keys = k[b, h, j * s.C:(j + 1) * s.C]
                want_sc.append(sum(logsumexp(sc * keys @ q[b, h * s.G + g, t]) for g in range(s.G)))
        wi, ws = pad(want_idx, want_sc, W_)
        assert r["idx"][i].tolist() == wi.tolist()
        np.testing.assert_allclose(r["score"][i], ws, rtol=1e-12, atol=1e-12)
        assert r["margin"][i] == math.inf


def brute_topk(q, k, b, h, t, C, K, G, s):
    """Exhaustive ranking of every eligible leaf by raw-key LSE."""
    qb = t // C
    E = list(range(1, qb - 1))
    sc = {j: sum(logsumexp(s * k[b, h, j * C:(j + 1) * C] @ q[b, h * G + g, t]) for g in range(G))
          for j in E}
    top = sorted(E, key=lambda j: (-sc[j], j))[:K]
    F = {0, qb - 1, qb} & set(range(qb + 1))
    out = sorted(set(top) | F)
    return out, [math.inf if j in F else sc[j] for j in out]


def test_exhaustive_regime_tiny_workload_K8():
    """16 leaves, K = 8: every level keeps all of its candidates down to level 2
    (<= 8 level-2 nodes), so the leaf candidates are all of E and the result
    is the exhaustive raw-key-LSE Top-8 (the tiny workload, K raised to 8)."""
    s = W.Shape(**{**W.TINY.__dict__, "K": 8})
    q, k = W.iid(s, 0)
    q, k = q.double().numpy(), k.double().numpy()
    o = oracle.Oracle.from_shape(s)
    r = o.select(q, k)
    for t in range(s.N):
        wi, ws = pad(*brute_topk(q, k, 0, 0, t, s.C, s.K, 1, 1 / math.sqrt(s.d)), s.K + 3)
        assert r["idx"][t].tolist() == wi.tolist(), t
        np.testing.assert_allclose(r["score"][t], ws, rtol=1e-12, atol=1e-12)


def test_exhaustive_regime_tiny_workload_K4_early_queries():
    """K = 4 (the tiny workload as specified): for qb <= 9 at most 4 level-2
    nodes are eligible, so the walk is exhaustive for positions t < 640."""
    s = W.TINY
    q, k = W.iid(s, 0)
    q, k = q.double().numpy(), k.double().numpy()
    o = oracle.Oracle.from_shape(s)
    sel = [(0, 0, t) for t in range(640)]
    r = o.select(q, k, sel=sel)
    for i, t in enumerate(range(640)):
        wi, ws = pad(*brute_topk(q, k, 0, 0, t, s.C, s.K, 1, 1 / math.sqrt(s.d)), s.K + 3)
        assert r["idx"][i].tolist() == wi.tolist(), t
        np.testing.assert_allclose(r["score"][i], ws, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------ needle
@pytest.mark.parametrize("seed", range(4))
def test_planted_needle_block_is_found(seed):
    gen = torch.Generator().manual_seed(300 + seed)
    C, d, G, K = 4, 8, 1 + seed % 3, 2
    N = 4 * 64 + 3
    s = W.Shape(B=1, N=N, Hq=G, Hkv=1, d=d, C=C, K=K, dtype="fp32")
    q, k = np_inputs(s, seed)
    o = oracle.Oracle.from_shape(s)
    for trial in range(6):
        t = int(torch.randint(8 * C, N, (1,), generator=gen))
        qb = t // C
        j = int(torch.randint(1, qb - 1, (1,), generator=gen))
        u = q[0, :, t].sum(axis=0)
        u /= np.linalg.norm(u)
        kk = k.copy()
        kk[0, 0, j * C:(j + 1) * C] = 40.0 * math.sqrt(d) * u
        r = o.select(q, kk, sel=[(0, 0, t)], trace=True)
        # A head whose query points away from the needle scores a lone needle
        # child very low, so the check needs every head to favour it.
        if all(q[0, g, t] @ u > 0 for g in range(G)):
            assert j in r["idx"][0].tolist(), (t, j)
            # its ancestors are kept at every level of the walk
            for level in range(2, o.num_levels + 1):
                anc = j >> (level - 1)
                kept = r["trace"][0, level - 1]
                if (kept >= 0).any():
                    assert anc in kept.tolist(), (level, anc, kept)


# ------------------------------------------------- intermediate LSE scores
@pytest.mark.parametrize("seed", range(4))
def test_intermediate_scores_match_scipy_on_direct_means(seed):
    gen = torch.Generator().manual_seed(400 + seed)
    s = W.random_shape(gen, max_blocks=40)
    q, k = np_inputs(s, seed)
    o = oracle.Oracle.from_shape(s)
    pyr = o.pyramid(k)
    sizes = level_sizes(-(-s.N // s.C))
    sc = 1.0 / math.sqrt(s.d)
    for _ in range(20):
        b = int(torch.randint(0, s.B, (1,), generator=gen))
        h = int(torch.randint(0, s.Hkv, (1,), generator=gen))
        t = int(torch.randint(0, s.N, (1,), generator=gen))
        for level in range(2, len(sizes) + 1):
            for j in range(sizes[level - 1]):
                if not o.eligible(t, level, j):
                    continue
                kids = [c for c in (2 * j, 2 * j + 1)
                        if c < sizes[level - 2] and o.eligible(t, level - 1, c)]
                mus = [k[b, h, slice(*span_keys(level - 1, c, s.C, s.N))].mean(axis=0) for c in kids]
                want = sum(logsumexp([sc * q[b, h * s.G + g, t] @ m for m in mus]) for g in range(s.G))
                got = o.score_nodes(q, k, pyr, b, h, t, level, [j])[0]
                assert abs(got - want) < 1e-10, (level, j, got, want)


def test_jensen_chain_per_node():
    """For a node whose two children hold equally many keys:
    s q.mu_node <= log-mean-exp over child means <= log-mean-exp over raw keys
    (the ordering of the scoring rule's justification; rcap.io 'The scoring
    rule matters', Appendix A as summarised there)."""
    s = W.Shape(B=1, N=64 * 64, Hq=1, Hkv=1, d=16, C=64, K=4, dtype="fp32")
    q, k = np_inputs(s, 11)
    o = oracle.Oracle.from_shape(s)
    pyr = o.pyramid(k)
    sizes = level_sizes(s.N // s.C)
    offs = np.cumsum([0] + sizes)
    sc = 1.0 / math.sqrt(s.d)
    t = s.N - 1  # qb = 63, E = [1, 61]
    checked = 0
    for level in range(2, len(sizes) + 1):
        for j in range(sizes[level - 1]):
            w = 1 << (level - 2)  # leaves per child
            c0, c1 = 2 * j, 2 * j + 1
            # both children fully inside E (equal sizes, both eligible)
            if c0 * w < 1 or (c1 + 1) * w - 1 > 61:
                continue
            qv = q[0, 0, t]
            lo, hi = span_keys(level, j, s.C, s.N)
            mean_score = sc * qv @ pyr[0, 0, offs[level - 1] + j]
            lme_children = o.score_nodes(q, k, pyr, 0, 0, t, level, [j])[0] - math.log(2.0)
            lme_raw = logsumexp(sc * k[0, 0, lo:hi] @ qv) - math.log(hi - lo)
            assert mean_score <= lme_children + 1e-12
            assert lme_children <= lme_raw + 1e-12
            checked += 1
    assert checked > 20


# -------------------------------------------------------------- invariances
def _shape_cpt_small():
    return W.Shape(B=1, N=2048 + 17, Hq=4, Hkv=2, d=16, C=16, K=3, dtype="fp32")


def test_shift_and_head_permutation_invariance():
    s = _shape_cpt_small()
    q, k = np_inputs(s, 21)
    o = oracle.Oracle.from_shape(s)
    base = o.select(q, k)
    ok = base["margin"] > 1e-9
    v = np.random.default_rng(0).normal(size=s.d)
    shifted = o.select(q, k + v)
    assert (shifted["idx"][ok] == base["idx"][ok]).all()
    perm = q.copy()
    perm[:, [0, 1]] = q[:, [1, 0]]  # swap the two heads of group 0
    perm[:, [2, 3]] = q[:, [3, 2]]
    swapped = o.select(perm, k)
    assert (swapped["idx"][ok] == base["idx"][ok]).all()
    fin = np.isfinite(base["score"]) & ok[:, None]
    np.testing.assert_allclose(swapped["score"][fin], base["score"][fin], rtol=1e-12, atol=1e-12)


def test_structure_of_outputs_and_work_bounds():
    s = _shape_cpt_small()
    q, k = np_inputs(s, 22)
    o = oracle.Oracle.from_shape(s)
    r = o.select(q, k, trace=True)
    sizes = level_sizes(-(-s.N // s.C))
    nb = sizes[0]
    i = 0
    for b in range(s.B):
        for h in range(s.Hkv):
            for t in range(s.N):
                qb = t // s.C
                idx = r["idx"][i]
                sc = r["score"][i]
                real = idx[idx >= 0]
                assert (idx[len(real):] == -1).all()
                assert (np.diff(real) > 0).all()
                assert real.max() <= qb
                F = {0, qb - 1, qb} & set(range(qb + 1))
                assert F <= set(real.tolist())
                for j, x in zip(real, sc[:len(real)]):
                    assert (x == math.inf) == (j in F)
                assert (sc[len(real):] == -math.inf).all()
                nE = max(0, qb - 2)
                assert len(real) == len(F) + min(s.K, nE)
                # trace: each kept set is eligible and nested in its parents
                tr = r["trace"][i]
                for level in range(1, len(sizes)):
                    kept = [x for x in tr[level - 1] if x >= 0]
                    up = [x for x in tr[level] if x >= 0]
                    for x in kept:
                        assert o.eligible(t, level, x)
                        if up:
                            assert (x >> 1) in up
                i += 1
    c = r["counters"]
    nq = s.B * s.Hkv * s.N
    assert c["levels_scored"] <= nq * math.ceil(math.log2(nb))
    assert c["cands_scored"] <= c["levels_scored"] * 2 * s.K
    assert c["child_dots"] <= 2 * c["cands_scored"]


# -------------------------------------------------- recursive brute force
@pytest.mark.parametrize("seed", range(30))
def test_recursive_reference_on_random_tiny_shapes(seed):
    gen = torch.Generator().manual_seed(500 + seed)
    s = W.random_shape(gen, max_blocks=40)
    q, k = np_inputs(s, seed)
    o = oracle.Oracle.from_shape(s)
    r = o.select(q, k)
    ref = RecursiveRef(q, k, s.C, s.K)
    i = 0
    for b in range(s.B):
        for h in range(s.Hkv):
            for t in range(s.N):
                wi, ws = pad(*ref.select(b, h, t), s.K + 3)
                if r["margin"][i] > 1e-9:
                    assert r["idx"][i].tolist() == wi.tolist(), (s, b, h, t)
                    np.testing.assert_allclose(r["score"][i], ws, rtol=1e-11, atol=1e-11)
                i += 1


# ------------------------------------------------------- decode vs prefill
@pytest.mark.parametrize("seed", range(4))
def test_decode_equals_prefill_of_the_prefix(seed):
    gen = torch.Generator().manual_seed(600 + seed)
    s = W.random_shape(gen, max_blocks=40)
    q4, k = np_inputs(s, seed)
    lens = [int(torch.randint(1, s.N + 1, (1,), generator=gen)) for _ in range(s.B)]
    qd = np.stack([q4[b, :, lens[b] - 1] for b in range(s.B)])  # [B, Hq, d]
    o = oracle.Oracle.from_shape(s)
    rd = o.select(qd, k, seq_lens=lens, decode=True)
    for b in range(s.B):
        L = lens[b]
        sb = W.Shape(B=1, N=L, Hq=s.Hq, Hkv=s.Hkv, d=s.d, C=s.C, K=s.K, dtype="fp32")
        ob = oracle.Oracle.from_shape(sb)
        rp = ob.select(q4[b:b + 1, :, :L], k[b:b + 1, :, :L],
                       sel=[(0, h, L - 1) for h in range(s.Hkv)])
        for h in range(s.Hkv):
            assert rd["idx"][b * s.Hkv + h].tolist() == rp["idx"][h].tolist()
            np.testing.assert_allclose(rd["score"][b * s.Hkv + h], rp["score"][h], rtol=1e-12, atol=1e-12)
        # and the capacity-layout pyramid agrees with the prefix pyramid node by node
        pc = o.pyramid(k, lens)[b]
        pp = ob.pyramid(k[b:b + 1, :, :L])[0]
        sizes_c = level_sizes(-(-s.N // s.C))
        sizes_p = level_sizes(-(-L // s.C))
        oc = np.cumsum([0] + sizes_c)
        op = np.cumsum([0] + sizes_p)
        for level, n in enumerate(sizes_p, start=1):
            np.testing.assert_allclose(pc[:, oc[level - 1]:oc[level - 1] + n],
                                       pp[:, op[level - 1]:op[level - 1] + n], rtol=1e-12, atol=1e-13)


# --------------------------------------------------------- flat comparator
def test_flat_single_head_is_argsort_of_mean_scores():
    """G = 1: softmax is monotone, so the flat Top-K is the Top-K of q.mu."""
    s = W.Shape(B=1, N=1500, Hq=2, Hkv=2, d=8, C=16, K=5, dtype="fp32")
    q, k = np_inputs(s, 31)
    o = oracle.Oracle.from_shape(s)
    pyr = o.pyramid(k)
    r = o.select_flat(q, pyr)
    i = 0
    for h in range(s.Hkv):
        mu = np.stack([k[0, h, j * s.C:(j + 1) * s.C].mean(axis=0) for j in range(s.N // s.C)])
        for t in range(s.N):
            qb = t // s.C
            z = mu[:qb] @ q[0, h, t]
            E = list(range(1, qb - 1))
            top = sorted(E, key=lambda j: (-z[j], j))[:s.K]
            F = {0, qb - 1, qb} & set(range(qb + 1))
            want = sorted(set(top) | F)
            got = [x for x in r["idx"][i] if x >= 0]
            if r["margin"][i] > 1e-12:
                assert got == want, (h, t)
            i += 1


def test_flat_scores_are_softmax_sums():
    s = W.Shape(B=1, N=777, Hq=4, Hkv=1, d=8, C=16, K=3, dtype="fp32")
    q, k = np_inputs(s, 32)
    o = oracle.Oracle.from_shape(s)
    pyr = o.pyramid(k)
    r = o.select_flat(q, pyr)
    mu = np.stack([k[0, 0, j * s.C:(j + 1) * s.C].mean(axis=0) for j in range(s.N // s.C)])
    sc = 1 / math.sqrt(s.d)
    for t in range(s.N):
        qb = t // s.C
        if qb < 4:
            continue
        p = sum(softmax(sc * mu[:qb] @ q[0, g, t]) for g in range(4))
        F = {0, qb - 1, qb}
        for j, x in zip(r["idx"][t], r["score"][t]):
            if j >= 0 and j not in F:
                assert abs(x - p[j]) < 1e-12


def test_flat_equals_pisa_when_K_covers_E():
    s = W.Shape(B=1, N=640, Hq=2, Hkv=1, d=8, C=16, K=40, dtype="fp32")
    q, k = np_inputs(s, 33)
    o = oracle.Oracle.from_shape(s)
    pyr = o.pyramid(k)
    a = o.select(q, k, pyr)
    f = o.select_flat(q, pyr)
    assert (a["idx"] == f["idx"]).all()
