"""Pins of the oracle's attention over the selected blocks (block-sparse
attention that reads only the chosen leaf blocks, causal inside each block;
agihunt.info summary, opening paragraph; rcap.io post, "Selection walks the
tree top-down": the kept leaf indices drive sparse attention over the
original keys).  CPU only.

What each pin catches:
  dense special case   every past block selected: PyTorch's causal
                       scaled_dot_product_attention (a library routine) --
                       wrong scale, dropped key, causal off-by-one, GQA head
                       mapping, wrong normaliser;
  masked library       random block subsets: the same library routine with a
                       boolean mask built from the definition of the attended
                       set -- wrong block span, ignored -1 slot, a block read
                       from the wrong key head;
  zero query           q = 0 gives the plain mean of v over the attended keys
                       (closed form, no exponentials);
  constant values      softmax weights sum to one;
  first position       t = 0 reads key 0 only;
  duplicates, order    a repeated block counts once; slot order is irrelevant.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from pyramid_top_block_mean_gb300 import workloads as W


def _inputs(B, N, Hq, Hkv, d, seed):
    shape = W.Shape(B=B, N=N, Hq=Hq, Hkv=Hkv, d=d, dtype="fp32")
    q, k = W.iid(shape, seed)
    v = W.values(shape, seed)
    return q.double(), k.double(), v.double()


def _library(q, k, v, mask, scale=None):
    """torch SDPA in fp64 with a boolean mask [B, Hkv, N, N] (True = attend)."""
    G = q.shape[1] // k.shape[1]
    kk = k.repeat_interleave(G, dim=1)
    vv = v.repeat_interleave(G, dim=1)
    m = mask.repeat_interleave(G, dim=1)
    return torch.nn.functional.scaled_dot_product_attention(q, kk, vv, attn_mask=m, scale=scale)


def _mask_from_idx(idx, N, C):
    """Boolean [B, Hkv, N, N]: key i attended by query t iff block(i) is a
    non-negative entry of idx[b, h, t] and i <= t."""
    B, Hkv = idx.shape[:2]
    mask = torch.zeros(B, Hkv, N, N, dtype=torch.bool)
    for b in range(B):
        for h in range(Hkv):
            for t in range(N):
                for j in idx[b, h, t]:
                    if j >= 0:
                        mask[b, h, t, j * C:min((j + 1) * C, N)] = True
    return mask & torch.ones(N, N, dtype=torch.bool).tril()


def _oracle_out(o, q, k, v, idx, C, K, scale=0.0, sel=None):
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    O = oracle.Oracle(B, N, Hq, Hkv, d, C, K, scale)
    return O.attend(q, k, v, idx, sel)


def _as_heads(out, B, Hkv, N, G, d):
    """[B*Hkv*N, G, d] -> [B, Hkv*G, N, d]."""
    return torch.from_numpy(out).reshape(B, Hkv, N, G, d).permute(0, 1, 3, 2, 4).reshape(B, Hkv * G, N, d)


@pytest.mark.parametrize("B,N,Hq,Hkv,d,C", [(1, 37, 4, 1, 8, 4), (2, 40, 4, 2, 16, 8), (1, 29, 3, 3, 5, 3)])
def test_dense_special_case_matches_causal_sdpa(B, N, Hq, Hkv, d, C):
    q, k, v = _inputs(B, N, Hq, Hkv, d, seed=11 + N)
    nb = -(-N // C)
    K = max(1, nb - 3 + 3)  # W = K + 3 >= nb slots
    idx = np.full((B, Hkv, N, K + 3), -1, np.int32)
    for t in range(N):
        blocks = list(range(t // C + 1))
        idx[:, :, t, :len(blocks)] = blocks
    got = _as_heads(_oracle_out(None, q, k, v, idx, C, K), B, Hkv, N, Hq // Hkv, d)
    G = Hq // Hkv
    ref = torch.nn.functional.scaled_dot_product_attention(
        q, k.repeat_interleave(G, 1), v.repeat_interleave(G, 1), is_causal=True)
    assert torch.allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_random_subsets_match_masked_sdpa():
    B, N, Hq, Hkv, d, C, K = 2, 48, 4, 2, 8, 4, 3
    q, k, v = _inputs(B, N, Hq, Hkv, d, seed=5)
    rng = np.random.default_rng(3)
    idx = np.full((B, Hkv, N, K + 3), -1, np.int32)
    for b in range(B):
        for h in range(Hkv):
            for t in range(N):
                qb = t // C
                cur = {qb}  # the current block always holds key t itself
                extra = rng.choice(qb + 1, size=min(qb + 1, rng.integers(0, K + 3)), replace=False)
                blocks = sorted(cur | set(int(x) for x in extra))[:K + 3]
                if qb not in blocks:
                    blocks[-1] = qb
                idx[b, h, t, :len(blocks)] = blocks
    got = _as_heads(_oracle_out(None, q, k, v, idx, C, K), B, Hkv, N, Hq // Hkv, d)
    ref = _library(q, k, v, _mask_from_idx(idx, N, C))
    assert torch.allclose(got, ref, rtol=1e-12, atol=1e-12)
    # an explicit scale goes inside the exponent
    got2 = _as_heads(_oracle_out(None, q, k, v, idx, C, K, scale=0.37), B, Hkv, N, Hq // Hkv, d)
    ref2 = _library(q, k, v, _mask_from_idx(idx, N, C), scale=0.37)
    assert torch.allclose(got2, ref2, rtol=1e-12, atol=1e-12)


def test_zero_query_is_plain_mean_of_attended_values():
    B, N, Hq, Hkv, d, C, K = 1, 40, 2, 1, 6, 8, 2
    _, k, v = _inputs(B, N, Hq, Hkv, d, seed=9)
    q = torch.zeros(B, Hq, N, d, dtype=torch.float64)
    idx = np.full((B, Hkv, N, K + 3), -1, np.int32)
    for t in range(N):
        qb = t // C
        idx[0, 0, t, :2] = sorted({0, qb}) + ([] if qb else [-1])
    got = _oracle_out(None, q, k, v, idx, C, K)
    vn = v.numpy()
    for t in range(N):
        qb = t // C
        keys = sorted(set(range(0, min(C, t + 1))) | set(range(qb * C, t + 1)))
        mean = vn[0, 0, keys].mean(axis=0)
        for g in range(Hq):
            np.testing.assert_allclose(got[t, g], mean, rtol=1e-13, atol=1e-13)


def test_constant_values_first_position_duplicates_and_order():
    B, N, Hq, Hkv, d, C, K = 1, 33, 4, 2, 8, 4, 4
    q, k, v = _inputs(B, N, Hq, Hkv, d, seed=21)
    idx = np.full((B, Hkv, N, K + 3), -1, np.int32)
    rng = np.random.default_rng(1)
    for h in range(Hkv):
        for t in range(N):
            qb = t // C
            blocks = sorted(set([qb]) | set(int(x) for x in rng.integers(0, qb + 1, size=3)))
            idx[0, h, t, :len(blocks)] = blocks
    # constant values: the output is that constant
    vc = torch.full_like(v, 0.625)
    got = _oracle_out(None, q, k, vc, idx, C, K)
    np.testing.assert_allclose(got, 0.625, rtol=0, atol=1e-14)
    # t = 0 reads key 0 only
    got = _oracle_out(None, q, k, v, idx, C, K)
    for h in range(Hkv):
        for g in range(Hq // Hkv):
            np.testing.assert_array_equal(got[h * N + 0, g], v.numpy()[0, h, 0])
    # a repeated block counts once, and the slot order does not matter
    dup = idx.copy()
    for h in range(Hkv):
        for t in range(N):
            row = [x for x in idx[0, h, t] if x >= 0]
            row = row[::-1] + [row[0]]
            dup[0, h, t, :] = -1
            dup[0, h, t, :len(row)] = row[:K + 3]
    got2 = _oracle_out(None, q, k, v, dup, C, K)
    np.testing.assert_allclose(got2, got, rtol=1e-13, atol=1e-13)


def test_selected_queries_match_full_run():
    B, N, Hq, Hkv, d, C, K = 2, 64, 4, 2, 8, 8, 2
    q, k, v = _inputs(B, N, Hq, Hkv, d, seed=31)
    O = oracle.Oracle(B, N, Hq, Hkv, d, C, K)
    idx = O.select(q, k)["idx"].reshape(B, Hkv, N, K + 3)
    full = O.attend(q, k, v, idx)
    sel = [(1, 1, 63), (0, 0, 5), (1, 0, 17)]
    part = O.attend(q, k, v, idx, sel)
    for i, (b, h, t) in enumerate(sel):
        np.testing.assert_array_equal(part[i], full[(b * Hkv + h) * N + t])
    # the same queries with only their head rows passed
    G = Hq // Hkv
    rows = np.stack([q.numpy()[b, h * G:(h + 1) * G, t] for (b, h, t) in sel])
    np.testing.assert_array_equal(O.attend(rows, k, v, idx, sel, qrows=True), part)


# ------------------------------------------------------- attention mass
def _mass_case(seed=3):
    s = W.Shape(B=1, N=64 * 12 + 9, Hq=4, Hkv=2, d=16, K=3, dtype="fp32")
    q, k = W.iid(s, seed)
    return s, q.double().numpy(), k.double().numpy()


def test_attention_mass_of_every_causal_block_is_one():
    s, q, k = _mass_case()
    sel = [(0, h, t) for h in range(s.Hkv) for t in (0, 63, 64, 300, s.N - 1)]
    idx = np.array([list(range(t // s.C + 1)) + [-1] * (20 - t // s.C - 1) for (_, _, t) in sel])
    r = oracle.attention_mass(q, k, idx, sel, s.C)
    np.testing.assert_allclose(r, 1.0, rtol=0, atol=1e-12)
    none = oracle.attention_mass(q, k, np.full((len(sel), 4), -1), sel, s.C)
    assert (none == 0.0).all()


def test_attention_mass_is_additive_over_disjoint_blocks_and_ignores_repeats():
    s, q, k = _mass_case(4)
    t = s.N - 1
    qb = t // s.C
    sel = [(0, 1, t)]
    parts = [oracle.attention_mass(q, k, np.array([[j]]), sel, s.C)[0] for j in range(qb + 1)]
    assert abs(sum(parts) - 1.0) < 1e-12
    both = oracle.attention_mass(q, k, np.array([[2, 5, 5, 2, qb + 3]]), sel, s.C)[0]
    assert abs(both - (parts[2] + parts[5])) < 1e-12


def test_attention_mass_of_one_block_is_the_exp_of_the_oracle_leaf_lse_gap():
    """G = 1: the mass of block j is exp(LSE(block j) - LSE(all keys <= t)),
    with LSE(block j) from the C oracle's leaf score (an independent
    implementation of the leaf log-sum-exp)."""
    s = W.Shape(B=1, N=64 * 10, Hq=1, Hkv=1, d=32, K=2, dtype="fp32")
    qt, kt = W.iid(s, 9)
    q, k = qt.double().numpy(), kt.double().numpy()
    o = oracle.Oracle.from_shape(s)
    pyr = o.pyramid(k)
    t = s.N - 1
    blocks = list(range(t // s.C + 1))
    lse_blocks = o.score_nodes(q, k, pyr, 0, 0, t, 1, blocks)
    total = np.logaddexp.reduce(lse_blocks)
    for j in (0, 3, 7, 9):
        m = oracle.attention_mass(q, k, np.array([[j]]), [(0, 0, t)], s.C)[0]
        assert abs(m - np.exp(lse_blocks[j] - total)) < 1e-12
