"""The comparison rule itself (tests/parity.py), on the CPU: the oracle's own
output passes, and outputs with one planted defect fail, through both the
vectorised fast path and the per-query path.  This keeps the GPU parity
tests from passing because the checker went blind."""

import numpy as np
import pytest

import oracle
from pyramid_top_block_mean_gb300 import workloads as W

from parity import Report, check_structure, compare, structure_ok


@pytest.fixture(scope="module")
def case():
    s = W.Shape(B=1, N=64 * 30 + 17, Hq=4, Hkv=2, d=64, K=4)
    q, k = W.iid(s, 41)
    o = oracle.Oracle.from_shape(s)
    qn, kn = q.double().numpy(), k.double().numpy()
    pyr = o.pyramid(kn)
    ref = o.select(qn, kn, pyr, trace=True)
    keys = [(b, h, t) for b in range(s.B) for h in range(s.Hkv) for t in range(s.N)]
    return s, o, qn, kn, pyr, ref, keys


def run(case, idx, score, trace=None):
    s, o, qn, kn, pyr, ref, keys = case
    return compare(o, qn, kn, pyr, ref, idx, score, trace, keys, Report())


def test_oracle_output_passes(case):
    s, o, qn, kn, pyr, ref, keys = case
    rep = run(case, ref["idx"].copy(), ref["score"].copy(), ref["trace"])
    assert rep.ok(), str(rep)
    assert rep.n == len(keys) and rep.exact == len(keys)


def _late_row(case):
    s, o, qn, kn, pyr, ref, keys = case
    # a late query of key head 1 whose margin is clear of the tie threshold
    for i in range(len(keys) - 1, 0, -1):
        if ref["margin"][i] > 0.05 and keys[i][2] // s.C > s.K + 4:
            return i
    raise AssertionError("no clear-margin query")


@pytest.mark.parametrize("defect", ["swap_index", "score_off", "forced_score", "order", "padding",
                                    "future_block", "missing_forced", "pad_score"])
def test_planted_defect_fails(case, defect):
    s, o, qn, kn, pyr, ref, keys = case
    idx, score = ref["idx"].copy(), ref["score"].copy()
    i = _late_row(case)
    t = keys[i][2]
    qb = t // s.C
    real = [j for j in idx[i] if j >= 0]
    F = {0, qb - 1, qb}
    top = [j for j in real if j not in F]
    if defect == "swap_index":
        other = next(j for j in range(1, qb - 1) if j not in real)
        row = sorted([j for j in real if j != top[0]] + [other])
        idx[i, :len(row)] = row
    elif defect == "score_off":
        c = next(c for c in range(s.K + 3) if np.isfinite(score[i, c]))
        score[i, c] += 3e-3
    elif defect == "forced_score":
        score[i, 0] = 1.0
    elif defect == "order":
        idx[i, [1, 2]] = idx[i, [2, 1]]
        score[i, [1, 2]] = score[i, [2, 1]]
    elif defect == "padding":
        idx[i, 1] = -1
    elif defect == "future_block":
        idx[i, len(real) - 1] = qb + 1
    elif defect == "missing_forced":
        other = next(j for j in range(1, qb - 1) if j not in real)
        row = sorted([j for j in real if j != 0] + [other])
        idx[i, :len(row)] = row
    elif defect == "pad_score":
        j = next(c for c in range(s.K + 3) if idx[i, c] < 0) if (idx[i] < 0).any() else None
        if j is None:
            # a full row: force a padding slot by dropping the last block
            idx[i, -1] = -1
            j = s.K + 2
        score[i, j] = 0.0
    rep = run(case, idx, score, ref["trace"])
    assert not rep.ok(), f"{defect} went unnoticed"


def test_vectorised_structure_agrees_with_per_query_check(case):
    s, o, qn, kn, pyr, ref, keys = case
    gen = np.random.default_rng(3)
    idx, score = ref["idx"].copy(), ref["score"].copy()
    rows = gen.choice(len(keys), 300, replace=False)
    for r in rows:
        kind = gen.integers(0, 5)
        c = int(gen.integers(0, s.K + 3))
        if kind == 0:
            idx[r, c] = -1
        elif kind == 1:
            idx[r, c] = int(gen.integers(0, 40))
        elif kind == 2:
            score[r, c] = float(gen.choice([np.inf, -np.inf, 0.5]))
        elif kind == 3:
            idx[r] = idx[r][::-1]
    ts = np.array([t for (_, _, t) in keys])
    fast = structure_ok(idx, score, ts, s.C, s.K)
    for r in range(len(keys)):
        slow = check_structure(idx[r], score[r], keys[r][2], s.C, s.K, Report(), "")
        assert bool(fast[r]) == slow, (r, idx[r], score[r])
