"""Pins of the oracle's prefix-consistent (leak-free) prefill reading.

Reading (agihunt.info summary, pyramid paragraph: decode routing walks the
pyramid of the keys seen so far; rcap.io, the pisa_select sketch walks node
summaries without a mask): a prefill query at position t reads every node
summary as the mean of the keys of the node's span at positions <= t, i.e.
the pyramid of the sequence's first t + 1 keys.  That is exactly what the
decode step at length t + 1 sees, so the pins are:
  * equality with the oracle's decode selection at length t + 1, for every t
    (indices, scores and margins), on random tiny shapes;
  * the independent recursive restatement (numpy means of the raw keys at
    positions <= t, scipy logsumexp) on random tiny shapes;
  * no leak: changing any key after t leaves query t's selection unchanged,
    while the default reading does see such a change;
  * queries whose path holds no later key (the last query of a sequence)
    select as in the default reading.
CPU only."""
import numpy as np
import pytest
import torch

import oracle
from pyramid_top_block_mean_gb300 import workloads as W

from test_oracle_pins import RecursiveRef, np_inputs, pad


@pytest.mark.parametrize("seed", range(5))
def test_prefix_prefill_equals_decode_at_every_length(seed):
    gen = torch.Generator().manual_seed(900 + seed)
    s = W.random_shape(gen, max_blocks=30)
    q, k = np_inputs(s, 40 + seed)
    op = oracle.Oracle.from_shape(s, prefix=True)
    rp = op.select(q, k)
    od = oracle.Oracle.from_shape(s)
    for t in range(s.N):
        lens = [t + 1] * s.B
        rd = od.select(q[:, :, t], k, seq_lens=lens, decode=True)
        for b in range(s.B):
            for h in range(s.Hkv):
                i = (b * s.Hkv + h) * s.N + t
                j = b * s.Hkv + h
                assert rp["idx"][i].tolist() == rd["idx"][j].tolist(), (s, b, h, t)
                np.testing.assert_allclose(rp["score"][i], rd["score"][j], rtol=1e-11, atol=1e-11)
                if np.isfinite(rd["margin"][j]):
                    assert abs(rp["margin"][i] - rd["margin"][j]) <= 1e-11


@pytest.mark.parametrize("seed", range(12))
def test_prefix_prefill_matches_recursive_restatement(seed):
    gen = torch.Generator().manual_seed(950 + seed)
    s = W.random_shape(gen, max_blocks=40)
    q, k = np_inputs(s, 70 + seed)
    r = oracle.Oracle.from_shape(s, prefix=True).select(q, k)
    ref = RecursiveRef(q, k, s.C, s.K, prefix=True)
    i = 0
    for b in range(s.B):
        for h in range(s.Hkv):
            for t in range(s.N):
                wi, ws = pad(*ref.select(b, h, t), s.K + 3)
                if r["margin"][i] > 1e-9:
                    assert r["idx"][i].tolist() == wi.tolist(), (s, b, h, t)
                    np.testing.assert_allclose(r["score"][i], ws, rtol=1e-11, atol=1e-11)
                i += 1


def test_prefix_selection_ignores_later_keys():
    s = W.Shape(B=1, N=64 * 37 + 5, Hq=4, Hkv=1, d=16, K=3, dtype="fp32")
    q, k = np_inputs(s, 5)
    ts = [64 * 9 + 3, 64 * 17 + 40, 64 * 30, 64 * 33 + 63]
    base_p = oracle.Oracle.from_shape(s, prefix=True).select(q, k, sel=[(0, 0, t) for t in ts])
    base_d = oracle.Oracle.from_shape(s).select(q, k, sel=[(0, 0, t) for t in ts])
    changed_default = 0
    for n, t in enumerate(ts):
        k2 = k.copy()
        rng = np.random.default_rng(t)
        k2[0, 0, t + 1:] = 4.0 * rng.standard_normal(k2[0, 0, t + 1:].shape)
        rp = oracle.Oracle.from_shape(s, prefix=True).select(q, k2, sel=[(0, 0, t)])
        assert rp["idx"][0].tolist() == base_p["idx"][n].tolist(), t
        np.testing.assert_allclose(rp["score"][0], base_p["score"][n], rtol=1e-12, atol=1e-12)
        rd = oracle.Oracle.from_shape(s).select(q, k2, sel=[(0, 0, t)])
        changed_default += rd["idx"][0].tolist() != base_d["idx"][n].tolist()
    assert changed_default >= 1  # the default reading does look at later keys


def test_last_query_is_the_same_under_both_readings():
    s = W.Shape(B=2, N=64 * 45, Hq=8, Hkv=2, d=32, K=4, dtype="fp32")
    q, k = np_inputs(s, 8)
    sel = [(b, h, s.N - 1) for b in range(s.B) for h in range(s.Hkv)]
    rp = oracle.Oracle.from_shape(s, prefix=True).select(q, k, sel=sel)
    rd = oracle.Oracle.from_shape(s).select(q, k, sel=sel)
    assert rp["idx"].tolist() == rd["idx"].tolist()
    np.testing.assert_allclose(rp["score"], rd["score"], rtol=1e-12, atol=1e-12)
