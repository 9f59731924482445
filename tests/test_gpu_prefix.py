"""GPU parity of the prefix-consistent (leak-free) prefill selection
(pisa_params.summaries = PISA_SUMMARIES_PREFIX) against the fp64 oracle's
prefix reading, through the C ABI.

Reading (agihunt.info summary, pyramid paragraph: decode routing walks the
pyramid of the keys seen so far; rcap.io, the pisa_select sketch): a query at
position t reads every node summary as the mean of the node's keys at
positions <= t, which is the decode step's view at length t + 1 (the oracle's
prefix mode is pinned to exactly that, CPU-side).  Same tolerance as every
prefill test (tests/parity.py): identical index sets except where the
oracle's K-th and (K+1)-th scores differ by < 1e-3 on some level, scores
within 2e-3, tie-exempt queries re-checked level by level from the GPU trace.

Cases: the tiny fp32 workload (CUDA-core routing), the planted pretrain
workload (tensor-core routing over difference rows), ragged shapes on both
routing kernels, K = 32, and a no-leak check: keys after position T replaced
by large noise leave every query t < T matching the same oracle answer.
"""
import pytest
import torch

import oracle
from pyramid_top_block_mean_gb300 import workloads as W

from parity import Report, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pisa():
    from pyramid_top_block_mean_gb300 import pisa as m
    return m


def run_prefix(pisa, s, q, k):
    p = pisa.params_from_shape(s, summaries=pisa.SUMMARIES_PREFIX)
    sel = pisa.Selector(p)
    L = pisa.pyramid_levels(p)
    tr = torch.full((s.B, s.Hkv, s.N, L, s.K), -7, dtype=torch.int32, device="cuda")
    sel.prefill(q.cuda(), k.cuda(), trace=tr)
    torch.cuda.synchronize()
    assert sel.device_status() == 0
    W_ = s.K + 3
    return dict(idx=sel.out_idx.reshape(-1, W_).cpu().numpy(),
                score=sel.out_score.reshape(-1, W_).cpu().double().numpy(),
                trace=tr.reshape(s.B * s.Hkv * s.N, -1, s.K).cpu().numpy())


def prefix_parity(pisa, s, q, k, rows=None):
    g = run_prefix(pisa, s, q, k)
    o = oracle.Oracle.from_shape(s, prefix=True)
    qn, kn = q.double().numpy(), k.double().numpy()
    pyr = o.pyramid(kn)
    keys = [(b, h, t) for b in range(s.B) for h in range(s.Hkv) for t in range(s.N)]
    if rows is not None:
        keys = [keys[i] for i in rows]
    ref = o.select(qn, kn, pyr, sel=keys)
    sel_rows = [(b * s.Hkv + h) * s.N + t for (b, h, t) in keys]
    rep = compare(o, qn, kn, pyr, ref, g["idx"][sel_rows], g["score"][sel_rows], g["trace"][sel_rows], keys,
                  Report())
    print(rep)
    assert rep.ok(), str(rep)
    return g, rep


def test_tiny_fp32_prefix(pisa):
    s = W.TINY
    q, k = W.iid(s, 0)
    prefix_parity(pisa, s, q, k)


def test_pretrain_planted_prefix(pisa):
    s = W.PRETRAIN
    q, k = W.planted(s, 1)
    _, rep = prefix_parity(pisa, s, q, k)
    assert rep.exempt < 0.2 * rep.n


@pytest.mark.parametrize("N,Hq,Hkv,d,K,dtype", [
    (4096 + 37, 16, 4, 128, 8, "bf16"),   # ragged tail, difference-row routing
    (2048 + 1, 8, 1, 64, 5, "bf16"),      # G = 8, d = 64: CUDA-core routing
    (3333, 4, 2, 128, 3, "fp32"),         # G = 2, fp32
    (5000, 8, 2, 64, 32, "bf16"),         # K = 32, difference-row routing, d = 64
    (3000, 4, 4, 128, 4, "bf16"),         # G = 1
])
def test_prefix_shapes(pisa, N, Hq, Hkv, d, K, dtype):
    s = W.Shape(B=2, N=N, Hq=Hq, Hkv=Hkv, d=d, K=K, dtype=dtype)
    q, k = W.iid(s, N % 89)
    prefix_parity(pisa, s, q, k)


def test_prefix_selection_ignores_later_keys(pisa):
    s = W.Shape(B=1, N=4096, Hq=16, Hkv=4, d=128, K=8)
    q, k = W.iid(s, 61)
    T = 2500
    k2 = k.float().clone()
    k2[:, :, T:] = 3.0 * torch.randn(k2[:, :, T:].shape, generator=torch.Generator().manual_seed(5))
    k2 = k2.to(s.torch_dtype)
    rows = [h * s.N + t for h in range(s.Hkv) for t in range(T)]
    o = oracle.Oracle.from_shape(s, prefix=True)
    keys = [(0, h, t) for h in range(s.Hkv) for t in range(T)]
    qn = q.double().numpy()
    for kk in (k, k2):
        g = run_prefix(pisa, s, q, kk)
        kn = kk.double().numpy()
        pyr = o.pyramid(kn)
        ref = o.select(qn, kn, pyr, sel=keys)
        rep = compare(o, qn, kn, pyr, ref, g["idx"][rows], g["score"][rows], g["trace"][rows], keys, Report())
        assert rep.ok(), str(rep)
        if kk is k:
            first = ref
    # the oracle's answers for t < T do not depend on the later keys
    assert (ref["idx"] == first["idx"]).all()
