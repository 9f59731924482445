"""Bounded device waits end in a status, not a hang: with the test-only
injection pisa_test_inject_leaf_timeout, the first CTA of the tcgen05 leaf
kernel announces its first key tile but never copies it, so the MMA issuer's
wait on that stage can only run out (after a 2 ms limit here).  The call must
come back, the workspace status word must read PISA_DEV_TIMEOUT, the GPU must
stay usable, and the next call with the injection cleared must select exactly
as the oracle does.  The fault is made on the host side (a copy that is never
issued); no trap, no bad address, nothing left in flight when the kernel
returns."""
import numpy as np
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


def test_exhausted_leaf_wait_sets_the_timeout_status_and_recovers(pisa):
    s = W.Shape(B=1, N=4096 + 37, Hq=16, Hkv=4, d=128, K=8)
    q, k = W.iid(s, 23)
    p = pisa.params_from_shape(s)
    sel = pisa.Selector(p)
    qd, kd = q.cuda(), k.cuda()
    lib = pisa.lib()
    try:
        lib.pisa_test_inject_leaf_timeout(2_000_000, 1)
        sel.prefill(qd, kd)
        torch.cuda.synchronize()
        assert sel.device_status() == pisa.DEV_TIMEOUT
    finally:
        lib.pisa_test_inject_leaf_timeout(0, 0)
    # the context is intact: plain work and a clean selection afterwards
    x = torch.arange(1 << 20, device="cuda", dtype=torch.float32)
    assert float(x.sum().item()) == float((1 << 20) * ((1 << 20) - 1) // 2)
    sel.prefill(qd, kd)
    torch.cuda.synchronize()
    assert sel.device_status() == 0
    o = oracle.Oracle.from_shape(s)
    qn, kn = q.double().numpy(), k.double().numpy()
    pyr = o.pyramid(kn)
    ref = o.select(qn, kn, pyr)
    keys = [(0, h, t) for h in range(s.Hkv) for t in range(s.N)]
    W_ = s.K + 3
    idx = sel.out_idx.reshape(-1, W_).cpu().numpy()
    score = sel.out_score.reshape(-1, W_).cpu().double().numpy()
    rep = compare(o, qn, kn, pyr, ref, idx, score, None, keys, Report())
    # without a trace a tie-exempt differing query would be reported; allow
    # only those, and demand no other failure
    bad = [f for f in rep.failures if "without a trace" not in f]
    assert not bad, str(rep)
    assert rep.exact >= 0.99 * rep.n
