"""GPU tests of the paged key cache (pisa_build_pyramid_paged,
pisa_select_decode_paged): pages of C keys [num_pages, H_kv, C, d] placed
in a shuffled pool with unused pages filled with large values.  The paged
calls must equal the contiguous calls on the same keys bit for bit (pyramid,
indices, scores, traces) and the fp64 oracle; a page index outside the pool
sets PISA_DEV_BAD_INDEX without being read."""
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


def paginate(kc, C, extra, seed):
    """Scatter a contiguous cache [B, Hkv, N, d] into a shuffled page pool."""
    B, Hkv, N, d = kc.shape
    npb = -(-N // C)
    num_pages = B * npb + extra
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(num_pages, generator=g)[:B * npb].reshape(B, npb).to(torch.int32)
    pages = torch.full((num_pages, Hkv, C, d), 4096.0, dtype=kc.dtype)
    padded = torch.zeros(B, Hkv, npb * C, d, dtype=kc.dtype)
    padded[:, :, :N] = kc
    for b in range(B):
        pages[perm[b].long()] = padded[b].reshape(Hkv, npb, C, d).permute(1, 0, 2, 3)
    return pages, perm


@pytest.mark.parametrize("d,G,K,dtype", [(128, 4, 8, "bf16"), (64, 2, 4, "fp32"), (128, 8, 16, "bf16")])
def test_paged_decode_equals_contiguous_and_oracle(pisa, d, G, K, dtype):
    s = W.Shape(B=5, N=4096 + 64, Hq=2 * G, Hkv=2, d=d, K=K, dtype=dtype)
    q_steps, kc = W.decode_inputs(s, 90 + K, steps=4)
    lens0 = [4096 + 1, 2048 + 64, 1025, 130, 3]
    pages, table = paginate(kc, s.C, extra=9, seed=K)
    p = pisa.params_from_shape(s)
    a = pisa.Selector(p, mode="decode")
    bsel = pisa.Selector(p, mode="decode")
    kcd, pgd, tbd = kc.cuda(), pages.cuda(), table.cuda()
    pre = torch.tensor([n - 1 for n in lens0], dtype=torch.int32, device="cuda")
    a.build(kcd, pre)
    bsel.build_paged(pgd, tbd, pre)
    torch.cuda.synchronize()
    assert bsel.device_status() == 0
    assert torch.equal(a.pyramid, bsel.pyramid), "paged build differs from the contiguous build"
    L = pisa.pyramid_levels(p)
    o = oracle.Oracle.from_shape(s)
    kn = kc.double().numpy()
    rep = Report()
    for st in range(4):
        lens = [n + st for n in lens0]
        ld = torch.tensor(lens, dtype=torch.int32, device="cuda")
        ta = torch.full((s.B, s.Hkv, L, s.K), -7, dtype=torch.int32, device="cuda")
        tb = torch.full_like(ta, -7)
        a.decode(q_steps[st].cuda(), kcd, ld, trace=ta)
        bsel.decode_paged(q_steps[st].cuda(), pgd, tbd, ld, trace=tb)
        torch.cuda.synchronize()
        assert a.device_status() == 0 and bsel.device_status() == 0
        assert torch.equal(a.out_idx, bsel.out_idx)
        assert torch.equal(a.out_score, bsel.out_score)
        assert torch.equal(ta, tb)
        assert torch.equal(a.pyramid, bsel.pyramid)
        W_ = s.K + 3
        qn = q_steps[st].double().numpy()
        pyr = o.pyramid(kn, lens)
        ref = o.select(qn, kn, pyr, seq_lens=lens, decode=True)
        keys = [(b, h, lens[b] - 1) for b in range(s.B) for h in range(s.Hkv)]
        compare(o, qn, kn, pyr, ref, bsel.out_idx.reshape(-1, W_).cpu().numpy(),
                bsel.out_score.reshape(-1, W_).cpu().double().numpy(),
                tb.reshape(s.B * s.Hkv, L, s.K).cpu().numpy(), keys, rep, qmode="decode", lengths=lens)
    print(rep)
    assert rep.ok(), str(rep)


def test_page_outside_the_pool_sets_status_and_is_not_read(pisa):
    s = W.Shape(B=3, N=1024, Hq=4, Hkv=1, d=128, K=4)
    q_steps, kc = W.decode_inputs(s, 5, steps=1)
    pages, table = paginate(kc, s.C, extra=0, seed=1)
    bad = table.clone()
    bad[1, 3] = pages.shape[0] + 5   # sequence 1, leaf 3: outside the pool
    p = pisa.params_from_shape(s)
    sel = pisa.Selector(p, mode="decode")
    lens = torch.tensor([700, 600, 500], dtype=torch.int32, device="cuda")
    sel.build_paged(pages.cuda(), bad.cuda(), lens - 1)
    torch.cuda.synchronize()
    assert sel.device_status() == pisa.DEV_BAD_INDEX
    sel.build_paged(pages.cuda(), table.cuda(), lens - 1)
    sel.decode_paged(q_steps[0].cuda(), pages.cuda(), bad.cuda(), lens)
    torch.cuda.synchronize()
    assert sel.device_status() == pisa.DEV_BAD_INDEX
    idx = sel.out_idx.cpu()
    assert (idx[1] == -1).all()            # the bad sequence is left empty
    assert (idx[0, 0, 0] == 0).item() and (idx[2, 0, 0] == 0).item()  # the others are selected
