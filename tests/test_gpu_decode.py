"""GPU parity of the single-launch decode step: incremental pyramid update
(bit-identical to a fresh build) and selection for the new query, against the
fp64 oracle, through the C ABI."""
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


def lens_tensor(lens):
    return torch.tensor(lens, dtype=torch.int32, device="cuda")


def run_steps(pisa, s, q_steps, kc, lens0, steps, check_rebuild=True):
    """Build the pyramid for lens0 - 1 keys, then run `steps` decode steps.
    Returns per-step (lens, idx, score, trace)."""
    p = pisa.params_from_shape(s)
    sel = pisa.Selector(p, mode="decode")
    kcd = kc.cuda()
    sel.build(kcd, lens_tensor([n - 1 for n in lens0]))
    L = pisa.pyramid_levels(p)
    out = []
    for st in range(steps):
        lens = [n + st for n in lens0]
        tr = torch.full((s.B, s.Hkv, L, s.K), -7, dtype=torch.int32, device="cuda")
        sel.decode(q_steps[st].cuda(), kcd, lens_tensor(lens), trace=tr)
        torch.cuda.synchronize()
        assert sel.device_status() == 0
        if check_rebuild:
            fresh = torch.empty_like(sel.pyramid)
            pisa.build_pyramid(p, kcd, fresh, lens_tensor(lens))
            torch.cuda.synchronize()
            assert torch.equal(fresh, sel.pyramid), f"step {st}: incremental pyramid != rebuild"
        W_ = s.K + 3
        out.append((lens, sel.out_idx.reshape(-1, W_).cpu().numpy(),
                    sel.out_score.reshape(-1, W_).cpu().double().numpy(),
                    tr.reshape(s.B * s.Hkv, L, s.K).cpu().numpy()))
    return out


def check_steps(s, q_steps, kc, results):
    o = oracle.Oracle.from_shape(s)
    kn = kc.double().numpy()
    rep = Report()
    for st, (lens, idx, score, trace) in enumerate(results):
        qn = q_steps[st].double().numpy()
        pyr = o.pyramid(kn, lens)
        ref = o.select(qn, kn, pyr, seq_lens=lens, decode=True)
        keys = [(b, h, lens[b] - 1) for b in range(s.B) for h in range(s.Hkv)]
        compare(o, qn, kn, pyr, ref, idx, score, trace, keys, rep, qmode="decode", lengths=lens)
    print(rep)
    assert rep.ok(), str(rep)


@pytest.mark.parametrize("d,G,K,dtype", [(128, 4, 8, "bf16"), (128, 4, 32, "bf16"), (64, 1, 4, "bf16"),
                                         (128, 2, 8, "fp32"), (64, 8, 16, "bf16")])
def test_decode_steps_match_oracle_and_rebuild(pisa, d, G, K, dtype):
    s = W.Shape(B=5, N=4096 + 64, Hq=2 * G, Hkv=2, d=d, K=K, dtype=dtype)
    q_steps, kc = W.decode_inputs(s, 11 + K, steps=6)
    # lengths that start a new leaf, end one, grow the tree, and tiny ones
    lens0 = [4096 + 1, 2048 + 64, 1025, 130, 3]
    results = run_steps(pisa, s, q_steps, kc, lens0, 6)
    check_steps(s, q_steps, kc, results)


def test_decode_bad_lengths_set_status(pisa):
    s = W.Shape(B=3, N=1024, Hq=4, Hkv=1, d=128, K=4)
    q_steps, kc = W.decode_inputs(s, 3, steps=1)
    p = pisa.params_from_shape(s)
    sel = pisa.Selector(p, mode="decode")
    kcd = kc.cuda()
    sel.build(kcd, lens_tensor([500, 500, 500]))
    sel.decode(q_steps[0].cuda(), kcd, lens_tensor([501, 0, 1025]))
    torch.cuda.synchronize()
    assert sel.device_status() == pisa.DEV_BAD_SEQ_LEN
    idx = sel.out_idx.cpu()
    assert (idx[1] == -1).all() and (idx[2] == -1).all()
    assert (idx[0, 0, 0] == 0).item()


def test_decode_full_size_sampled(pisa):
    """The decode workload at full size (64 sequences, 131072 cached keys,
    32/8 heads, K = 32): 16 steps from position 131072 (the first step opens
    leaf 2048 and adds a level).  Every step is checked for 3 sampled
    (sequence, key head) pairs; the pyramid after the last step must equal a
    fresh build bit for bit."""
    s = W.DECODE
    g = torch.Generator(device="cuda")
    g.manual_seed(4)
    kcd = torch.randn(s.B, s.Hkv, s.N, s.d, device="cuda", generator=g, dtype=torch.bfloat16)
    qd = torch.randn(W.DECODE_STEPS, s.B, s.Hq, s.d, device="cuda", generator=g, dtype=torch.bfloat16)
    p = pisa.params_from_shape(s)
    sel = pisa.Selector(p, mode="decode")
    L = pisa.pyramid_levels(p)
    sel.build(kcd, lens_tensor([W.DECODE_CACHED] * s.B))
    picks = [(0, 0), (17, 5), (63, 7)]
    kn = {bh: kcd[bh[0], bh[1]].double().cpu().numpy()[None, None] for bh in picks}
    rep = Report()
    for st in range(W.DECODE_STEPS):
        n = W.DECODE_CACHED + 1 + st
        tr = torch.full((s.B, s.Hkv, L, s.K), -7, dtype=torch.int32, device="cuda")
        sel.decode(qd[st], kcd, lens_tensor([n] * s.B), trace=tr)
        torch.cuda.synchronize()
        assert sel.device_status() == 0
        W_ = s.K + 3
        idx = sel.out_idx.cpu().numpy()
        sc = sel.out_score.cpu().double().numpy()
        trn = tr.cpu().numpy()
        for (b, h) in picks:
            o = oracle.Oracle(1, n, s.G, 1, s.d, s.C, s.K)
            kk = kn[(b, h)][:, :, :n]
            qrow = qd[st, b, h * s.G:(h + 1) * s.G].double().cpu().numpy()[None]
            pyr = o.pyramid(kk)
            ref = o.select(qrow, kk, pyr, sel=[(0, 0, n - 1)], qrows=True)
            compare(o, qrow, kk, pyr, ref, idx[b, h][None], sc[b, h][None], trn[b, h][None],
                    [(0, 0, n - 1)], rep, qmode="rows")
    print(rep)
    assert rep.ok(), str(rep)
    fresh = torch.empty_like(sel.pyramid)
    pisa.build_pyramid(p, kcd, fresh, lens_tensor([W.DECODE_CACHED + W.DECODE_STEPS] * s.B))
    torch.cuda.synchronize()
    assert torch.equal(fresh, sel.pyramid)


def test_decode_nonfinite_keys_stay_well_formed(pisa):
    """Cache keys holding NaN and +-inf: the decode walk and its leaf Top-K
    rank NaN scores as -inf, so each sequence still gets its forced blocks
    plus exactly min(K, |E|) causal blocks and the status stays clear."""
    from parity import check_structure
    s = W.Shape(B=3, N=4096, Hq=8, Hkv=2, d=128, K=8)
    q_steps, kc = W.decode_inputs(s, 23, steps=2)
    kc = kc.float()
    kc[0, 0, 64 * 7:64 * 8] = float("nan")
    kc[1, 1, 64 * 20 + 5, 3] = float("inf")
    kc[2, 0, 64 * 30:64 * 31, :8] = -float("inf")
    kc = kc.to(torch.bfloat16)
    lens0 = [4000, 3000, 2500]
    results = run_steps(pisa, s, q_steps, kc, lens0, 2, check_rebuild=False)
    rep = Report()
    for lens, idx, _, _ in results:
        for b in range(s.B):
            for h in range(s.Hkv):
                ok = check_structure(idx[b * s.Hkv + h], None, lens[b] - 1, s.C, s.K, rep, f"(b={b},h={h})")
                assert ok, rep.failures
