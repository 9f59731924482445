"""GPU parity of the PISA-1 and PISA-2 block scorers (pisa_params.scorer)
against the fp64 oracle, through the C ABI: prefill on both routing kernels
(tensor-core bf16 with G = 4, CUDA-core for fp32 or other G) and both leaf
kernels, and the decode step (bf16 tensor-core leaves and fp32 leaves).  The
tie-aware comparison of tests/parity.py applies unchanged: the oracle scores
every level with the same scorer."""
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


@pytest.mark.parametrize("scorer", [1, 2])
@pytest.mark.parametrize("N,Hq,Hkv,d,K,dtype", [(4096 + 37, 16, 4, 128, 8, "bf16"),
                                                (2049, 4, 2, 64, 5, "fp32"),
                                                (3000, 16, 2, 128, 8, "bf16")])
def test_prefill_scorers_match_oracle(pisa, scorer, N, Hq, Hkv, d, K, dtype):
    s = W.Shape(B=2, N=N, Hq=Hq, Hkv=Hkv, d=d, K=K, dtype=dtype)
    q, k = W.iid(s, 50 + scorer)
    p = pisa.params_from_shape(s, scorer=scorer)
    sel = pisa.Selector(p)
    L = pisa.pyramid_levels(p)
    tr = torch.full((s.B, s.Hkv, s.N, L, s.K), -7, dtype=torch.int32, device="cuda")
    sel.prefill(q.cuda(), k.cuda(), trace=tr)
    torch.cuda.synchronize()
    assert sel.device_status() == 0
    W_ = s.K + 3
    o = oracle.Oracle.from_shape(s, scorer=scorer)
    qn, kn = q.double().numpy(), k.double().numpy()
    pyr = o.pyramid(kn)
    ref = o.select(qn, kn, pyr)
    keys = [(b, h, t) for b in range(s.B) for h in range(s.Hkv) for t in range(s.N)]
    rep = compare(o, qn, kn, pyr, ref, sel.out_idx.reshape(-1, W_).cpu().numpy(),
                  sel.out_score.reshape(-1, W_).cpu().double().numpy(),
                  tr.reshape(s.B * s.Hkv * s.N, L, s.K).cpu().numpy(), keys, Report())
    print(rep)
    assert rep.ok(), str(rep)
    # the scorer changes the selection: some query differs from the LSE walk
    lse = oracle.Oracle.from_shape(s).select(qn, kn, pyr)["idx"]
    assert (lse != ref["idx"]).any(axis=1).mean() > 0.01


@pytest.mark.parametrize("scorer", [1, 2])
@pytest.mark.parametrize("d,G,K,dtype", [(128, 4, 8, "bf16"), (128, 2, 8, "fp32")])
def test_decode_scorers_match_oracle(pisa, scorer, d, G, K, dtype):
    s = W.Shape(B=5, N=4096 + 64, Hq=2 * G, Hkv=2, d=d, K=K, dtype=dtype)
    q_steps, kc = W.decode_inputs(s, 70 + scorer, steps=3)
    lens0 = [4096 + 1, 2048 + 64, 1025, 130, 3]
    p = pisa.params_from_shape(s, scorer=scorer)
    sel = pisa.Selector(p, mode="decode")
    kcd = kc.cuda()
    sel.build(kcd, torch.tensor([n - 1 for n in lens0], dtype=torch.int32, device="cuda"))
    L = pisa.pyramid_levels(p)
    o = oracle.Oracle.from_shape(s, scorer=scorer)
    kn = kc.double().numpy()
    rep = Report()
    for st in range(3):
        lens = [n + st for n in lens0]
        tr = torch.full((s.B, s.Hkv, L, s.K), -7, dtype=torch.int32, device="cuda")
        sel.decode(q_steps[st].cuda(), kcd, torch.tensor(lens, dtype=torch.int32, device="cuda"), trace=tr)
        torch.cuda.synchronize()
        assert sel.device_status() == 0
        W_ = s.K + 3
        qn = q_steps[st].double().numpy()
        pyr = o.pyramid(kn, lens)
        ref = o.select(qn, kn, pyr, seq_lens=lens, decode=True)
        keys = [(b, h, lens[b] - 1) for b in range(s.B) for h in range(s.Hkv)]
        compare(o, qn, kn, pyr, ref, sel.out_idx.reshape(-1, W_).cpu().numpy(),
                sel.out_score.reshape(-1, W_).cpu().double().numpy(),
                tr.reshape(s.B * s.Hkv, L, s.K).cpu().numpy(), keys, rep, qmode="decode", lengths=lens)
    print(rep)
    assert rep.ok(), str(rep)
