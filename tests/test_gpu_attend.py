"""GPU parity of block-sparse attention over a selection (pisa_attend_prefill
for every query position, pisa_attend_decode for one decode query per
sequence) against the fp64 oracle, through the C ABI.

Tolerance.  The kernel rounds three times to bf16: the probabilities fed to
the P V product (relative 2^-9 each, so at most 2^-9 max|v| on a block's
normalised output), each block's normalised partial (2^-9 of a convex
combination of values) and the final output (2^-9 |o|).  The fp32 score
accumulation and ex2/lg2 approximations add relative errors near 1e-5 to the
weights.  The bound used is 3 * 2^-9 * max|v| + 1e-4 per element.  The
decode kernel keeps its running output in fp32 and rounds only P and the
output, so the same bound covers it.
"""
import numpy as np
import pytest
import torch

import oracle
from pyramid_top_block_mean_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pisa():
    from pyramid_top_block_mean_gb300 import pisa as m
    return m


def tol(v):
    return 3 * 2.0 ** -9 * float(v.abs().max()) + 1e-4


def select(pisa, s, q, k):
    p = pisa.params_from_shape(s)
    sel = pisa.Selector(p, with_scores=False)
    idx, _ = sel.prefill(q, k)
    torch.cuda.synchronize()
    assert sel.device_status() == 0
    return idx


def attend(pisa, s, q, k, v, idx):
    p = pisa.params_from_shape(s)
    at = pisa.Attention(p)
    out = at(q, k, v, idx)
    torch.cuda.synchronize()
    assert at.device_status() == 0
    return out


def to_heads(o, s):
    """oracle [B*Hkv*N, G, d] -> [B, Hq, N, d]"""
    G = s.Hq // s.Hkv
    t = torch.from_numpy(o).reshape(s.B, s.Hkv, s.N, G, s.d).permute(0, 1, 3, 2, 4)
    return t.reshape(s.B, s.Hq, s.N, s.d)


def check_full(pisa, s, seed, idx=None):
    q, k = W.iid(s, seed)
    v = W.values(s, seed)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    if idx is None:
        idx = select(pisa, s, qc, kc)
    out = attend(pisa, s, qc, kc, vc, idx.cuda())
    ref = to_heads(oracle.Oracle.from_shape(s).attend(q, k, v, idx.cpu().numpy()), s)
    err = (out.cpu().double() - ref).abs().max().item()
    print(f"N={s.N} d={s.d} G={s.G} K={s.K}: max err {err:.3e} (tol {tol(v):.3e})")
    assert err <= tol(v), err
    return out, ref


@pytest.mark.parametrize("N,Hq,Hkv,d,K", [(1000, 16, 4, 128, 8), (4096 + 37, 8, 2, 128, 8),
                                          (3000, 4, 4, 64, 4), (2048 + 1, 16, 2, 64, 8),
                                          (700, 4, 2, 128, 2), (1, 4, 1, 128, 8), (65, 8, 4, 64, 8)])
def test_attend_matches_oracle_on_selector_output(pisa, N, Hq, Hkv, d, K):
    s = W.Shape(B=2, N=N, Hq=Hq, Hkv=Hkv, d=d, K=K)
    check_full(pisa, s, seed=N + d)


def test_attend_K32_slots_above_31(pisa):
    # 35 slots per query: the pair encoding needs six slot bits
    s = W.Shape(B=1, N=5000, Hq=16, Hkv=4, d=128, K=32)
    check_full(pisa, s, seed=3)


def test_attend_hand_made_rows(pisa):
    """Empty and out-of-range slots, repeated blocks, blocks after the
    query's own block, rows with no key at all, unsorted rows."""
    s = W.Shape(B=1, N=640, Hq=8, Hkv=2, d=128, K=4)
    Wd = s.K + 3
    nb = -(-s.N // s.C)
    g = torch.Generator().manual_seed(7)
    idx = torch.randint(-3, nb + 3, (s.B, s.Hkv, s.N, Wd), generator=g, dtype=torch.int32)
    t = torch.arange(s.N)
    idx[..., 0] = (t // s.C).to(torch.int32)      # the query's own block: every row has key t
    idx[..., 1] = idx[..., 2]                      # a repeated block
    idx[0, 1, 100:110, :] = -1                     # rows with no block at all
    idx[0, 1, 100:110, 3] = 9                      # ... or only a future block (query blocks 1)
    q, k = W.iid(s, 11)
    v = W.values(s, 11)
    out = attend(pisa, s, q.cuda(), k.cuda(), v.cuda(), idx.cuda()).cpu().double()
    # rows with no attended key are zero
    assert (out[0, 4:8, 100:110] == 0).all()
    # every other row against the oracle (which rejects key-less rows)
    keep = [(0, h, tt) for h in range(s.Hkv) for tt in range(s.N) if not (h == 1 and 100 <= tt < 110)]
    o = oracle.Oracle.from_shape(s)
    ref = o.attend(q, k, v, idx.numpy(), sel=keep)
    G = s.G
    got = torch.stack([out[0, h * G:(h + 1) * G, tt] for (_, h, tt) in keep]).numpy()
    err = np.abs(got - ref).max()
    assert err <= tol(v), err


def test_attend_flat_selection(pisa):
    # the flat comparator's output drives the same attention
    s = W.Shape(B=1, N=3000, Hq=16, Hkv=4, d=128, K=8)
    q, k = W.iid(s, 19)
    p = pisa.params_from_shape(s)
    sel = pisa.Selector(p, mode="flat", with_scores=False)
    idx, _ = sel.flat(q.cuda(), k.cuda())
    torch.cuda.synchronize()
    check_full(pisa, s, seed=19, idx=idx.clone())


@pytest.mark.parametrize("N", [65536, 262144])
def test_attend_full_size_sampled(pisa, N):
    """The benchmark's workload: the selector's output at N tokens, the
    attention over it, and 192 sampled queries (first blocks, the ragged
    middle, the last positions) against the oracle."""
    s = W.sweep(N)
    q, k = W.iid(s, 1)
    v = W.values(s, 1)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    idx = select(pisa, s, qc, kc)
    out = attend(pisa, s, qc, kc, vc, idx)
    rng = np.random.default_rng(N)
    ts = list(range(0, 40)) + list(rng.integers(0, N, 112)) + list(range(N - 40, N))
    sel = [(0, int(rng.integers(0, s.Hkv)), int(t)) for t in ts]
    G = s.G
    rows = np.stack([q[0, h * G:(h + 1) * G, t].double().numpy() for (_, h, t) in sel])
    o = oracle.Oracle.from_shape(s)
    ref = o.attend(rows, k, v, idx.cpu().numpy(), sel=sel, qrows=True)
    outc = out.cpu()
    got = torch.stack([outc[0, h * G:(h + 1) * G, t] for (_, h, t) in sel]).double().numpy()
    err = np.abs(got - ref).max()
    print(f"N={N}: max err {err:.3e} over {len(sel)} queries (tol {tol(v):.3e})")
    assert err <= tol(v), err


def decode_reference(s, qd, kc, v, lens, idx_rows):
    """The oracle's attention for the decode queries: the idx rows [B, Hkv, W]
    placed at t = len - 1 of a full -1 array, q passed as rows."""
    Wd = s.K + 3
    full = np.full((s.B, s.Hkv, s.N, Wd), -1, np.int32)
    sel = []
    for b in range(s.B):
        for h in range(s.Hkv):
            full[b, h, lens[b] - 1] = idx_rows[b, h]
            sel.append((b, h, lens[b] - 1))
    G = s.G
    rows = np.stack([qd[b, h * G:(h + 1) * G].double().numpy() for (b, h, _) in sel])
    o = oracle.Oracle.from_shape(s)
    return o.attend(rows, kc, v, full, sel=sel, qrows=True)  # [B*Hkv, G, d]


@pytest.mark.parametrize("d,G,K", [(128, 4, 8), (64, 2, 4), (128, 8, 32), (64, 1, 16)])
def test_attend_decode_matches_oracle(pisa, d, G, K):
    s = W.Shape(B=5, N=4096 + 64, Hq=2 * G, Hkv=2, d=d, K=K)
    q_steps, kc = W.decode_inputs(s, 30 + K, steps=1)
    v = W.values(s, 30 + K)
    lens = [4096 + 1, 2048 + 64, 1025, 130, 3]
    p = pisa.params_from_shape(s)
    sel = pisa.Selector(p, mode="decode", with_scores=False)
    kcd, vd = kc.cuda(), v.cuda()
    ld = torch.tensor(lens, dtype=torch.int32, device="cuda")
    sel.build(kcd, ld - 1)
    idx, _ = sel.decode(q_steps[0].cuda(), kcd, ld)
    at = pisa.Attention(p, mode="decode")
    out = at.decode(q_steps[0].cuda(), kcd, vd, ld, idx)
    torch.cuda.synchronize()
    assert sel.device_status() == 0 and at.device_status() == 0
    ref = decode_reference(s, q_steps[0], kc, v, lens, idx.cpu().numpy())
    got = out.cpu().double().numpy().reshape(s.B * s.Hkv, G, d)
    err = np.abs(got - ref).max()
    print(f"decode d={d} G={G} K={K}: max err {err:.3e} (tol {tol(v):.3e})")
    assert err <= tol(v), err


def test_attend_decode_hand_made_rows(pisa):
    s = W.Shape(B=4, N=1024, Hq=8, Hkv=2, d=128, K=4)
    q_steps, kc = W.decode_inputs(s, 8, steps=1)
    v = W.values(s, 8)
    lens = [1000, 640, 65, 1]
    Wd = s.K + 3
    g = torch.Generator().manual_seed(3)
    idx = torch.randint(-3, 20, (s.B, s.Hkv, Wd), generator=g, dtype=torch.int32)
    for b, n in enumerate(lens):
        idx[b, :, 0] = (n - 1) // 64  # the query's own block
        idx[b, :, 1] = idx[b, :, 0]   # repeated
    p = pisa.params_from_shape(s)
    at = pisa.Attention(p, mode="decode")
    ld = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = at.decode(q_steps[0].cuda(), kc.cuda(), v.cuda(), ld, idx.cuda())
    torch.cuda.synchronize()
    assert at.device_status() == 0
    ref = decode_reference(s, q_steps[0], kc, v, lens, idx.numpy())
    got = out.cpu().double().numpy().reshape(s.B * s.Hkv, s.G, s.d)
    err = np.abs(got - ref).max()
    assert err <= tol(v), err
