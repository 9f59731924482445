"""The allocation-free prefill entry point, pisa_select_prefill_static.

Some callers cannot allocate device memory at the point where they select
blocks: code running inside a runtime that owns every device allocation (a
plug-in or a host callback that may not call cudaMalloc or a framework
allocator).  For them the library keeps its prefill workspace in one fixed
device array.  This test calls that entry point through the C ABI twice in a
row, on two different inputs, and checks each result against the regular
pisa_select_prefill (which uses a caller-owned workspace).  Both run the same
kernels on the same inputs, so indices and scores must be bit-identical.
Between the two checked calls a third call on another shape leaves different
contents in the shared array, so a region that a call forgot to clear would
show up as a difference.  The array's device status word must stay clear.
It also checks that a problem whose workspace exceeds the fixed array is
refused.

This file is collected last on purpose (tests/test_zz_*), and it passes both
alone in a fresh process and after the other GPU tests.
"""
import ctypes

import pytest
import torch

from pyramid_top_block_mean_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pisa():
    from pyramid_top_block_mean_gb300 import pisa as m
    return m


def _static_call(pisa, p, q, k, pyr, idx, score):
    st = torch.cuda.current_stream()
    return pisa.lib().pisa_select_prefill_static(ctypes.byref(p), q.data_ptr(), k.data_ptr(), pyr.data_ptr(),
                                                 idx.data_ptr(), score.data_ptr(), st.cuda_stream)


def _static_status(pisa):
    code = ctypes.c_int32(-1)
    rc = pisa.lib().pisa_read_static_status(ctypes.byref(code), torch.cuda.current_stream().cuda_stream)
    return rc, code.value


def _filler_call(pisa):
    """A call on another shape (ragged, other K and G) that leaves its own
    contents in the shared array."""
    s = W.Shape(B=1, N=3000 + 17, Hq=8, Hkv=1, d=128, K=5)
    q, k = W.iid(s, 77)
    p = pisa.params_from_shape(s)
    sel = pisa.Selector(p)
    sel.build(k.cuda())
    idx = torch.empty_like(sel.out_idx)
    score = torch.empty_like(sel.out_score)
    assert _static_call(pisa, p, q.cuda(), k.cuda(), sel.pyramid, idx, score) == pisa.PISA_OK


def test_static_workspace_matches_regular_entry_point_twice(pisa):
    s = W.PRETRAIN
    p = pisa.params_from_shape(s)
    for n, seed in enumerate((21, 22)):  # two checked calls in a row on different inputs
        if n == 1:
            _filler_call(pisa)
        q, k = W.planted(s, seed)
        q, k = q.cuda(), k.cuda()
        ref = pisa.Selector(p)
        ref.prefill(q, k)
        idx = torch.full_like(ref.out_idx, -7)
        score = torch.full_like(ref.out_score, float("nan"))
        assert _static_call(pisa, p, q, k, ref.pyramid, idx, score) == pisa.PISA_OK
        torch.cuda.synchronize()
        assert _static_status(pisa) == (pisa.PISA_OK, 0)
        assert torch.equal(idx, ref.out_idx)
        assert torch.equal(score, ref.out_score)


def test_static_workspace_refuses_too_large_problems(pisa):
    s = W.sweep(262144)
    p = pisa.params_from_shape(s)
    assert pisa.workspace_bytes(p, pisa.MODE_PREFILL) > (64 << 20)
    dummy = torch.empty(16, dtype=torch.uint8, device="cuda")
    rc = _static_call(pisa, p, dummy, dummy, dummy, dummy, dummy)
    assert rc == -4  # PISA_ERR_WORKSPACE, and nothing was launched
