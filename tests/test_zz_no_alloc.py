"""The allocation-free prefill entry point, pisa_select_prefill_static.

Some callers cannot allocate device memory at the point where they select
blocks: code running inside a runtime that owns every device allocation (a
plug-in or a host callback that may not call cudaMalloc or a framework
allocator).  For them the library keeps its prefill workspace in one fixed
device array.  This test calls that entry point through the C ABI twice in a
row, on two different inputs, and checks each result against the regular
pisa_select_prefill (which uses a caller-owned workspace): identical block
indices and scores within the tests' 2e-3 tolerance.  It also checks that a
problem whose workspace exceeds the fixed array is refused.

This file is collected last on purpose (tests/test_zz_*), and it passes both
alone in a fresh process and after the other GPU tests.
"""
import ctypes

import numpy as np
import pytest
import torch

from pyramid_top_block_mean_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SCORE_TOL = 2e-3


@pytest.fixture(scope="module")
def pisa():
    from pyramid_top_block_mean_gb300 import pisa as m
    f = m.lib().pisa_select_prefill_static
    f.argtypes = [ctypes.POINTER(m.Params)] + [ctypes.c_void_p] * 6
    f.restype = ctypes.c_int
    return m


def _static_call(pisa, p, q, k, pyr, idx, score):
    st = torch.cuda.current_stream()
    return pisa.lib().pisa_select_prefill_static(ctypes.byref(p), q.data_ptr(), k.data_ptr(), pyr.data_ptr(),
                                                 idx.data_ptr(), score.data_ptr(), st.cuda_stream)


def test_static_workspace_matches_regular_entry_point_twice(pisa):
    s = W.PRETRAIN
    p = pisa.params_from_shape(s)
    for seed in (21, 22):  # two calls in a row on different inputs
        q, k = W.planted(s, seed)
        q, k = q.cuda(), k.cuda()
        ref = pisa.Selector(p)
        ref.prefill(q, k)
        idx = torch.full_like(ref.out_idx, -7)
        score = torch.full_like(ref.out_score, float("nan"))
        assert _static_call(pisa, p, q, k, ref.pyramid, idx, score) == pisa.PISA_OK
        torch.cuda.synchronize()
        assert torch.equal(idx, ref.out_idx)
        a = score.cpu().double().numpy()
        b = ref.out_score.cpu().double().numpy()
        fin = np.isfinite(b)
        assert (np.isinf(a) == ~fin).all()
        assert np.abs(a[fin] - b[fin]).max() <= SCORE_TOL


def test_static_workspace_refuses_too_large_problems(pisa):
    s = W.sweep(262144)
    p = pisa.params_from_shape(s)
    assert pisa.workspace_bytes(p, pisa.MODE_PREFILL) > (64 << 20)
    dummy = torch.empty(16, dtype=torch.uint8, device="cuda")
    rc = _static_call(pisa, p, dummy, dummy, dummy, dummy, dummy)
    assert rc == -4  # PISA_ERR_WORKSPACE, and nothing was launched
