"""The C-ABI library loads, exports every entry point that include/pisa.h
declares, and rejects bad arguments on the host before any launch (these
calls never reach the GPU, so they run without one)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pisa():
    from pyramid_top_block_mean_gb300 import build
    build.build()
    from pyramid_top_block_mean_gb300 import pisa as m
    return m


def declared_functions():
    src = open(os.path.join(ROOT, "include", "pisa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pisa_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(pisa):
    names = declared_functions()
    assert len(names) >= 11
    for n in names:
        assert hasattr(pisa.lib(), n), n
    assert set(names) == set(pisa.EXPORTED)


def test_abi_version_and_status_strings(pisa):
    assert pisa.abi_version() == 3
    for code in range(-6, 1):
        assert pisa.status_string(code).startswith(pisa.STATUS_NAMES[code])


def test_size_queries_match_the_pyramid_shape(pisa):
    import oracle
    for N in [1, 63, 64, 65, 1000, 4096, 4096 + 37, 16384, 262144]:
        p = pisa.make_params(2, N, 16, 4, 128, K=8)
        assert pisa.pyramid_nodes(p) == oracle.lib().po_num_nodes(N, 64)
        assert pisa.pyramid_levels(p) == oracle.lib().po_num_levels(N, 64)
        assert pisa.pyramid_bytes(p) == 2 * 4 * pisa.pyramid_nodes(p) * 128 * 4
        for mode in (0, 1, 2, 3):
            assert pisa.workspace_bytes(p, mode) >= 256


@pytest.mark.parametrize("field,value,code", [
    ("H_q", 15, -1), ("H_kv", 0, -1), ("K", 0, -1), ("N", -1, -1), ("B", -1, -1), ("qtile", 0, -1),
    ("scale", -1.0, -1), ("d", 96, -2), ("C", 32, -2), ("g", 3, -2), ("K", 33, -2), ("dtype", 7, -2),
    ("H_q", 48, -2),  # G = 12
    ("N", (1 << 26) + 1, -2), ("struct_size", 8, -1), ("scorer", 3, -1), ("scorer", -1, -1),
    ("summaries", 2, -1), ("summaries", -1, -1),
])
def test_bad_params_are_rejected(pisa, field, value, code):
    p = pisa.make_params(1, 4096, 16, 4, 128, K=8)
    setattr(p, field, value)
    assert pisa.workspace_bytes(p, 0) == 0
    assert pisa.pyramid_nodes(p) == 0
    fake = ctypes.c_void_p(0x10000)
    rc = pisa.lib().pisa_select_prefill(ctypes.byref(p), fake, fake, fake, fake, 1 << 40, fake, None, None, None)
    assert rc == code


def test_null_misaligned_and_small_workspace_rejected_before_launch(pisa):
    L = pisa.lib()
    p = pisa.make_params(1, 4096, 16, 4, 128, K=8)
    a = ctypes.c_void_p(0x10000)
    mis = ctypes.c_void_p(0x10008)
    big = 1 << 40
    ws_need = pisa.workspace_bytes(p, 0)
    assert L.pisa_select_prefill(ctypes.byref(p), None, a, a, a, big, a, None, None, None) == -1
    assert L.pisa_select_prefill(ctypes.byref(p), mis, a, a, a, big, a, None, None, None) == -3
    assert L.pisa_select_prefill(ctypes.byref(p), a, a, a, a, ws_need - 1, a, None, None, None) == -4
    assert L.pisa_build_pyramid(ctypes.byref(p), None, None, a, None) == -1
    assert L.pisa_build_pyramid(ctypes.byref(p), mis, None, a, None) == -3
    assert L.pisa_select_decode(ctypes.byref(p), a, a, None, a, a, big, a, None, None, None) == -1
    assert L.pisa_select_decode(ctypes.byref(p), a, a, a, a, a, 16, a, None, None, None) == -4
    assert L.pisa_select_flat(ctypes.byref(p), a, a, a, 16, a, None, None) == -4
    assert L.pisa_select_flat(ctypes.byref(p), a, mis, a, big, a, None, None) == -3
    code = ctypes.c_int32(0)
    assert L.pisa_read_device_status(None, ctypes.byref(code), None) == -1


def test_empty_problems_are_no_ops(pisa):
    L = pisa.lib()
    for B, N in [(0, 4096), (1, 0)]:
        p = pisa.make_params(B, N, 16, 4, 128, K=8)
        assert L.pisa_select_prefill(ctypes.byref(p), None, None, None, None, 0, None, None, None, None) == 0
        assert L.pisa_build_pyramid(ctypes.byref(p), None, None, None, None) == 0


def test_params_without_the_summaries_field_are_rejected(pisa):
    # a caller built against the second ABI passes the shorter struct
    p = pisa.make_params(1, 4096, 16, 4, 128, K=8)
    p.struct_size = pisa.Params.summaries.offset
    assert pisa.workspace_bytes(p, 0) == 0
    base = pisa.workspace_bytes(pisa.make_params(1, 4096, 16, 4, 128, K=8), 0)
    pre = pisa.workspace_bytes(pisa.make_params(1, 4096, 16, 4, 128, K=8, summaries=pisa.SUMMARIES_PREFIX), 0)
    assert 0 < base < pre  # the prefix-consistent walk keeps its path dots in the workspace


def test_prefix_route_stage_alone_is_refused_before_launch(pisa):
    # prefix-consistent walks read each query's own raw keys, which only
    # pisa_select_prefill receives
    p = pisa.make_params(1, 4096, 16, 4, 128, K=8, summaries=pisa.SUMMARIES_PREFIX)
    a = ctypes.c_void_p(0x10000)
    assert pisa.lib().pisa_prefill_route(ctypes.byref(p), a, a, a, 1 << 40, None, None) == -2


def test_params_without_the_scorer_field_are_rejected(pisa):
    # a caller built against the first ABI passes the shorter struct
    p = pisa.make_params(1, 4096, 16, 4, 128, K=8)
    p.struct_size = pisa.Params.scorer.offset
    assert pisa.workspace_bytes(p, 0) == 0
    for sc in (0, 1, 2):
        assert pisa.workspace_bytes(pisa.make_params(1, 4096, 16, 4, 128, K=8, scorer=sc), 0) > 0


def test_paged_entry_points_check_their_pool_before_launch(pisa):
    L = pisa.lib()
    p = pisa.make_params(2, 4096, 16, 4, 128, K=8)
    a = ctypes.c_void_p(0x10000)
    mis = ctypes.c_void_p(0x10008)
    odd = ctypes.c_void_p(0x10002)
    big = 1 << 40
    # build: null table, no pages, misaligned pool or table, small workspace
    assert L.pisa_build_pyramid_paged(ctypes.byref(p), a, 10, None, None, a, a, big, None) == -1
    assert L.pisa_build_pyramid_paged(ctypes.byref(p), a, 0, a, None, a, a, big, None) == -1
    assert L.pisa_build_pyramid_paged(ctypes.byref(p), mis, 10, a, None, a, a, big, None) == -3
    assert L.pisa_build_pyramid_paged(ctypes.byref(p), a, 10, odd, None, a, a, big, None) == -3
    assert L.pisa_build_pyramid_paged(ctypes.byref(p), a, 10, a, None, a, a, 16, None) == -4
    # decode: the same, plus the decode arguments
    assert L.pisa_select_decode_paged(ctypes.byref(p), a, a, 10, None, a, a, a, big, a, None, None, None) == -1
    assert L.pisa_select_decode_paged(ctypes.byref(p), a, a, 0, a, a, a, a, big, a, None, None, None) == -1
    assert L.pisa_select_decode_paged(ctypes.byref(p), a, mis, 10, a, a, a, a, big, a, None, None, None) == -3
    assert L.pisa_select_decode_paged(ctypes.byref(p), a, a, 10, a, None, a, a, big, a, None, None, None) == -1


def test_attention_entry_points_check_their_arguments(pisa):
    L = pisa.lib()
    a = ctypes.c_void_p(0x10000)
    mis = ctypes.c_void_p(0x10008)
    big = 1 << 40
    p = pisa.make_params(2, 4096, 16, 4, 128, K=8)
    # prefill: null and misaligned pointers, a small workspace, fp32 inputs
    assert L.pisa_attend_prefill(ctypes.byref(p), a, a, None, a, a, big, a, None) == -1
    assert L.pisa_attend_prefill(ctypes.byref(p), a, a, mis, a, a, big, a, None) == -3
    assert L.pisa_attend_prefill(ctypes.byref(p), a, a, a, a, a, 16, a, None) == -4
    f32 = pisa.make_params(2, 4096, 16, 4, 128, K=8, dtype="fp32")
    assert L.pisa_attend_prefill(ctypes.byref(f32), a, a, a, a, a, big, a, None) == -2
    assert pisa.workspace_bytes(p, pisa.MODE_ATTEND) > 2 * 2 * 16 * 4096 * 11 * 128
    # decode: the capacity must be a multiple of 16
    odd = pisa.make_params(2, 4096 + 8, 16, 4, 128, K=8)
    assert L.pisa_attend_decode(ctypes.byref(odd), a, a, a, a, a, a, big, a, None) == -2
    assert L.pisa_attend_decode(ctypes.byref(p), a, a, None, a, a, a, big, a, None) == -1
    assert L.pisa_attend_decode(ctypes.byref(p), a, a, a, a, a, a, 16, a, None) == -4
    assert L.pisa_attend_decode(ctypes.byref(f32), a, a, a, a, a, a, big, a, None) == -2


def test_bucket_grids_beyond_32_bit_tiles_are_refused_before_launch(pisa):
    # B * H_kv * N * K fits in 32 bits, but the (query chunk x node) bucket
    # grid, which grows with N^2, does not
    L = pisa.lib()
    a = ctypes.c_void_p(0x10000)
    huge = 1 << 62
    p = pisa.make_params(1, 1 << 26, 8, 8, 128, K=1)
    assert L.pisa_select_prefill(ctypes.byref(p), a, a, a, a, huge, a, None, None, None) == -2
    pa = pisa.make_params(1, 1 << 26, 4, 4, 128, K=1)
    assert L.pisa_attend_prefill(ctypes.byref(pa), a, a, a, a, a, huge, a, None) == -2


def test_the_product_package_never_touches_the_oracle():
    # the library and its binding stand alone: no module of the package
    # imports, loads or builds anything under oracle/
    import pathlib
    import re
    root = pathlib.Path(__file__).resolve().parent.parent / "pyramid_top_block_mean_gb300"
    pat = re.compile(r"\b(import\s+oracle|from\s+oracle|pisa_oracle|libpisa_oracle)\b")
    hits = [str(f) for f in root.rglob("*") if f.suffix in (".py", ".cu", ".cuh", ".h", ".cpp")
            and pat.search(f.read_text(errors="ignore"))]
    assert hits == []
