"""Thin ctypes binding of the selector's C ABI (include/pisa.h).

Argument marshalling only: every step of the selection runs in the CUDA
kernels of libpisa.so.  PyTorch provides device memory and streams.  Importing
this module loads the library and raises ImportError when it is missing; there
is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpisa.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
        "(the selector has no CPU fallback)")

_lib = ctypes.CDLL(LIB_PATH)

PISA_OK = 0
STATUS_NAMES = {0: "PISA_OK", -1: "PISA_ERR_INVALID_ARG", -2: "PISA_ERR_UNSUPPORTED",
                -3: "PISA_ERR_MISALIGNED", -4: "PISA_ERR_WORKSPACE", -5: "PISA_ERR_CUDA",
                -6: "PISA_ERR_DEVICE"}
BF16, FP32 = 0, 1
SCORER_LSE, SCORER_MEAN, SCORER_MEAN_VAR = 0, 1, 2
SUMMARIES_ALL, SUMMARIES_PREFIX = 0, 1
MODE_PREFILL, MODE_DECODE, MODE_FLAT, MODE_ATTEND = 0, 1, 2, 3
DEV_OK, DEV_BAD_SEQ_LEN, DEV_TIMEOUT, DEV_BAD_INDEX = 0, 1, 2, 3

EXPORTED = ["pisa_abi_version", "pisa_status_string", "pisa_pyramid_levels", "pisa_pyramid_nodes",
            "pisa_pyramid_bytes", "pisa_workspace_bytes", "pisa_build_pyramid", "pisa_select_prefill",
            "pisa_prefill_route", "pisa_prefill_leaves", "pisa_select_decode", "pisa_select_flat",
            "pisa_read_device_status", "pisa_select_prefill_static", "pisa_kernel_launches",
            "pisa_attend_prefill", "pisa_build_pyramid_paged", "pisa_select_decode_paged", "pisa_attend_decode",
            "pisa_read_static_status", "pisa_test_inject_leaf_timeout"]


class Params(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_uint32), ("dtype", ctypes.c_int32),
                ("B", ctypes.c_int64), ("N", ctypes.c_int64),
                ("H_q", ctypes.c_int32), ("H_kv", ctypes.c_int32), ("d", ctypes.c_int32),
                ("C", ctypes.c_int32), ("g", ctypes.c_int32), ("K", ctypes.c_int32),
                ("qtile", ctypes.c_int32), ("scale", ctypes.c_float), ("scorer", ctypes.c_int32),
                ("summaries", ctypes.c_int32)]


_P = ctypes.POINTER(Params)
_vp = ctypes.c_void_p
_lib.pisa_abi_version.restype = ctypes.c_int
_lib.pisa_kernel_launches.restype = ctypes.c_uint64
_lib.pisa_status_string.argtypes = [ctypes.c_int]
_lib.pisa_status_string.restype = ctypes.c_char_p
_lib.pisa_pyramid_levels.argtypes = [_P]
_lib.pisa_pyramid_levels.restype = ctypes.c_int32
_lib.pisa_pyramid_nodes.argtypes = [_P]
_lib.pisa_pyramid_nodes.restype = ctypes.c_int64
_lib.pisa_pyramid_bytes.argtypes = [_P]
_lib.pisa_pyramid_bytes.restype = ctypes.c_size_t
_lib.pisa_workspace_bytes.argtypes = [_P, ctypes.c_int32]
_lib.pisa_workspace_bytes.restype = ctypes.c_size_t
_lib.pisa_build_pyramid.argtypes = [_P, _vp, _vp, _vp, _vp]
_lib.pisa_build_pyramid.restype = ctypes.c_int
_lib.pisa_select_prefill.argtypes = [_P, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp, _vp, _vp, _vp]
_lib.pisa_select_prefill.restype = ctypes.c_int
_lib.pisa_prefill_route.argtypes = [_P, _vp, _vp, _vp, ctypes.c_size_t, _vp, _vp]
_lib.pisa_prefill_route.restype = ctypes.c_int
_lib.pisa_prefill_leaves.argtypes = [_P, _vp, _vp, _vp, ctypes.c_size_t, _vp, _vp, _vp]
_lib.pisa_prefill_leaves.restype = ctypes.c_int
_lib.pisa_select_decode.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp, _vp, _vp, _vp]
_lib.pisa_select_decode.restype = ctypes.c_int
_lib.pisa_select_flat.argtypes = [_P, _vp, _vp, _vp, ctypes.c_size_t, _vp, _vp, _vp]
_lib.pisa_select_flat.restype = ctypes.c_int
_lib.pisa_build_pyramid_paged.argtypes = [_P, _vp, ctypes.c_int64, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
_lib.pisa_build_pyramid_paged.restype = ctypes.c_int
_lib.pisa_select_decode_paged.argtypes = [_P, _vp, _vp, ctypes.c_int64, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp,
                                          _vp, _vp, _vp]
_lib.pisa_select_decode_paged.restype = ctypes.c_int
_lib.pisa_attend_decode.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp, _vp]
_lib.pisa_attend_decode.restype = ctypes.c_int
_lib.pisa_attend_prefill.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp, _vp]
_lib.pisa_attend_prefill.restype = ctypes.c_int
_lib.pisa_read_device_status.argtypes = [_vp, ctypes.POINTER(ctypes.c_int32), _vp]
_lib.pisa_read_device_status.restype = ctypes.c_int
_lib.pisa_select_prefill_static.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, _vp]
_lib.pisa_select_prefill_static.restype = ctypes.c_int
_lib.pisa_read_static_status.argtypes = [ctypes.POINTER(ctypes.c_int32), _vp]
_lib.pisa_read_static_status.restype = ctypes.c_int
_lib.pisa_test_inject_leaf_timeout.argtypes = [ctypes.c_uint64, ctypes.c_int32]
_lib.pisa_test_inject_leaf_timeout.restype = None


class PisaError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_string(code)}")


def lib() -> ctypes.CDLL:
    return _lib


def status_string(code: int) -> str:
    return _lib.pisa_status_string(code).decode()


def abi_version() -> int:
    return _lib.pisa_abi_version()


def kernel_launches() -> int:
    """Kernel launches the library has issued in this process so far."""
    return _lib.pisa_kernel_launches()


def make_params(B: int, N: int, H_q: int, H_kv: int, d: int, C: int = 64, g: int = 2, K: int = 8,
                qtile: int = 4, dtype: str = "bf16", scale: float = 0.0, scorer: int = 0,
                summaries: int = 0) -> Params:
    """scorer: SCORER_LSE (PISA), SCORER_MEAN (PISA-1) or SCORER_MEAN_VAR (PISA-2);
    summaries: SUMMARIES_ALL or SUMMARIES_PREFIX (prefix-consistent prefill)."""
    return Params(ctypes.sizeof(Params), BF16 if dtype == "bf16" else FP32, B, N, H_q, H_kv, d, C, g, K,
                  qtile, scale, scorer, summaries)


def params_from_shape(s, N: Optional[int] = None, scorer: int = 0, summaries: int = 0) -> Params:
    return make_params(s.B, s.N if N is None else N, s.Hq, s.Hkv, s.d, s.C, s.g, s.K, s.qtile, s.dtype,
                       scorer=scorer, summaries=summaries)


def pyramid_levels(p: Params) -> int:
    return _lib.pisa_pyramid_levels(ctypes.byref(p))


def pyramid_nodes(p: Params) -> int:
    return _lib.pisa_pyramid_nodes(ctypes.byref(p))


def pyramid_bytes(p: Params) -> int:
    return _lib.pisa_pyramid_bytes(ctypes.byref(p))


def workspace_bytes(p: Params, mode: int) -> int:
    return _lib.pisa_workspace_bytes(ctypes.byref(p), mode)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(rc: int, what: str):
    if rc != PISA_OK:
        raise PisaError(rc, what)


def build_pyramid(p: Params, k: torch.Tensor, pyramid: torch.Tensor, seq_lens: Optional[torch.Tensor] = None,
                  stream=None, check: bool = True) -> int:
    rc = _lib.pisa_build_pyramid(ctypes.byref(p), _ptr(k), _ptr(seq_lens), _ptr(pyramid), _stream(stream))
    if check:
        _check(rc, "pisa_build_pyramid")
    return rc


def select_prefill(p: Params, q, k, pyramid, ws, out_idx, out_score=None, trace=None, stream=None,
                   check: bool = True) -> int:
    rc = _lib.pisa_select_prefill(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(pyramid), _ptr(ws),
                                  0 if ws is None else ws.numel() * ws.element_size(),
                                  _ptr(out_idx), _ptr(out_score), _ptr(trace), _stream(stream))
    if check:
        _check(rc, "pisa_select_prefill")
    return rc


def prefill_route(p: Params, q, pyramid, ws, trace=None, stream=None, check: bool = True) -> int:
    rc = _lib.pisa_prefill_route(ctypes.byref(p), _ptr(q), _ptr(pyramid), _ptr(ws),
                                 ws.numel() * ws.element_size(), _ptr(trace), _stream(stream))
    if check:
        _check(rc, "pisa_prefill_route")
    return rc


def prefill_leaves(p: Params, q, k, ws, out_idx, out_score=None, stream=None, check: bool = True) -> int:
    rc = _lib.pisa_prefill_leaves(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(ws), ws.numel() * ws.element_size(),
                                  _ptr(out_idx), _ptr(out_score), _stream(stream))
    if check:
        _check(rc, "pisa_prefill_leaves")
    return rc


def select_decode(p: Params, q, k_cache, seq_lens, pyramid, ws, out_idx, out_score=None, trace=None,
                  stream=None, check: bool = True) -> int:
    rc = _lib.pisa_select_decode(ctypes.byref(p), _ptr(q), _ptr(k_cache), _ptr(seq_lens), _ptr(pyramid),
                                 _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                                 _ptr(out_idx), _ptr(out_score), _ptr(trace), _stream(stream))
    if check:
        _check(rc, "pisa_select_decode")
    return rc


def select_flat(p: Params, q, pyramid, ws, out_idx, out_score=None, stream=None, check: bool = True) -> int:
    rc = _lib.pisa_select_flat(ctypes.byref(p), _ptr(q), _ptr(pyramid), _ptr(ws),
                               0 if ws is None else ws.numel() * ws.element_size(),
                               _ptr(out_idx), _ptr(out_score), _stream(stream))
    if check:
        _check(rc, "pisa_select_flat")
    return rc


def build_pyramid_paged(p: Params, k_pages, page_table, pyramid, ws, seq_lens=None, stream=None,
                        check: bool = True) -> int:
    """k_pages [num_pages, H_kv, C, d]; page_table int32 [B, ceil(N / C)]."""
    rc = _lib.pisa_build_pyramid_paged(ctypes.byref(p), _ptr(k_pages), k_pages.shape[0], _ptr(page_table),
                                       _ptr(seq_lens), _ptr(pyramid), _ptr(ws), ws.numel() * ws.element_size(),
                                       _stream(stream))
    if check:
        _check(rc, "pisa_build_pyramid_paged")
    return rc


def select_decode_paged(p: Params, q, k_pages, page_table, seq_lens, pyramid, ws, out_idx, out_score=None,
                        trace=None, stream=None, check: bool = True) -> int:
    rc = _lib.pisa_select_decode_paged(ctypes.byref(p), _ptr(q), _ptr(k_pages), k_pages.shape[0], _ptr(page_table),
                                       _ptr(seq_lens), _ptr(pyramid), _ptr(ws), ws.numel() * ws.element_size(),
                                       _ptr(out_idx), _ptr(out_score), _ptr(trace), _stream(stream))
    if check:
        _check(rc, "pisa_select_decode_paged")
    return rc


def attend_prefill(p: Params, q, k, v, idx, ws, out, stream=None, check: bool = True) -> int:
    rc = _lib.pisa_attend_prefill(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(idx), _ptr(ws),
                                  0 if ws is None else ws.numel() * ws.element_size(), _ptr(out),
                                  _stream(stream))
    if check:
        _check(rc, "pisa_attend_prefill")
    return rc


def attend_decode(p: Params, q, k_cache, v_cache, seq_lens, idx, ws, out, stream=None, check: bool = True) -> int:
    rc = _lib.pisa_attend_decode(ctypes.byref(p), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens), _ptr(idx),
                                 _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(), _ptr(out),
                                 _stream(stream))
    if check:
        _check(rc, "pisa_attend_decode")
    return rc


def read_device_status(ws: torch.Tensor, stream=None) -> int:
    code = ctypes.c_int32(0)
    rc = _lib.pisa_read_device_status(_ptr(ws), ctypes.byref(code), _stream(stream))
    if rc not in (PISA_OK, -6):
        _check(rc, "pisa_read_device_status")
    return code.value


class Selector:
    """Owns the device buffers (torch tensors) for one problem shape and runs
    the selector through the C ABI.  `mode` is "prefill", "decode" or "flat"."""

    def __init__(self, p: Params, device="cuda", mode: str = "prefill", with_scores: bool = True):
        self.p = p
        self.device = torch.device(device)
        W = p.K + 3
        P = pyramid_nodes(p)
        self.pyramid = torch.empty(p.B, p.H_kv, P, p.d, dtype=torch.float32, device=self.device)
        m = {"prefill": MODE_PREFILL, "decode": MODE_DECODE, "flat": MODE_FLAT}[mode]
        nbytes = workspace_bytes(p, m)
        self.ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=self.device)
        if mode == "decode":
            shape = (p.B, p.H_kv, W)
        else:
            shape = (p.B, p.H_kv, p.N, W)
        self.out_idx = torch.empty(shape, dtype=torch.int32, device=self.device)
        self.out_score = torch.empty(shape, dtype=torch.float32, device=self.device) if with_scores else None

    def build(self, k, seq_lens=None, stream=None):
        build_pyramid(self.p, k, self.pyramid, seq_lens, stream)

    def prefill(self, q, k, trace=None, stream=None, build: bool = True):
        if build:
            build_pyramid(self.p, k, self.pyramid, None, stream)
        select_prefill(self.p, q, k, self.pyramid, self.ws, self.out_idx, self.out_score, trace, stream)
        return self.out_idx, self.out_score

    def decode(self, q, k_cache, seq_lens, trace=None, stream=None):
        select_decode(self.p, q, k_cache, seq_lens, self.pyramid, self.ws, self.out_idx, self.out_score, trace,
                      stream)
        return self.out_idx, self.out_score

    def build_paged(self, k_pages, page_table, seq_lens=None, stream=None):
        build_pyramid_paged(self.p, k_pages, page_table, self.pyramid, self.ws, seq_lens, stream)

    def decode_paged(self, q, k_pages, page_table, seq_lens, trace=None, stream=None):
        select_decode_paged(self.p, q, k_pages, page_table, seq_lens, self.pyramid, self.ws, self.out_idx,
                            self.out_score, trace, stream)
        return self.out_idx, self.out_score

    def flat(self, q, k=None, stream=None, build: bool = True):
        if build:
            build_pyramid(self.p, k, self.pyramid, None, stream)
        select_flat(self.p, q, self.pyramid, self.ws, self.out_idx, self.out_score, stream)
        return self.out_idx, self.out_score

    def device_status(self, stream=None) -> int:
        return read_device_status(self.ws, stream)


class Attention:
    """Owns the workspace and output of block-sparse attention over a
    selection for one problem shape: prefill (pisa_attend_prefill, every
    query position) or decode (pisa_attend_decode, one query per sequence)."""

    def __init__(self, p: Params, device="cuda", mode: str = "prefill"):
        self.p = p
        self.mode = mode
        self.device = torch.device(device)
        m = MODE_ATTEND if mode == "prefill" else MODE_DECODE
        self.ws = torch.empty(max(workspace_bytes(p, m), 256), dtype=torch.uint8, device=self.device)
        shape = (p.B, p.H_q, p.N, p.d) if mode == "prefill" else (p.B, p.H_q, p.d)
        self.out = torch.empty(shape, dtype=torch.bfloat16, device=self.device)

    def __call__(self, q, k, v, idx, stream=None):
        attend_prefill(self.p, q, k, v, idx, self.ws, self.out, stream)
        return self.out

    def decode(self, q, k_cache, v_cache, seq_lens, idx, stream=None):
        attend_decode(self.p, q, k_cache, v_cache, seq_lens, idx, self.ws, self.out, stream)
        return self.out

    def device_status(self, stream=None) -> int:
        return read_device_status(self.ws, stream)
