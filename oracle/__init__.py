"""ctypes front end of the fp64 CPU oracle (oracle/pisa_oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the
benchmark's CPU-baseline leg may import this module; the product path never
does.  Inputs are converted to fp64 exactly (bf16 and fp32 embed in fp64).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pisa_oracle.c")
_LIB = os.path.join(_HERE, "libpisa_oracle.so")

_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_dp = ctypes.POINTER(ctypes.c_double)
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)


class _Params(ctypes.Structure):
    _fields_ = [("B", _i64), ("N", _i64), ("Hq", _i32), ("Hkv", _i32),
                ("d", _i32), ("C", _i32), ("K", _i32), ("scale", ctypes.c_double),
                ("scorer", _i32), ("prefix", _i32)]


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-shared", "-fPIC", _SRC,
               "-o", _LIB + ".tmp", "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        L.po_num_levels.argtypes = [_i64, _i32]
        L.po_num_levels.restype = ctypes.c_int
        L.po_num_nodes.argtypes = [_i64, _i32]
        L.po_num_nodes.restype = _i64
        L.po_build_pyramid.argtypes = [ctypes.POINTER(_Params), _dp, _i32p, _dp]
        L.po_build_pyramid.restype = ctypes.c_int
        L.po_select.argtypes = [ctypes.POINTER(_Params), _dp, _dp, _dp, _i32p,
                                ctypes.c_int, _i64, _i64p, _i32p, _dp, _dp,
                                _i32p, _i64p]
        L.po_select.restype = ctypes.c_int
        L.po_score_nodes.argtypes = [ctypes.POINTER(_Params), _dp, _dp, _dp, _i64,
                                     ctypes.c_int, _i64, _i32, _i64, ctypes.c_int,
                                     _i64, _i64p, _dp]
        L.po_score_nodes.restype = ctypes.c_int
        L.po_node_eligible.argtypes = [ctypes.POINTER(_Params), _i64, ctypes.c_int, _i64]
        L.po_node_eligible.restype = ctypes.c_int
        L.po_select_flat.argtypes = [ctypes.POINTER(_Params), _dp, _dp, _i64, _i64p,
                                     _i32p, _dp, _dp]
        L.po_select_flat.restype = ctypes.c_int
        L.po_sparse_attention.argtypes = [ctypes.POINTER(_Params), _dp, _dp, _dp, _i32p,
                                          _i64, _i64p, ctypes.c_int, _dp]
        L.po_sparse_attention.restype = ctypes.c_int
        L.po_num_threads.restype = ctypes.c_int
        L.po_set_num_threads.argtypes = [ctypes.c_int]
        _lib = L
    return _lib


def _f64(x) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray, t):
    return a.ctypes.data_as(t)


class Oracle:
    """Oracle bound to one problem shape (B, N, Hq, Hkv, d, C, K, scale), block
    scorer (0: log-sum-exp, 1: PISA-1, 2: PISA-2) and summary reading
    (prefix=False: node summaries over all keys of the span; prefix=True: a
    prefill query at position t reads summaries of the keys at positions
    <= t only, the prefix-consistent reading)."""

    def __init__(self, B, N, Hq, Hkv, d, C, K, scale: float = 0.0, scorer: int = 0, prefix: bool = False):
        self.p = _Params(B, N, Hq, Hkv, d, C, K, scale, scorer, int(bool(prefix)))
        self.B, self.N, self.Hq, self.Hkv, self.d, self.C, self.K = B, N, Hq, Hkv, d, C, K
        self.scorer = scorer
        self.prefix = bool(prefix)

    @classmethod
    def from_shape(cls, s, scale: float = 0.0, scorer: int = 0, prefix: bool = False):
        return cls(s.B, s.N, s.Hq, s.Hkv, s.d, s.C, s.K, scale, scorer, prefix)

    @property
    def num_levels(self) -> int:
        return lib().po_num_levels(self.N, self.C)

    @property
    def num_nodes(self) -> int:
        return lib().po_num_nodes(self.N, self.C)

    def level_sizes(self):
        nb = -(-self.N // self.C)
        sizes = [nb]
        while sizes[-1] > 1:
            sizes.append(-(-sizes[-1] // 2))
        return sizes

    def pyramid(self, k, seq_lens: Optional[Sequence[int]] = None) -> np.ndarray:
        k = _f64(k)
        out = np.zeros((self.B, self.Hkv, self.num_nodes, self.d), np.float64)
        sl = None if seq_lens is None else np.ascontiguousarray(seq_lens, np.int32)
        rc = lib().po_build_pyramid(ctypes.byref(self.p), _ptr(k, _dp),
                                    None if sl is None else _ptr(sl, _i32p), _ptr(out, _dp))
        if rc != 0:
            raise ValueError("oracle pyramid: bad arguments")
        return out

    def select(self, q, k, pyr=None, sel=None, seq_lens=None, decode=False,
               trace=False, qrows=False):
        """Returns dict(idx [nq, K+3] int32, score [nq, K+3], margin [nq],
        trace [nq, L, K] or None, counters {...}).
        qrows: q holds only the selected queries' head rows [nsel, G, d]."""
        q = _f64(q); k = _f64(k)
        if pyr is None:
            pyr = self.pyramid(k, seq_lens)
        pyr = _f64(pyr)
        sl = None if seq_lens is None else np.ascontiguousarray(seq_lens, np.int32)
        if decode:
            nq = self.B * self.Hkv
            selp = None
        elif sel is None:
            nq = self.B * self.Hkv * self.N
            selp = None
        else:
            selp = np.ascontiguousarray(np.asarray(sel, np.int64).reshape(-1, 3))
            nq = selp.shape[0]
        W = self.K + 3
        idx = np.empty((nq, W), np.int32)
        score = np.empty((nq, W), np.float64)
        margin = np.empty((nq,), np.float64)
        L = self.num_levels
        tr = np.empty((nq, L, self.K), np.int32) if trace else None
        cnt = np.zeros(4, np.int64)
        rc = lib().po_select(ctypes.byref(self.p), _ptr(q, _dp), _ptr(k, _dp), _ptr(pyr, _dp),
                             None if sl is None else _ptr(sl, _i32p),
                             1 if decode else (2 if qrows else 0),
                             nq, None if selp is None else _ptr(selp, _i64p),
                             _ptr(idx, _i32p), _ptr(score, _dp), _ptr(margin, _dp),
                             None if tr is None else _ptr(tr, _i32p), _ptr(cnt, _i64p))
        if rc != 0:
            raise ValueError("oracle select: bad arguments")
        return dict(idx=idx, score=score, margin=margin, trace=tr,
                    counters=dict(levels_scored=int(cnt[0]), child_dots=int(cnt[1]),
                                  leaf_keys=int(cnt[2]), cands_scored=int(cnt[3])))

    def score_nodes(self, q, k, pyr, b, h, t, level, nodes, len_=None, decode=False, qrows=False):
        """decode: q is [B, Hq, d]; qrows: q is this query's [G, d] rows."""
        q = _f64(q); k = _f64(k); pyr = _f64(pyr)
        nodes = np.ascontiguousarray(nodes, np.int64)
        out = np.empty(len(nodes), np.float64)
        rc = lib().po_score_nodes(ctypes.byref(self.p), _ptr(q, _dp), _ptr(k, _dp), _ptr(pyr, _dp),
                                  self.N if len_ is None else len_,
                                  1 if decode else (2 if qrows else 0),
                                  b, h, t, level, len(nodes), _ptr(nodes, _i64p), _ptr(out, _dp))
        if rc != 0:
            raise ValueError("oracle score_nodes: bad arguments")
        return out

    def eligible(self, t, level, j) -> bool:
        return bool(lib().po_node_eligible(ctypes.byref(self.p), t, level, j))

    def select_flat(self, q, pyr, sel=None):
        q = _f64(q); pyr = _f64(pyr)
        if sel is None:
            nq = self.B * self.Hkv * self.N
            selp = None
        else:
            selp = np.ascontiguousarray(np.asarray(sel, np.int64).reshape(-1, 3))
            nq = selp.shape[0]
        W = self.K + 3
        idx = np.empty((nq, W), np.int32)
        score = np.empty((nq, W), np.float64)
        margin = np.empty((nq,), np.float64)
        rc = lib().po_select_flat(ctypes.byref(self.p), _ptr(q, _dp), _ptr(pyr, _dp), nq,
                                  None if selp is None else _ptr(selp, _i64p),
                                  _ptr(idx, _i32p), _ptr(score, _dp), _ptr(margin, _dp))
        if rc != 0:
            raise ValueError("oracle flat: bad arguments")
        return dict(idx=idx, score=score, margin=margin)


    def attend(self, q, k, v, idx, sel=None, qrows: bool = False) -> np.ndarray:
        """Attention of the queries over their selected blocks (causal inside
        each block); idx is the full [B, Hkv, N, K+3] selection.  Returns
        [nq, G, d] fp64 for the sel triples (b, h, t), or every query.  With
        qrows, q holds only the selected queries' head rows [nsel, G, d]."""
        q = _f64(q); k = _f64(k); v = _f64(v)
        idx = np.ascontiguousarray(np.asarray(idx, np.int32).reshape(-1))
        if idx.size != self.B * self.Hkv * self.N * (self.K + 3):
            raise ValueError("oracle attend: idx has the wrong size")
        if sel is None:
            nq = self.B * self.Hkv * self.N
            selp = None
        else:
            selp = np.ascontiguousarray(np.asarray(sel, np.int64).reshape(-1, 3))
            nq = selp.shape[0]
        G = self.Hq // self.Hkv
        out = np.empty((nq, G, self.d), np.float64)
        rc = lib().po_sparse_attention(ctypes.byref(self.p), _ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp),
                                       _ptr(idx, _i32p), nq,
                                       None if selp is None else _ptr(selp, _i64p), int(bool(qrows)),
                                       _ptr(out, _dp))
        if rc != 0:
            raise ValueError("oracle attend: bad arguments or a query with no key")
        return out


def attention_mass(q, k, idx, sel, C: int, scale: float = 0.0, qrows: bool = False) -> np.ndarray:
    """Attention-mass ratio of a selection (agihunt.info summary, quality
    paragraph: the share of full attention's softmax mass that falls on the
    selected blocks).  For query (b, h, t) and each head g of its GQA group,
    the causal softmax over keys 0..t of s q_g . k_i is summed over the keys
    of the distinct blocks listed in its row of idx (entries outside
    [0, t // C] add nothing), then averaged over the group's heads.
    q [B, Hq, N, d] (or, with qrows, [nsel, G, d]), k [B, Hkv, N, d],
    idx [nsel, W] the selection rows of the sel triples (b, h, t).
    Plain fp64 numpy, one query at a time; returns [nsel]."""
    q = _f64(q)
    k = _f64(k)
    idx = np.asarray(idx)
    Hkv, d = k.shape[1], k.shape[3]
    G = q.shape[1] // Hkv if not qrows else q.shape[1]
    s = scale if scale > 0 else 1.0 / np.sqrt(d)
    out = np.empty(len(sel), np.float64)
    for n, (b, h, t) in enumerate(sel):
        keys = k[b, h, :t + 1]
        blocks = {int(j) for j in idx[n] if 0 <= j <= t // C}
        mask = np.zeros(t + 1, bool)
        for j in blocks:
            mask[j * C:min((j + 1) * C, t + 1)] = True
        r = 0.0
        for g in range(G):
            qg = q[n, g] if qrows else q[b, h * G + g, t]
            x = s * (keys @ qg)
            m = x.max()
            w = np.exp(x - m)
            r += w[mask].sum() / w.sum()
        out[n] = r / G
    return out


def num_threads() -> int:
    return lib().po_num_threads()


def set_num_threads(n: int) -> None:
    lib().po_set_num_threads(n)
