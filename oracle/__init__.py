"""CPU oracle of content-routed sparse attention (ctypes wrapper of oracle.c).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA path in ``content_routed_sparse_build_b300`` and neither side
imports the other.

The oracle follows the definition written at the top of oracle.c: span
means as summaries, unscaled q . summary scores over the complete spans
before the query's own span, the k best under (score descending, index
ascending), and exact softmax attention (double accumulation) over the kept
spans plus the causal part of the local span.  Every function is pinned by
the ``-m "not gpu"`` tests in tests/test_oracle_pins.py; no function is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
SO = os.path.join(HERE, "liboracle.so")
SRC = os.path.join(HERE, "oracle.c")

_DT = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2, torch.float64: 3}
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (OpenMP for the loop over query rows)."""
    if force or not os.path.exists(SO) or os.path.getmtime(SRC) > os.path.getmtime(SO):
        tmp = SO + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
               "-Wall", "-o", tmp, SRC, "-lm"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("oracle build failed:\n%s\n%s" % (res.stdout, res.stderr))
        os.replace(tmp, SO)
    return SO


def _load():
    global _lib
    if _lib is None:
        # ORACLE_SO points the tests' mutation check at a deliberately broken
        # build of oracle.c; it is never set otherwise.
        lib = ctypes.CDLL(os.environ.get("ORACLE_SO") or build())
        P, I, I64, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_set_threads.argtypes = [I]
        lib.oracle_max_threads.restype = I
        lib.oracle_summaries.argtypes = [I, P, I, I, I64, I64, I, I, I64, I64, P, I64]
        lib.oracle_route.restype = I
        lib.oracle_route.argtypes = [I, P, I, I, I, I64, I64, I, I, I, P, I64, P, I64, P, P, P]
        lib.oracle_route_group.restype = I
        lib.oracle_route_group.argtypes = [I, P, I, I, I, I64, I64, I, I, I, P, I64, P, I64, P, P, P]
        lib.oracle_attend.restype = I
        lib.oracle_attend.argtypes = [I, P, P, P, I, I, I, I64, I64, I64, I, I, I, D, P, P, I64,
                                      P, P, P]
        lib.oracle_quantize_rows.argtypes = [I, P, I64, I, P, P]
        lib.oracle_quantize_rows4.argtypes = [I, P, I64, I, P, P]
        _lib = lib
    return _lib


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def threads() -> int:
    return int(_load().oracle_max_threads())


def _host(t: torch.Tensor) -> torch.Tensor:
    if t.device.type != "cpu" or not t.is_contiguous():
        raise ValueError("oracle inputs must be contiguous host tensors")
    if t.dtype not in _DT:
        raise ValueError("unsupported dtype %s" % t.dtype)
    return t


def summaries(K: torch.Tensor, L: int, S: int, j0: int = 0, j1: int | None = None,
              out: np.ndarray | None = None) -> np.ndarray:
    """Span means of K [B, Hkv, L_cap, d] for spans [j0, j1); float64 [B, Hkv, ns_cap, d]."""
    _host(K)
    B, Hkv, L_cap, d = K.shape
    ns_cap = (L_cap + S - 1) // S
    if j1 is None:
        j1 = (L + S - 1) // S
    if out is None:
        out = np.zeros((B, Hkv, ns_cap, d), np.float64)
    assert out.shape == (B, Hkv, ns_cap, d) and out.dtype == np.float64 and out.flags.c_contiguous
    _load().oracle_summaries(_DT[K.dtype], K.data_ptr(), B, Hkv, L_cap, L, d, S, j0, j1,
                             out.ctypes.data, ns_cap)
    return out


def route(Q: torch.Tensor, q_pos0: int, summ: np.ndarray, Hkv: int, S: int, topk: int,
          rows: np.ndarray | None = None, want_scores: bool = False):
    """Selections for Q [B, Hq, n_q, d].

    Returns (sel int32 [n, topk], margin float64 [n]) and, if asked, the
    selected spans' scores; n is every row of [B, Hq, n_q] or len(rows).
    """
    _host(Q)
    B, Hq, n_q, d = Q.shape
    ns_cap = summ.shape[2]
    summ = np.ascontiguousarray(summ, dtype=np.float64)
    rp, nr = None, 0
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        rp, nr = rows.ctypes.data, len(rows)
    n = nr if rows is not None else B * Hq * n_q
    sel = np.zeros((n, topk), np.int32)
    margin = np.zeros(n, np.float64)
    sc = np.zeros((n, topk), np.float64) if want_scores else None
    rc = _load().oracle_route(_DT[Q.dtype], Q.data_ptr(), B, Hq, Hkv, n_q, q_pos0, d, S, topk,
                              summ.ctypes.data, ns_cap, rp, nr, sel.ctypes.data, margin.ctypes.data,
                              sc.ctypes.data if sc is not None else None)
    if rc != 0:
        raise ValueError("oracle_route: a candidate span has no summary")
    return (sel, margin, sc) if want_scores else (sel, margin)


def route_group(Q: torch.Tensor, q_pos0: int, summ: np.ndarray, Hkv: int, S: int, topk: int,
                rows: np.ndarray | None = None, want_scores: bool = False):
    """Group-shared selections for Q [B, Hq, n_q, d]: one per (b, kv-head,
    query), scored by the sum of the group's heads' scores, repeated on every
    head row of the group.  Returns as route()."""
    _host(Q)
    B, Hq, n_q, d = Q.shape
    ns_cap = summ.shape[2]
    summ = np.ascontiguousarray(summ, dtype=np.float64)
    rp, nr = None, 0
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        rp, nr = rows.ctypes.data, len(rows)
    n = nr if rows is not None else B * Hq * n_q
    sel = np.zeros((n, topk), np.int32)
    margin = np.zeros(n, np.float64)
    sc = np.zeros((n, topk), np.float64) if want_scores else None
    rc = _load().oracle_route_group(_DT[Q.dtype], Q.data_ptr(), B, Hq, Hkv, n_q, q_pos0, d, S, topk,
                                    summ.ctypes.data, ns_cap, rp, nr, sel.ctypes.data,
                                    margin.ctypes.data, sc.ctypes.data if sc is not None else None)
    if rc != 0:
        raise ValueError("oracle_route_group: a candidate span has no summary")
    return (sel, margin, sc) if want_scores else (sel, margin)


def attend(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, q_pos0: int, S: int,
           sel: np.ndarray, scale: float | None = None, rows: np.ndarray | None = None):
    """Outputs for Q [B, Hq, n_q, d] given selections.

    Returns (O float64 [n, d], lse float64 [n], weight sums float64 [n]).
    """
    for t in (Q, K, V):
        _host(t)
    B, Hq, n_q, d = Q.shape
    _, Hkv, L_cap, _ = K.shape
    topk = sel.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    sel = np.ascontiguousarray(sel, dtype=np.int32)
    rp, nr = None, 0
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        rp, nr = rows.ctypes.data, len(rows)
    n = nr if rows is not None else B * Hq * n_q
    assert sel.shape[0] == n
    O = np.zeros((n, d), np.float64)
    lse = np.zeros(n, np.float64)
    ws = np.zeros(n, np.float64)
    rc = _load().oracle_attend(_DT[Q.dtype], Q.data_ptr(), K.data_ptr(), V.data_ptr(), B, Hq, Hkv,
                               n_q, q_pos0, L_cap, d, S, topk, float(scale), sel.ctypes.data, rp, nr,
                               O.ctypes.data, lse.ctypes.data, ws.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_attend: a selected span is not a complete span before the query")
    return O, lse, ws


def quantize_rows(X: torch.Tensor):
    """8-bit rows of X [..., d]: (q int8 [..., d], scale float32 [...]).

    Symmetric, one fp32 scale per row: s = max|x| / 127, q = rint(x / s)
    clamped to [-127, 127] (0 when s == 0), every step in fp32."""
    _host(X)
    d = X.shape[-1]
    rows = X.numel() // d
    q = np.zeros(X.shape, np.int8)
    s = np.zeros(X.shape[:-1], np.float32)
    _load().oracle_quantize_rows(_DT[X.dtype], X.data_ptr(), rows, d, q.ctypes.data, s.ctypes.data)
    return q, s


def quantize_rows4(X: torch.Tensor):
    """4-bit rows of X [..., d]: (q int8 in [-7, 7] [..., d], scale float32 [...]).

    Symmetric, one fp32 scale per row: s = max|x| / 7, q = rint(x / s)
    clamped to [-7, 7] (0 when s == 0), every step in fp32."""
    _host(X)
    d = X.shape[-1]
    rows = X.numel() // d
    q = np.zeros(X.shape, np.int8)
    s = np.zeros(X.shape[:-1], np.float32)
    _load().oracle_quantize_rows4(_DT[X.dtype], X.data_ptr(), rows, d, q.ctypes.data, s.ctypes.data)
    return q, s


def dequantize_rows(q: np.ndarray, s: np.ndarray) -> torch.Tensor:
    """q * s in float64 (exact), as a host tensor of q's shape."""
    return torch.from_numpy(q.astype(np.float64) * s.astype(np.float64)[..., None])
