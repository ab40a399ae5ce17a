"""Content-routed sparse attention for B300 (sm_103a).

A thin ctypes binding of libssa.so, whose C ABI is declared in
include/ssa.h.  The functions here only marshal arguments: every step of
the method runs in the library's CUDA kernels, on the caller's stream, in
the caller's (PyTorch-allocated) device memory.  There is no CPU path: if
the library cannot be built or loaded, importing it raises.

Entry points (same names as the C ABI):
  ssa_build_summaries  span means of the keys
  ssa_route            span scores + top-k selection
  ssa_route_group      one top-k per kv-head group (summed scores of its heads)
  ssa_attend_decode    one query per head, split over spans, LSE merge
  ssa_attend_prefill   a chunk of queries, span-major tiles, LSE merge
  ssa_attend_decode_noalloc  ssa_attend_decode on a library-owned scratch block
  ssa_workspace_size / ssa_workspace_error / ssa_status_string
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

SSA_OK = 0
SSA_ERR_INVALID_ARG = 1
SSA_ERR_UNSUPPORTED = 2
SSA_ERR_WORKSPACE = 3
SSA_ERR_CUDA = 4
SSA_ERR_DEVICE = 5

SSA_F32, SSA_BF16, SSA_F16 = 0, 1, 2
SSA_OP_ROUTE, SSA_OP_DECODE, SSA_OP_PREFILL, SSA_OP_ROUTE_GROUP = 0, 1, 2, 3
SSA_DEVERR_BAD_SELECTION = 0x1
SSA_DEVERR_WAIT_TIMEOUT = 0x2
SSA_DEVERR_OVERFLOW = 0x4

DTYPE_CODE = {torch.float32: SSA_F32, torch.bfloat16: SSA_BF16, torch.float16: SSA_F16}


class ssa_params(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
        ("d", ctypes.c_int32), ("L", ctypes.c_int64), ("L_cap", ctypes.c_int64),
        ("S", ctypes.c_int32), ("topk", ctypes.c_int32), ("scale", ctypes.c_float),
        ("dtype", ctypes.c_int32),
    ]


class SSAError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__("%s: %s (status %d)" % (what, ssa_status_string(status), status))
        self.status = status


_lib = None
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t


def library_path() -> str:
    return _build.SO


def lib() -> ctypes.CDLL:
    """Load libssa.so, building it first if it is missing or stale."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        PP = ctypes.POINTER(ssa_params)
        L.ssa_build_summaries.argtypes = [PP, _P, _I64, _I64, _P, _P]
        L.ssa_route.argtypes = [PP, _P, _I64, _I64, _P, _P, _P, _P, _SZ, _P]
        L.ssa_route_group.argtypes = [PP, _P, _I64, _I64, _P, _P, _P, _P, _SZ, _P]
        L.ssa_attend_decode.argtypes = [PP, _P, _I64, _P, _P, _P, _P, _P, _P, _SZ, _P]
        L.ssa_attend_prefill.argtypes = [PP, _P, _I64, _I64, _P, _P, _P, _P, _P, _P, _SZ, _P]
        L.ssa_workspace_size.argtypes = [PP, _I64, ctypes.c_int]
        L.ssa_workspace_size.restype = _SZ
        L.ssa_workspace_error.argtypes = [_P, ctypes.POINTER(ctypes.c_uint32), _P]
        L.ssa_status_string.argtypes = [ctypes.c_int]
        L.ssa_status_string.restype = ctypes.c_char_p
        L.ssa_version.restype = ctypes.c_int
        for name in ("ssa_build_summaries", "ssa_route", "ssa_route_group", "ssa_attend_decode",
                     "ssa_attend_prefill", "ssa_workspace_error"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def params(B: int, Hq: int, Hkv: int, d: int, L: int, S: int, topk: int, dtype, L_cap: int = 0,
           scale: float = 0.0) -> ssa_params:
    code = DTYPE_CODE[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return ssa_params(B, Hq, Hkv, d, L, L_cap, S, topk, scale, code)


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    return ctypes.c_void_p(int(stream))


def _check(rc: int, what: str) -> None:
    if rc != SSA_OK:
        raise SSAError(rc, what)


def ssa_status_string(status: int) -> str:
    return lib().ssa_status_string(int(status)).decode()


def ssa_workspace_size(p: ssa_params, n_q: int, op: int) -> int:
    return int(lib().ssa_workspace_size(ctypes.byref(p), int(n_q), int(op)))


def workspace(p: ssa_params, n_q: int, op: int, device=None) -> torch.Tensor | None:
    """A zeroed workspace tensor of the size the operation needs (None if 0)."""
    n = ssa_workspace_size(p, n_q, op)
    if n == 0:
        return None
    t = torch.zeros(n + 256, dtype=torch.uint8, device=device or "cuda")
    off = (-t.data_ptr()) % 256
    return t[off: off + n]


def _ws_args(ws: torch.Tensor | None):
    if ws is None:
        return None, 0
    return ctypes.c_void_p(ws.data_ptr()), ws.numel() * ws.element_size()


def ssa_build_summaries(p: ssa_params, K: torch.Tensor, span_begin: int, span_end: int,
                        summ: torch.Tensor, stream=None) -> None:
    rc = lib().ssa_build_summaries(ctypes.byref(p), _ptr(K), int(span_begin), int(span_end),
                                   _ptr(summ), _stream(stream))
    _check(rc, "ssa_build_summaries")


def ssa_route(p: ssa_params, Q: torch.Tensor, n_q: int, q_pos0: int, summ: torch.Tensor,
              sel: torch.Tensor, sel_score: torch.Tensor | None = None,
              ws: torch.Tensor | None = None, stream=None) -> None:
    wp, wn = _ws_args(ws)
    rc = lib().ssa_route(ctypes.byref(p), _ptr(Q), int(n_q), int(q_pos0), _ptr(summ), _ptr(sel),
                         _ptr(sel_score), wp, wn, _stream(stream))
    _check(rc, "ssa_route")


def ssa_route_group(p: ssa_params, Q: torch.Tensor, n_q: int, q_pos0: int, summ: torch.Tensor,
                    sel: torch.Tensor, sel_score: torch.Tensor | None = None,
                    ws: torch.Tensor | None = None, stream=None) -> None:
    wp, wn = _ws_args(ws)
    rc = lib().ssa_route_group(ctypes.byref(p), _ptr(Q), int(n_q), int(q_pos0), _ptr(summ), _ptr(sel),
                               _ptr(sel_score), wp, wn, _stream(stream))
    _check(rc, "ssa_route_group")


def ssa_attend_decode(p: ssa_params, Q: torch.Tensor, pos: int, K: torch.Tensor, V: torch.Tensor,
                      sel: torch.Tensor, O: torch.Tensor, lse: torch.Tensor | None,
                      ws: torch.Tensor | None, stream=None) -> None:
    wp, wn = _ws_args(ws)
    rc = lib().ssa_attend_decode(ctypes.byref(p), _ptr(Q), int(pos), _ptr(K), _ptr(V), _ptr(sel),
                                 _ptr(O), _ptr(lse), wp, wn, _stream(stream))
    _check(rc, "ssa_attend_decode")


def ssa_attend_prefill(p: ssa_params, Q: torch.Tensor, n_q: int, q_pos0: int, K: torch.Tensor,
                       V: torch.Tensor, sel: torch.Tensor, O: torch.Tensor,
                       lse: torch.Tensor | None, ws: torch.Tensor | None, stream=None) -> None:
    wp, wn = _ws_args(ws)
    rc = lib().ssa_attend_prefill(ctypes.byref(p), _ptr(Q), int(n_q), int(q_pos0), _ptr(K),
                                  _ptr(V), _ptr(sel), _ptr(O), _ptr(lse), wp, wn, _stream(stream))
    _check(rc, "ssa_attend_prefill")


class ScratchBlock:
    """The library-owned decode scratch of one device, as returned by
    ssa_attend_decode_noalloc; pass it to ssa_workspace_error."""

    def __init__(self, address: int):
        self.address = address

    def data_ptr(self) -> int:
        return self.address


SSA_NOALLOC_SCRATCH_BYTES = 8 << 20


def ssa_attend_decode_noalloc(p: ssa_params, Q: torch.Tensor, pos: int, K: torch.Tensor,
                              V: torch.Tensor, sel: torch.Tensor, O: torch.Tensor,
                              lse: torch.Tensor | None, stream=None) -> ScratchBlock:
    """ssa_attend_decode on the library's own scratch block; returns the block."""
    f = lib().ssa_attend_decode_noalloc
    f.argtypes = [ctypes.POINTER(ssa_params), _P, _I64, _P, _P, _P, _P, _P, ctypes.POINTER(_P), _P]
    f.restype = ctypes.c_int
    scratch = _P(0)
    rc = f(ctypes.byref(p), _ptr(Q), int(pos), _ptr(K), _ptr(V), _ptr(sel), _ptr(O), _ptr(lse),
           ctypes.byref(scratch), _stream(stream))
    _check(rc, "ssa_attend_decode_noalloc")
    return ScratchBlock(int(scratch.value))


def ssa_workspace_error(ws: torch.Tensor, stream=None) -> int:
    """Synchronise, read and clear the device error record; returns its bits."""
    bits = ctypes.c_uint32(0)
    rc = lib().ssa_workspace_error(_ptr(ws), ctypes.byref(bits), _stream(stream))
    if rc not in (SSA_OK, SSA_ERR_DEVICE):
        raise SSAError(rc, "ssa_workspace_error")
    return int(bits.value)


def ssa_version() -> int:
    return int(lib().ssa_version())
