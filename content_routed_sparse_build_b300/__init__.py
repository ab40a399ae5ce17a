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
  ssa_decode_step      route + attend of one decode step (three launches)
  ssa_attend_prefill   a chunk of queries, span-major tiles, LSE merge
  ssa_attend_decode_noalloc  ssa_attend_decode on a library-owned scratch block
  ssa_quantize_kv / ssa_build_summaries_q8 / ssa_attend_decode_q8 / ssa_decode_step_q8
                       the 8-bit cache: quantised rows, their summaries, decode over them
  ssa_quantize_kv4 / ssa_build_summaries_q4 / ssa_attend_decode_q4 / ssa_decode_step_q4
                       the same for the 4-bit cache
  ssa_snapshot_save / ssa_snapshot_load / ssa_snapshot_read_header
                       the cache rows and summaries of a session, to and from a file
  ssa_workspace_size / ssa_workspace_error / ssa_status_string
  ssa_attend_path      which implementation an attention call takes
  ssa_selftest_wait_timeout
                       a bounded wait run out on purpose: the status path of every kernel
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
SSA_ERR_IO = 6

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
        L.ssa_decode_step.argtypes = [PP, _P, _I64, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]
        L.ssa_workspace_size.argtypes = [PP, _I64, ctypes.c_int]
        L.ssa_workspace_size.restype = _SZ
        L.ssa_workspace_error.argtypes = [_P, ctypes.POINTER(ctypes.c_uint32), _P]
        L.ssa_status_string.argtypes = [ctypes.c_int]
        L.ssa_status_string.restype = ctypes.c_char_p
        L.ssa_version.restype = ctypes.c_int
        for name in ("ssa_build_summaries", "ssa_route", "ssa_route_group", "ssa_attend_decode",
                     "ssa_attend_prefill", "ssa_decode_step", "ssa_workspace_error"):
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


SSA_PATH_INVALID, SSA_PATH_FAST, SSA_PATH_ROWS = 0, 1, 2


def ssa_attend_path(p: ssa_params, n_q: int, op: int) -> int:
    """Which implementation an attention call takes (SSA_PATH_*); host only."""
    f = lib().ssa_attend_path
    f.argtypes = [ctypes.POINTER(ssa_params), _I64, ctypes.c_int]
    f.restype = ctypes.c_int
    return int(f(ctypes.byref(p), int(n_q), int(op)))


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


def ssa_decode_step(p: ssa_params, Q: torch.Tensor, pos: int, summ: torch.Tensor, K: torch.Tensor,
                    V: torch.Tensor, sel: torch.Tensor, O: torch.Tensor, lse: torch.Tensor | None,
                    ws: torch.Tensor | None, stream=None) -> None:
    wp, wn = _ws_args(ws)
    rc = lib().ssa_decode_step(ctypes.byref(p), _ptr(Q), int(pos), _ptr(summ), _ptr(K), _ptr(V), _ptr(sel),
                               _ptr(O), _ptr(lse), wp, wn, _stream(stream))
    _check(rc, "ssa_decode_step")


def ssa_decode_step_group(p: ssa_params, Q: torch.Tensor, pos: int, summ: torch.Tensor, K: torch.Tensor,
                          V: torch.Tensor, sel: torch.Tensor, O: torch.Tensor, lse: torch.Tensor | None,
                          ws: torch.Tensor | None, stream=None) -> None:
    f = lib().ssa_decode_step_group
    f.argtypes = [ctypes.POINTER(ssa_params), _P, _I64, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]
    f.restype = ctypes.c_int
    wp, wn = _ws_args(ws)
    _check(f(ctypes.byref(p), _ptr(Q), int(pos), _ptr(summ), _ptr(K), _ptr(V), _ptr(sel), _ptr(O), _ptr(lse), wp,
             wn, _stream(stream)), "ssa_decode_step_group")


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


def q8_cache(p: ssa_params, device=None):
    """Empty 8-bit cache tensors (Kq, Ks, Vq, Vs) laid out for p (L_cap a
    multiple of 32)."""
    L_cap = p.L_cap or p.L
    if L_cap % 32:
        raise ValueError("the 8-bit cache needs L_cap % 32 == 0")
    dev = device if device is not None else torch.device("cuda")
    Kq = torch.empty((p.B, p.Hkv, L_cap, p.d), dtype=torch.int8, device=dev)
    Vq = torch.empty((p.B, p.Hkv, L_cap // 32, p.d, 32), dtype=torch.int8, device=dev)
    Ks = torch.empty((p.B, p.Hkv, L_cap), dtype=torch.float32, device=dev)
    Vs = torch.empty((p.B, p.Hkv, L_cap), dtype=torch.float32, device=dev)
    return Kq, Ks, Vq, Vs


def ssa_quantize_kv(p: ssa_params, K: torch.Tensor, V: torch.Tensor, t_begin: int, t_end: int,
                    Kq: torch.Tensor, Ks: torch.Tensor, Vq: torch.Tensor, Vs: torch.Tensor, stream=None) -> None:
    f = lib().ssa_quantize_kv
    f.argtypes = [ctypes.POINTER(ssa_params), _P, _P, _I64, _I64, _P, _P, _P, _P, _P]
    f.restype = ctypes.c_int
    _check(f(ctypes.byref(p), _ptr(K), _ptr(V), int(t_begin), int(t_end), _ptr(Kq), _ptr(Ks), _ptr(Vq),
             _ptr(Vs), _stream(stream)), "ssa_quantize_kv")


def ssa_build_summaries_q8(p: ssa_params, Kq: torch.Tensor, Ks: torch.Tensor, span_begin: int, span_end: int,
                           summ: torch.Tensor, stream=None) -> None:
    f = lib().ssa_build_summaries_q8
    f.argtypes = [ctypes.POINTER(ssa_params), _P, _P, _I64, _I64, _P, _P]
    f.restype = ctypes.c_int
    _check(f(ctypes.byref(p), _ptr(Kq), _ptr(Ks), int(span_begin), int(span_end), _ptr(summ), _stream(stream)),
           "ssa_build_summaries_q8")


def ssa_attend_decode_q8(p: ssa_params, Q: torch.Tensor, pos: int, Kq: torch.Tensor, Ks: torch.Tensor,
                         Vq: torch.Tensor, Vs: torch.Tensor, sel: torch.Tensor, O: torch.Tensor,
                         lse: torch.Tensor | None, ws: torch.Tensor | None, stream=None) -> None:
    f = lib().ssa_attend_decode_q8
    f.argtypes = [ctypes.POINTER(ssa_params), _P, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]
    f.restype = ctypes.c_int
    wp, wn = _ws_args(ws)
    _check(f(ctypes.byref(p), _ptr(Q), int(pos), _ptr(Kq), _ptr(Ks), _ptr(Vq), _ptr(Vs), _ptr(sel), _ptr(O),
             _ptr(lse), wp, wn, _stream(stream)), "ssa_attend_decode_q8")


def q4_cache(p: ssa_params, device=None):
    """Zeroed 4-bit cache tensors (Kq4, Ks, Vq4, Vs) laid out for p (d = 128,
    L_cap a multiple of 32): Kq4 and Vq4 as int32 words [B, Hkv, L_cap / 32,
    512], the scales fp32 [B, Hkv, L_cap]."""
    L_cap = p.L_cap or p.L
    if L_cap % 32 or p.d != 128:
        raise ValueError("the 4-bit cache needs d == 128 and L_cap % 32 == 0")
    dev = device if device is not None else torch.device("cuda")
    Kq4 = torch.zeros((p.B, p.Hkv, L_cap // 32, 512), dtype=torch.int32, device=dev)
    Vq4 = torch.zeros((p.B, p.Hkv, L_cap // 32, 512), dtype=torch.int32, device=dev)
    Ks = torch.empty((p.B, p.Hkv, L_cap), dtype=torch.float32, device=dev)
    Vs = torch.empty((p.B, p.Hkv, L_cap), dtype=torch.float32, device=dev)
    return Kq4, Ks, Vq4, Vs


def ssa_quantize_kv4(p: ssa_params, K: torch.Tensor, V: torch.Tensor, t_begin: int, t_end: int, Kq4: torch.Tensor,
                     Ks: torch.Tensor, Vq4: torch.Tensor, Vs: torch.Tensor, stream=None) -> None:
    f = lib().ssa_quantize_kv4
    f.argtypes = [ctypes.POINTER(ssa_params), _P, _P, _I64, _I64, _P, _P, _P, _P, _P]
    f.restype = ctypes.c_int
    _check(f(ctypes.byref(p), _ptr(K), _ptr(V), int(t_begin), int(t_end), _ptr(Kq4), _ptr(Ks), _ptr(Vq4), _ptr(Vs),
             _stream(stream)), "ssa_quantize_kv4")


def ssa_build_summaries_q4(p: ssa_params, Kq4: torch.Tensor, Ks: torch.Tensor, span_begin: int, span_end: int,
                           summ: torch.Tensor, stream=None) -> None:
    f = lib().ssa_build_summaries_q4
    f.argtypes = [ctypes.POINTER(ssa_params), _P, _P, _I64, _I64, _P, _P]
    f.restype = ctypes.c_int
    _check(f(ctypes.byref(p), _ptr(Kq4), _ptr(Ks), int(span_begin), int(span_end), _ptr(summ), _stream(stream)),
           "ssa_build_summaries_q4")


def ssa_attend_decode_q4(p: ssa_params, Q: torch.Tensor, pos: int, Kq4: torch.Tensor, Ks: torch.Tensor,
                         Vq4: torch.Tensor, Vs: torch.Tensor, sel: torch.Tensor, O: torch.Tensor,
                         lse: torch.Tensor | None, ws: torch.Tensor | None, stream=None) -> None:
    f = lib().ssa_attend_decode_q4
    f.argtypes = [ctypes.POINTER(ssa_params), _P, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]
    f.restype = ctypes.c_int
    wp, wn = _ws_args(ws)
    _check(f(ctypes.byref(p), _ptr(Q), int(pos), _ptr(Kq4), _ptr(Ks), _ptr(Vq4), _ptr(Vs), _ptr(sel), _ptr(O),
             _ptr(lse), wp, wn, _stream(stream)), "ssa_attend_decode_q4")


def ssa_decode_step_q4(p: ssa_params, Q: torch.Tensor, pos: int, summ: torch.Tensor, Kq4: torch.Tensor,
                       Ks: torch.Tensor, Vq4: torch.Tensor, Vs: torch.Tensor, sel: torch.Tensor, O: torch.Tensor,
                       lse: torch.Tensor | None, ws: torch.Tensor | None, stream=None) -> None:
    f = lib().ssa_decode_step_q4
    f.argtypes = [ctypes.POINTER(ssa_params), _P, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]
    f.restype = ctypes.c_int
    wp, wn = _ws_args(ws)
    _check(f(ctypes.byref(p), _ptr(Q), int(pos), _ptr(summ), _ptr(Kq4), _ptr(Ks), _ptr(Vq4), _ptr(Vs), _ptr(sel),
             _ptr(O), _ptr(lse), wp, wn, _stream(stream)), "ssa_decode_step_q4")


def ssa_selftest_wait_timeout(limit_ns: int, ws: torch.Tensor, stream=None) -> None:
    """Runs the bounded-wait self test: a wait on a barrier nothing completes
    gives up after limit_ns and records SSA_DEVERR_WAIT_TIMEOUT in ws."""
    f = lib().ssa_selftest_wait_timeout
    f.argtypes = [ctypes.c_uint64, _P, _SZ, _P]
    f.restype = ctypes.c_int
    wp, wn = _ws_args(ws)
    _check(f(int(limit_ns), wp, wn, _stream(stream)), "ssa_selftest_wait_timeout")


def ssa_decode_step_q8(p: ssa_params, Q: torch.Tensor, pos: int, summ: torch.Tensor, Kq: torch.Tensor,
                       Ks: torch.Tensor, Vq: torch.Tensor, Vs: torch.Tensor, sel: torch.Tensor, O: torch.Tensor,
                       lse: torch.Tensor | None, ws: torch.Tensor | None, stream=None) -> None:
    f = lib().ssa_decode_step_q8
    f.argtypes = [ctypes.POINTER(ssa_params), _P, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]
    f.restype = ctypes.c_int
    wp, wn = _ws_args(ws)
    _check(f(ctypes.byref(p), _ptr(Q), int(pos), _ptr(summ), _ptr(Kq), _ptr(Ks), _ptr(Vq), _ptr(Vs), _ptr(sel),
             _ptr(O), _ptr(lse), wp, wn, _stream(stream)), "ssa_decode_step_q8")


SSA_SNAPSHOT_MAGIC = b"SSAKVSN1"
SSA_SNAPSHOT_VERSION = 1


class ssa_snapshot_header(ctypes.Structure):
    _fields_ = [("magic", ctypes.c_char * 8), ("version", ctypes.c_uint32), ("dtype", ctypes.c_int32),
                ("B", ctypes.c_int32), ("Hkv", ctypes.c_int32), ("d", ctypes.c_int32), ("S", ctypes.c_int32),
                ("n_tokens", ctypes.c_int64), ("n_summ", ctypes.c_int64), ("payload_bytes", ctypes.c_uint64),
                ("reserved", ctypes.c_uint8 * 8)]


def _staging(staging, nbytes: int):
    """(pointer, bytes) of a staging buffer: the caller's host tensor, or a
    fresh page-locked one of nbytes."""
    if staging is None:
        staging = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    return staging, _P(staging.data_ptr()), staging.numel() * staging.element_size()


def ssa_snapshot_save(p: ssa_params, n_tokens: int, K: torch.Tensor, V: torch.Tensor, summ: torch.Tensor,
                      path: str, staging: torch.Tensor | None = None, stream=None) -> None:
    """Write rows 0 .. n_tokens-1 of K and V and the complete spans' summaries to path."""
    f = lib().ssa_snapshot_save
    f.argtypes = [ctypes.POINTER(ssa_params), _I64, _P, _P, _P, ctypes.c_char_p, _P, _SZ, _P]
    f.restype = ctypes.c_int
    buf, ptr, nb = _staging(staging, 64 << 20)
    rc = f(ctypes.byref(p), int(n_tokens), _ptr(K), _ptr(V), _ptr(summ), os.fsencode(path), ptr, nb,
           _stream(stream))
    _check(rc, "ssa_snapshot_save")


def ssa_snapshot_load(p: ssa_params, path: str, K: torch.Tensor, V: torch.Tensor, summ: torch.Tensor,
                      staging: torch.Tensor | None = None, stream=None) -> int:
    """Restore a snapshot into K, V and summ; returns its n_tokens."""
    f = lib().ssa_snapshot_load
    f.argtypes = [ctypes.POINTER(ssa_params), ctypes.c_char_p, _P, _P, _P, ctypes.POINTER(_I64), _P, _SZ, _P]
    f.restype = ctypes.c_int
    buf, ptr, nb = _staging(staging, 64 << 20)
    n = _I64(0)
    rc = f(ctypes.byref(p), os.fsencode(path), _ptr(K), _ptr(V), _ptr(summ), ctypes.byref(n), ptr, nb,
           _stream(stream))
    _check(rc, "ssa_snapshot_load")
    return int(n.value)


def ssa_snapshot_read_header(path: str) -> ssa_snapshot_header:
    """The checked header of a snapshot file (host only)."""
    f = lib().ssa_snapshot_read_header
    f.argtypes = [ctypes.c_char_p, ctypes.POINTER(ssa_snapshot_header)]
    f.restype = ctypes.c_int
    h = ssa_snapshot_header()
    _check(f(os.fsencode(path), ctypes.byref(h)), "ssa_snapshot_read_header")
    return h


def ssa_workspace_error(ws: torch.Tensor, stream=None) -> int:
    """Synchronise, read and clear the device error record; returns its bits."""
    bits = ctypes.c_uint32(0)
    rc = lib().ssa_workspace_error(_ptr(ws), ctypes.byref(bits), _stream(stream))
    if rc not in (SSA_OK, SSA_ERR_DEVICE):
        raise SSAError(rc, "ssa_workspace_error")
    return int(bits.value)


def ssa_version() -> int:
    return int(lib().ssa_version())
