"""Seeded synthetic inputs for content-routed sparse attention.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle's tests.  It creates input tensors only: the per-element values
(synth_core.h) and the structure added to the keys (needle spans and a
per-span low-rank term, built here in float64 from the same seeded values).
It holds none of the attention method's arithmetic.

Elements are addressed by their linear index in the full tensor, so any
sub-range (a span of one head, a single query row) can be regenerated on its
own, on the host or on the device, with identical bits.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from . import build as _build

# Tensor ids: one Philox key stream per role.
TID_Q = 1
TID_K = 2
TID_V = 3
TID_LOWRANK_W = 5
TID_LOWRANK_Z = 6
TID_NEEDLE = 7

_DTYPE_CODE = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}

_host = None
_dev = None


def _host_lib():
    global _host
    if _host is None:
        lib = ctypes.CDLL(_build.build_host())
        lib.synth_fill_host.restype = ctypes.c_int
        lib.synth_fill_host.argtypes = [
            ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_uint32, ctypes.c_uint32, ctypes.c_int32]
        lib.synth_philox_block.argtypes = [ctypes.c_void_p] * 3
        lib.synth_round_f32.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                        ctypes.c_void_p]
        _host = lib
    return _host


def _dev_lib():
    global _dev
    if _dev is None:
        lib = ctypes.CDLL(_build.build_device())
        lib.synth_fill_device.restype = ctypes.c_int
        lib.synth_fill_device.argtypes = [
            ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_uint32, ctypes.c_uint32, ctypes.c_void_p]
        _dev = lib
    return _dev


def host_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def philox_block(ctr, key) -> np.ndarray:
    """One Philox4x32-10 output block (4 words), for known-answer tests."""
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
    o = np.zeros(4, np.uint32)
    _host_lib().synth_philox_block(c.ctypes.data, k.ctypes.data, o.ctypes.data)
    return o


def round_f32(x: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    """The generator's fp32 -> bf16/fp16 rounding, returned as raw uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.zeros(x.shape, np.uint16)
    _host_lib().synth_round_f32(x.ctypes.data, x.size, _DTYPE_CODE[dtype], out.ctypes.data)
    return out


def fill_(out: torch.Tensor, seed: int, tid: int, *, e0: int = 0, d: int | None = None,
          attempt: torch.Tensor | None = None, bias: torch.Tensor | None = None,
          rows_per_head: int = 0, S: int = 0, stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """Write elements [e0, e0 + out.numel()) of the tensor (seed, tid) into ``out``.

    ``d`` is the row length (defaults to out.shape[-1]).  ``attempt`` holds one
    int32 per global row of the full tensor (redraws rows); ``bias`` is the
    fp32 table [heads, ceil(rows_per_head / S), d] added to rows of head
    ``row // rows_per_head`` in block ``(row % rows_per_head) // S``.  All
    tensors must live on out's device.
    """
    if not out.is_contiguous():
        raise ValueError("out must be contiguous")
    if out.dtype not in _DTYPE_CODE:
        raise ValueError("unsupported dtype %s" % out.dtype)
    d = int(d if d is not None else out.shape[-1])
    n = out.numel()
    for t in (attempt, bias):
        if t is not None and (t.device != out.device or not t.is_contiguous()):
            raise ValueError("attempt/bias must be contiguous and on out's device")
    if attempt is not None and attempt.dtype != torch.int32:
        raise ValueError("attempt must be int32")
    if bias is not None and bias.dtype != torch.float32:
        raise ValueError("bias must be float32")
    ap = attempt.data_ptr() if attempt is not None else None
    bp = bias.data_ptr() if bias is not None else None
    if out.device.type == "cpu":
        rc = _host_lib().synth_fill_host(_DTYPE_CODE[out.dtype], out.data_ptr(), e0, e0 + n, d,
                                         rows_per_head, S, bp, ap, seed & 0xffffffff, tid,
                                         host_threads())
    else:
        st = stream if stream is not None else torch.cuda.current_stream(out.device)
        with torch.cuda.device(out.device):
            rc = _dev_lib().synth_fill_device(_DTYPE_CODE[out.dtype], out.data_ptr(), e0, e0 + n,
                                              d, rows_per_head, S, bp, ap, seed & 0xffffffff,
                                              tid, ctypes.c_void_p(st.cuda_stream))
    if rc != 0:
        raise RuntimeError("synth fill failed with code %d" % rc)
    return out


def normal(shape, dtype: torch.dtype, seed: int, tid: int, device="cpu", **kw) -> torch.Tensor:
    """A full tensor of the generator's approximately-N(0,1) values."""
    out = torch.empty(tuple(shape), dtype=dtype, device=device)
    return fill_(out, seed, tid, **kw)


def f64_values(n: int, seed: int, tid: int) -> np.ndarray:
    """n fp32 generator values of stream (seed, tid), widened to float64."""
    t = torch.empty(n, dtype=torch.float32)
    fill_(t, seed, tid, d=1)
    return t.numpy().astype(np.float64)


def stats_hint() -> str:
    return "Irwin-Hall(8) approximation of N(0,1): mean 0, variance 1, range +-4.9"
