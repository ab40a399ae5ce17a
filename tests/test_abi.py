"""The C ABI: the library loads, exports every symbol include/*.h declares,
and rejects bad arguments on the host before anything reaches a GPU."""
import ctypes
import glob
import os
import re

import pytest
import torch

import content_routed_sparse_build_b300 as ssa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        names += re.findall(r"SSA_API\s+[\w\s\*]+?\b(ssa_\w+)\s*\(", src)
    return sorted(set(names))


def test_every_declared_symbol_is_exported():
    names = _declared()
    assert {"ssa_build_summaries", "ssa_route", "ssa_attend_decode", "ssa_attend_prefill",
            "ssa_workspace_size", "ssa_status_string"} <= set(names)
    lib = ctypes.CDLL(ssa.library_path() if os.path.exists(ssa.library_path()) else ssa.lib()._name)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version():
    for s in range(6):
        assert ssa.ssa_status_string(s) and ssa.ssa_status_string(s) != "unknown status"
    assert ssa.ssa_status_string(99) == "unknown status"
    assert ssa.ssa_version() >= 100


def test_workspace_sizes():
    p = ssa.params(1, 32, 4, 128, 1 << 20, 1024, 16, torch.bfloat16)
    assert ssa.ssa_workspace_size(p, 1, ssa.SSA_OP_ROUTE) == 0
    assert ssa.ssa_workspace_size(p, 1, ssa.SSA_OP_DECODE) >= 256
    assert ssa.ssa_workspace_size(p, 8192, ssa.SSA_OP_PREFILL) >= 256
    bad = ssa.params(1, 32, 4, 96, 1 << 20, 1024, 16, torch.bfloat16)
    assert ssa.ssa_workspace_size(bad, 1, ssa.SSA_OP_DECODE) == 0


# The calls below pass pointer values that are never dereferenced: each one
# is rejected by host validation.  They are kept off machines with a GPU.
needs_no_gpu = pytest.mark.skipif(torch.cuda.is_available(), reason="host-validation only")
FAKE = ctypes.c_void_p(4096)


def _call_route(p, Q=FAKE, n_q=1, pos=0, summ=FAKE, sel=FAKE):
    return ssa.lib().ssa_route(ctypes.byref(p), Q, n_q, pos, summ, sel, None, None, 0, None)


@needs_no_gpu
def test_route_validation():
    ok = ssa.params(1, 8, 2, 128, 4096, 64, 8, torch.bfloat16)
    assert _call_route(ok, Q=None) == ssa.SSA_ERR_INVALID_ARG
    assert _call_route(ok, sel=None) == ssa.SSA_ERR_INVALID_ARG
    assert _call_route(ok, Q=ctypes.c_void_p(4098)) == ssa.SSA_ERR_INVALID_ARG   # misaligned
    assert _call_route(ok, pos=4096) == ssa.SSA_ERR_INVALID_ARG                  # beyond L
    assert _call_route(ok, n_q=-1) == ssa.SSA_ERR_INVALID_ARG
    assert _call_route(ssa.params(1, 8, 3, 128, 4096, 64, 8, 1)) == ssa.SSA_ERR_INVALID_ARG
    assert _call_route(ssa.params(1, 8, 2, 96, 4096, 64, 8, 1)) == ssa.SSA_ERR_UNSUPPORTED
    assert _call_route(ssa.params(1, 8, 2, 128, 4096, 64, 65, 1)) == ssa.SSA_ERR_UNSUPPORTED
    assert _call_route(ssa.params(1, 64, 2, 128, 4096, 64, 8, 1)) == ssa.SSA_ERR_UNSUPPORTED
    assert _call_route(ssa.params(1, 8, 2, 128, 4096, 0, 8, 1)) == ssa.SSA_ERR_INVALID_ARG
    assert _call_route(ssa.params(1, 8, 2, 128, 4096, 64, 8, 7)) == ssa.SSA_ERR_INVALID_ARG
    assert _call_route(ssa.params(1, 8, 2, 128, 4096, 64, 8, 1, L_cap=100)) == ssa.SSA_ERR_INVALID_ARG
    assert _call_route(ssa.params(1, 8, 2, 128, 4096, 64, 8, 1, scale=-1.0)) == ssa.SSA_ERR_INVALID_ARG
    assert _call_route(ssa.params(1, 8, 2, 128, 4096, 64, 8, 1, scale=float("nan"))) == ssa.SSA_ERR_INVALID_ARG
    assert ssa.lib().ssa_route(None, FAKE, 1, 0, FAKE, FAKE, None, None, 0, None) == ssa.SSA_ERR_INVALID_ARG


@needs_no_gpu
def test_attend_and_summary_validation():
    p = ssa.params(1, 8, 2, 128, 4096, 64, 8, torch.bfloat16)
    L = ssa.lib()
    need = ssa.ssa_workspace_size(p, 1, ssa.SSA_OP_DECODE)
    args = lambda pos, ws, n: (ctypes.byref(p), FAKE, pos, FAKE, FAKE, FAKE, FAKE, None, ws, n, None)
    assert L.ssa_attend_decode(*args(4096, FAKE, need)) == ssa.SSA_ERR_INVALID_ARG
    assert L.ssa_attend_decode(*args(-1, FAKE, need)) == ssa.SSA_ERR_INVALID_ARG
    assert L.ssa_attend_decode(*args(10, None, 0)) == ssa.SSA_ERR_WORKSPACE
    assert L.ssa_attend_decode(*args(10, FAKE, need - 1)) == ssa.SSA_ERR_WORKSPACE
    assert L.ssa_attend_decode(*args(10, ctypes.c_void_p(4096 + 16), need)) == ssa.SSA_ERR_WORKSPACE
    need_p = ssa.ssa_workspace_size(p, 100, ssa.SSA_OP_PREFILL)
    pre = lambda n_q, q0, ws, n: (ctypes.byref(p), FAKE, n_q, q0, FAKE, FAKE, FAKE, FAKE, None, ws, n, None)
    assert L.ssa_attend_prefill(*pre(100, 4000, FAKE, need_p)) == ssa.SSA_ERR_INVALID_ARG
    assert L.ssa_attend_prefill(*pre(100, 0, None, 0)) == ssa.SSA_ERR_WORKSPACE
    assert L.ssa_build_summaries(ctypes.byref(p), FAKE, 0, 65, FAKE, None) == ssa.SSA_ERR_INVALID_ARG
    assert L.ssa_build_summaries(ctypes.byref(p), FAKE, 5, 4, FAKE, None) == ssa.SSA_ERR_INVALID_ARG
    assert L.ssa_build_summaries(ctypes.byref(p), None, 0, 4, FAKE, None) == ssa.SSA_ERR_INVALID_ARG
    assert L.ssa_workspace_error(None, None, None) == ssa.SSA_ERR_WORKSPACE


@needs_no_gpu
def test_route_group_validation_and_workspace():
    p = ssa.params(1, 32, 4, 128, 1 << 20, 1024, 16, torch.bfloat16)
    n = ssa.ssa_workspace_size(p, 8192, ssa.SSA_OP_ROUTE_GROUP)
    # header + the summed queries (fp32) + the group selections and scores
    assert n >= 256 + 4 * 8192 * 128 * 4 + 2 * 4 * 8192 * 16 * 4
    L = ssa.lib()
    call = lambda p, ws=None, wsn=0, **kw: L.ssa_route_group(
        ctypes.byref(p), kw.get("Q", FAKE), kw.get("n_q", 1), kw.get("pos", 0), FAKE, FAKE, None,
        ws, wsn, None)
    assert call(p) == ssa.SSA_ERR_WORKSPACE                       # missing workspace
    assert call(p, ws=ctypes.c_void_p(4096), wsn=16) == ssa.SSA_ERR_WORKSPACE
    assert call(p, Q=None) == ssa.SSA_ERR_INVALID_ARG
    assert call(ssa.params(1, 8, 3, 128, 4096, 64, 8, 1)) == ssa.SSA_ERR_INVALID_ARG


@needs_no_gpu
def test_q8_validation():
    L = ssa.lib()
    P, I8 = ctypes.c_void_p, ctypes.c_int64
    L.ssa_quantize_kv.argtypes = [ctypes.POINTER(ssa.ssa_params), P, P, I8, I8, P, P, P, P, P]
    L.ssa_build_summaries_q8.argtypes = [ctypes.POINTER(ssa.ssa_params), P, P, I8, I8, P, P]
    L.ssa_attend_decode_q8.argtypes = [ctypes.POINTER(ssa.ssa_params), P, I8, P, P, P, P, P, P, P, P,
                                       ctypes.c_size_t, P]
    p = ssa.params(1, 8, 2, 128, 4096, 64, 8, torch.bfloat16)
    q = lambda p, t0, t1, **kw: L.ssa_quantize_kv(ctypes.byref(p), FAKE, kw.get("V", FAKE), t0, t1, FAKE, FAKE,
                                                  FAKE, FAKE, None)
    assert q(p, 0, 4097) == ssa.SSA_ERR_INVALID_ARG             # past L
    assert q(p, 10, 5) == ssa.SSA_ERR_INVALID_ARG
    assert q(p, 0, 10, V=None) == ssa.SSA_ERR_INVALID_ARG
    assert q(ssa.params(1, 8, 2, 128, 4001, 64, 8, torch.bfloat16), 0, 10) == ssa.SSA_ERR_UNSUPPORTED  # L_cap % 32
    assert L.ssa_build_summaries_q8(ctypes.byref(p), FAKE, FAKE, 0, 65, FAKE, None) == ssa.SSA_ERR_INVALID_ARG
    need = ssa.ssa_workspace_size(p, 1, ssa.SSA_OP_DECODE)
    d = lambda p, pos, ws, n: L.ssa_attend_decode_q8(ctypes.byref(p), FAKE, pos, FAKE, FAKE, FAKE, FAKE, FAKE,
                                                     FAKE, None, ws, n, None)
    assert d(p, 4096, FAKE, need) == ssa.SSA_ERR_INVALID_ARG          # pos == L
    assert d(p, 10, None, 0) == ssa.SSA_ERR_WORKSPACE
    assert d(ssa.params(1, 8, 2, 64, 4096, 64, 8, torch.bfloat16), 10, FAKE, need) == ssa.SSA_ERR_UNSUPPORTED
    assert d(ssa.params(1, 8, 2, 128, 4096, 64, 8, torch.float32), 10, FAKE, need) == ssa.SSA_ERR_UNSUPPORTED
    # the fused 8-bit step takes what the 8-bit attention takes, plus the summaries
    L.ssa_decode_step_q8.argtypes = [ctypes.POINTER(ssa.ssa_params), P, I8, P, P, P, P, P, P, P, P, P,
                                     ctypes.c_size_t, P]
    st = lambda p, pos, ws, n, **kw: L.ssa_decode_step_q8(
        ctypes.byref(p), FAKE, pos, kw.get("summ", FAKE), FAKE, FAKE, FAKE, FAKE, kw.get("sel", FAKE), FAKE, None,
        ws, n, None)
    assert st(p, 4096, FAKE, need) == ssa.SSA_ERR_INVALID_ARG         # pos == L
    assert st(p, 10, FAKE, need, summ=None) == ssa.SSA_ERR_INVALID_ARG
    assert st(p, 10, FAKE, need, sel=None) == ssa.SSA_ERR_INVALID_ARG
    assert st(p, 10, None, 0) == ssa.SSA_ERR_WORKSPACE
    assert st(p, 10, FAKE, need - 1) == ssa.SSA_ERR_WORKSPACE
    assert st(ssa.params(1, 8, 2, 64, 4096, 64, 8, torch.bfloat16), 10, FAKE, need) == ssa.SSA_ERR_UNSUPPORTED
    assert st(ssa.params(1, 8, 2, 128, 4001, 64, 8, torch.bfloat16), 10, FAKE, need) == ssa.SSA_ERR_UNSUPPORTED


@needs_no_gpu
def test_q4_validation():
    L = ssa.lib()
    P, I8, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    pp = ctypes.POINTER(ssa.ssa_params)
    L.ssa_quantize_kv4.argtypes = [pp, P, P, I8, I8, P, P, P, P, P]
    L.ssa_build_summaries_q4.argtypes = [pp, P, P, I8, I8, P, P]
    L.ssa_attend_decode_q4.argtypes = [pp, P, I8, P, P, P, P, P, P, P, P, SZ, P]
    L.ssa_decode_step_q4.argtypes = [pp, P, I8, P, P, P, P, P, P, P, P, P, SZ, P]
    p = ssa.params(1, 8, 2, 128, 4096, 64, 8, torch.bfloat16)
    p_d64 = ssa.params(1, 8, 2, 64, 4096, 64, 8, torch.bfloat16)
    p_ragged = ssa.params(1, 8, 2, 128, 4001, 64, 8, torch.bfloat16)
    q = lambda p, t0, t1, **kw: L.ssa_quantize_kv4(ctypes.byref(p), FAKE, kw.get("V", FAKE), t0, t1, FAKE, FAKE,
                                                   FAKE, FAKE, None)
    assert q(p, 0, 4097) == ssa.SSA_ERR_INVALID_ARG             # past L
    assert q(p, 10, 5) == ssa.SSA_ERR_INVALID_ARG
    assert q(p, -1, 5) == ssa.SSA_ERR_INVALID_ARG
    assert q(p, 0, 10, V=None) == ssa.SSA_ERR_INVALID_ARG
    assert q(p, 0, 10, V=ctypes.c_void_p(4104)) == ssa.SSA_ERR_INVALID_ARG   # not 16-byte aligned
    assert q(p_ragged, 0, 10) == ssa.SSA_ERR_UNSUPPORTED        # L_cap % 32
    assert q(p_d64, 0, 10) == ssa.SSA_ERR_UNSUPPORTED
    s = lambda p, j0, j1: L.ssa_build_summaries_q4(ctypes.byref(p), FAKE, FAKE, j0, j1, FAKE, None)
    assert s(p, 0, 65) == ssa.SSA_ERR_INVALID_ARG               # past the last span
    assert s(p, 3, 2) == ssa.SSA_ERR_INVALID_ARG
    assert s(p_d64, 0, 1) == ssa.SSA_ERR_UNSUPPORTED
    need = ssa.ssa_workspace_size(p, 1, ssa.SSA_OP_DECODE)
    d = lambda p, pos, ws, n: L.ssa_attend_decode_q4(ctypes.byref(p), FAKE, pos, FAKE, FAKE, FAKE, FAKE, FAKE,
                                                     FAKE, None, ws, n, None)
    assert d(p, 4096, FAKE, need) == ssa.SSA_ERR_INVALID_ARG          # pos == L
    assert d(p, 10, None, 0) == ssa.SSA_ERR_WORKSPACE
    assert d(p, 10, FAKE, need - 1) == ssa.SSA_ERR_WORKSPACE
    assert d(p_d64, 10, FAKE, need) == ssa.SSA_ERR_UNSUPPORTED
    assert d(p_ragged, 10, FAKE, need) == ssa.SSA_ERR_UNSUPPORTED
    assert d(ssa.params(1, 8, 2, 128, 4096, 64, 8, torch.float32), 10, FAKE, need) == ssa.SSA_ERR_UNSUPPORTED
    st = lambda p, pos, ws, n, **kw: L.ssa_decode_step_q4(
        ctypes.byref(p), FAKE, pos, kw.get("summ", FAKE), FAKE, FAKE, FAKE, FAKE, kw.get("sel", FAKE), FAKE, None,
        ws, n, None)
    assert st(p, 4096, FAKE, need) == ssa.SSA_ERR_INVALID_ARG
    assert st(p, 10, FAKE, need, summ=None) == ssa.SSA_ERR_INVALID_ARG
    assert st(p, 10, FAKE, need, sel=None) == ssa.SSA_ERR_INVALID_ARG
    assert st(p, 10, None, 0) == ssa.SSA_ERR_WORKSPACE
    assert st(p_d64, 10, FAKE, need) == ssa.SSA_ERR_UNSUPPORTED


@needs_no_gpu
def test_decode_step_group_validation():
    p = ssa.params(1, 8, 2, 128, 4096, 64, 8, torch.bfloat16)
    L = ssa.lib()
    L.ssa_decode_step_group.argtypes = [ctypes.POINTER(ssa.ssa_params), ctypes.c_void_p, ctypes.c_int64] + \
        [ctypes.c_void_p] * 7 + [ctypes.c_size_t, ctypes.c_void_p]
    need = ssa.ssa_workspace_size(p, 1, ssa.SSA_OP_DECODE)
    step = lambda p, pos, ws, n, **kw: L.ssa_decode_step_group(
        ctypes.byref(p), kw.get("Q", FAKE), pos, kw.get("summ", FAKE), FAKE, FAKE, kw.get("sel", FAKE), FAKE,
        None, ws, n, None)
    assert step(p, 4096, FAKE, need) == ssa.SSA_ERR_INVALID_ARG        # pos == L
    assert step(p, -1, FAKE, need) == ssa.SSA_ERR_INVALID_ARG
    assert step(p, 10, FAKE, need, summ=None) == ssa.SSA_ERR_INVALID_ARG
    assert step(p, 10, FAKE, need, sel=None) == ssa.SSA_ERR_INVALID_ARG
    assert step(p, 10, FAKE, need, Q=ctypes.c_void_p(4098)) == ssa.SSA_ERR_INVALID_ARG
    assert step(p, 10, None, 0) == ssa.SSA_ERR_WORKSPACE
    assert step(p, 10, FAKE, need - 1) == ssa.SSA_ERR_WORKSPACE
    # only the fast decode path: fp32 and d = 96 are refused
    assert step(ssa.params(1, 8, 2, 128, 4096, 64, 8, torch.float32), 10, FAKE, need) == ssa.SSA_ERR_UNSUPPORTED
    assert step(ssa.params(1, 8, 2, 96, 4096, 64, 8, 1), 10, FAKE, need) == ssa.SSA_ERR_UNSUPPORTED


@needs_no_gpu
def test_decode_step_validation():
    p = ssa.params(1, 8, 2, 128, 4096, 64, 8, torch.bfloat16)
    L = ssa.lib()
    need = ssa.ssa_workspace_size(p, 1, ssa.SSA_OP_DECODE)
    step = lambda p, pos, ws, n, **kw: L.ssa_decode_step(
        ctypes.byref(p), kw.get("Q", FAKE), pos, kw.get("summ", FAKE), FAKE, FAKE, kw.get("sel", FAKE), FAKE,
        None, ws, n, None)
    assert step(p, 4096, FAKE, need) == ssa.SSA_ERR_INVALID_ARG        # pos == L
    assert step(p, -1, FAKE, need) == ssa.SSA_ERR_INVALID_ARG
    assert step(p, 10, FAKE, need, summ=None) == ssa.SSA_ERR_INVALID_ARG
    assert step(p, 10, FAKE, need, sel=None) == ssa.SSA_ERR_INVALID_ARG
    assert step(p, 10, FAKE, need, Q=ctypes.c_void_p(4098)) == ssa.SSA_ERR_INVALID_ARG
    assert step(p, 10, None, 0) == ssa.SSA_ERR_WORKSPACE
    assert step(p, 10, FAKE, need - 1) == ssa.SSA_ERR_WORKSPACE
    assert step(ssa.params(1, 8, 2, 96, 4096, 64, 8, 1), 10, FAKE, need) == ssa.SSA_ERR_UNSUPPORTED


def test_attend_path_reports_the_implementation():
    """The fast paths and the row kernel are chosen by the parameters alone;
    the query says which one a call takes."""
    P = lambda **kw: ssa.params(kw.get("B", 1), kw.get("Hq", 32), kw.get("Hkv", 4), kw.get("d", 128), 1 << 20, 1024,
                                16, kw.get("dt", torch.bfloat16))
    assert ssa.ssa_attend_path(P(), 1, ssa.SSA_OP_DECODE) == ssa.SSA_PATH_FAST
    assert ssa.ssa_attend_path(P(), 8192, ssa.SSA_OP_PREFILL) == ssa.SSA_PATH_FAST
    assert ssa.ssa_attend_path(P(dt=torch.float16, d=64), 8192, ssa.SSA_OP_PREFILL) == ssa.SSA_PATH_FAST
    # fp32 takes the row kernel in both
    assert ssa.ssa_attend_path(P(dt=torch.float32), 1, ssa.SSA_OP_DECODE) == ssa.SSA_PATH_ROWS
    assert ssa.ssa_attend_path(P(dt=torch.float32), 4096, ssa.SSA_OP_PREFILL) == ssa.SSA_PATH_ROWS
    # 128 / g not whole: prefill tiles of 128 rows cannot hold whole queries
    assert ssa.ssa_attend_path(P(Hq=12, Hkv=1), 100, ssa.SSA_OP_PREFILL) == ssa.SSA_PATH_ROWS
    # row ids past the 32-bit bucket entries
    assert ssa.ssa_attend_path(P(B=4, Hq=32), 1 << 18, ssa.SSA_OP_PREFILL) == ssa.SSA_PATH_ROWS
    # invalid parameters, other ops
    assert ssa.ssa_attend_path(P(d=96), 1, ssa.SSA_OP_DECODE) == ssa.SSA_PATH_INVALID
    assert ssa.ssa_attend_path(P(), 1, ssa.SSA_OP_ROUTE) == ssa.SSA_PATH_INVALID


@needs_no_gpu
def test_selftest_wait_validation():
    L = ssa.lib()
    L.ssa_selftest_wait_timeout.argtypes = [ctypes.c_uint64, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    assert L.ssa_selftest_wait_timeout(2_000_000_000, FAKE, 256, None) == ssa.SSA_ERR_INVALID_ARG  # above 1 s
    assert L.ssa_selftest_wait_timeout(1000, None, 0, None) == ssa.SSA_ERR_WORKSPACE
    assert L.ssa_selftest_wait_timeout(1000, FAKE, 255, None) == ssa.SSA_ERR_WORKSPACE
