"""Oracle of the cache-snapshot file: a plain writer and reader of the format.

TEST INFRASTRUCTURE, like the rest of ``oracle/``: only ``tests/`` may use it.
It shares no code with the library.

What it restates: the superlinear release post (geeks.co.kr/post/2077),
"why this matters", keeps the cache instead of re-processing the context
and saves / restores a session on disk.  The byte layout is the one the
library's public header defines for ssa_snapshot_header and the payload
after it; this module writes it field by field with ``struct`` and numpy,
so a test can compare the library's file with this one byte for byte.

Layout (little-endian): magic "SSAKVSN1", u32 version 1, i32 dtype code,
i32 B, Hkv, d, S, i64 n_tokens, i64 n_summ = n_tokens // S, u64 payload
bytes, 8 zero bytes; then K rows [B][Hkv][n_tokens][d], V rows likewise
(raw element bytes), then the fp32 summaries [B][Hkv][n_summ][d].
"""
from __future__ import annotations

import struct

import numpy as np

MAGIC = b"SSAKVSN1"
VERSION = 1
_HDR = struct.Struct("<8sIiiiiiqqQ8s")
assert _HDR.size == 64
_ES = {0: 4, 1: 2, 2: 2}   # element bytes per dtype code (fp32, bf16, fp16)


def encode(dtype_code: int, S: int, K_rows: np.ndarray, V_rows: np.ndarray, summ_rows: np.ndarray) -> bytes:
    """File bytes of a snapshot.  K_rows / V_rows: [B, Hkv, n_tokens, d] as
    raw element words (uint16 for 16-bit types, uint32 / float32 for fp32);
    summ_rows: float32 [B, Hkv, n_tokens // S, d]."""
    B, Hkv, n_tokens, d = K_rows.shape
    n_summ = n_tokens // S
    assert V_rows.shape == K_rows.shape
    assert summ_rows.shape == (B, Hkv, n_summ, d) and summ_rows.dtype == np.float32
    es = _ES[dtype_code]
    assert K_rows.dtype.itemsize == es and V_rows.dtype.itemsize == es
    body = (np.ascontiguousarray(K_rows).astype(K_rows.dtype.newbyteorder("<")).tobytes()
            + np.ascontiguousarray(V_rows).astype(V_rows.dtype.newbyteorder("<")).tobytes()
            + np.ascontiguousarray(summ_rows).astype("<f4").tobytes())
    want = B * Hkv * (2 * n_tokens * d * es + n_summ * d * 4)
    assert len(body) == want
    head = _HDR.pack(MAGIC, VERSION, dtype_code, B, Hkv, d, S, n_tokens, n_summ, len(body), bytes(8))
    return head + body


def decode(data: bytes) -> dict:
    """Fields and arrays of a snapshot's bytes (raises ValueError when the
    bytes are not a well-formed snapshot)."""
    if len(data) < 64:
        raise ValueError("shorter than the header")
    magic, ver, dt, B, Hkv, d, S, n_tokens, n_summ, payload, res = _HDR.unpack_from(data, 0)
    if magic != MAGIC or ver != VERSION or res != bytes(8) or dt not in _ES:
        raise ValueError("not a snapshot header")
    if n_summ != n_tokens // S or len(data) != 64 + payload:
        raise ValueError("sizes disagree")
    es = _ES[dt]
    kv = B * Hkv * n_tokens * d
    word = np.dtype("<u2") if es == 2 else np.dtype("<u4")
    off = 64
    K = np.frombuffer(data, word, kv, off).reshape(B, Hkv, n_tokens, d)
    off += kv * es
    V = np.frombuffer(data, word, kv, off).reshape(B, Hkv, n_tokens, d)
    off += kv * es
    summ = np.frombuffer(data, "<f4", B * Hkv * n_summ * d, off).reshape(B, Hkv, n_summ, d)
    off += B * Hkv * n_summ * d * 4
    if off != len(data):
        raise ValueError("payload size disagrees")
    return {"dtype": dt, "B": B, "Hkv": Hkv, "d": d, "S": S, "n_tokens": n_tokens, "n_summ": n_summ,
            "K": K, "V": V, "summ": summ}
