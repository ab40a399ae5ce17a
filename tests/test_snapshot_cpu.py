"""Cache snapshots on the CPU: the oracle's file format pinned to literal
bytes, the library's header reader against oracle-written files, and the
argument checks the save / load entry points make before touching the GPU
or the file system's contents.

Superlinear release post (geeks.co.kr/post/2077), "why this matters": the
cache is kept, in memory and on disk per session, instead of re-processing
the context."""
import ctypes
import struct

import numpy as np
import pytest
import torch

import content_routed_sparse_build_b300 as ssa
from oracle import snapshot as osnap

# ---------------------------------------------------------------- oracle pins


def test_oracle_snapshot_bytes_of_a_tiny_cache_are_the_literal_layout():
    # B1 Hkv1 d2 S2, three fp16 rows: one complete span
    K = np.array([[[[0x3C00, 0x4000], [0x4200, 0x4400], [0x4500, 0x4600]]]], np.uint16)   # 1 2 3 4 5 6
    V = np.array([[[[0xBC00, 0x0000], [0x0001, 0x7BFF], [0x8000, 0x3800]]]], np.uint16)
    summ = np.array([[[[2.0, 3.0]]]], np.float32)          # mean of rows 0 and 1 of K
    got = osnap.encode(2, 2, K, V, summ)
    want = bytes.fromhex(
        "53 53 41 4b 56 53 4e 31"        # "SSAKVSN1"
        "01 00 00 00" "02 00 00 00"       # version 1, dtype fp16
        "01 00 00 00" "01 00 00 00" "02 00 00 00" "02 00 00 00"   # B Hkv d S
        "03 00 00 00 00 00 00 00"         # n_tokens 3
        "01 00 00 00 00 00 00 00"         # n_summ 1
        "20 00 00 00 00 00 00 00"         # payload 12 + 12 + 8 = 32 bytes
        "00 00 00 00 00 00 00 00"         # reserved
        "00 3c 00 40 00 42 00 44 00 45 00 46"
        "00 bc 00 00 01 00 ff 7b 00 80 00 38"
        "00 00 00 40 00 00 40 40")        # 2.0f 3.0f
    assert got == want
    back = osnap.decode(got)
    assert back["n_tokens"] == 3 and back["n_summ"] == 1 and back["S"] == 2
    assert np.array_equal(back["K"], K) and np.array_equal(back["V"], V)
    assert np.array_equal(back["summ"], summ)


def test_oracle_snapshot_rejects_malformed_bytes():
    K = np.zeros((1, 2, 5, 4), np.uint16)
    good = osnap.encode(1, 2, K, K, np.zeros((1, 2, 2, 4), np.float32))
    osnap.decode(good)
    for bad in (good[:-1], good + b"\0", b"X" + good[1:], good[:56] + b"\1" + good[57:]):
        with pytest.raises(ValueError):
            osnap.decode(bad)


# ---------------------------------------------------------------- header reader


def _write(tmp_path, name, data):
    p = tmp_path / name
    p.write_bytes(data)
    return str(p)


def test_library_reads_oracle_written_headers(tmp_path):
    rng = np.random.default_rng(5)
    for dt, word, es in ((0, np.uint32, 4), (1, np.uint16, 2), (2, np.uint16, 2)):
        K = rng.integers(0, 1 << 16, size=(2, 3, 7, 64)).astype(word)
        V = rng.integers(0, 1 << 16, size=(2, 3, 7, 64)).astype(word)
        summ = rng.standard_normal((2, 3, 2, 64)).astype(np.float32)
        path = _write(tmp_path, "s%d.bin" % dt, osnap.encode(dt, 3, K, V, summ))
        h = ssa.ssa_snapshot_read_header(path)
        assert bytes(h.magic) == ssa.SSA_SNAPSHOT_MAGIC and h.version == ssa.SSA_SNAPSHOT_VERSION
        assert (h.dtype, h.B, h.Hkv, h.d, h.S, h.n_tokens, h.n_summ) == (dt, 2, 3, 64, 3, 7, 2)
        assert h.payload_bytes == 2 * 3 * (2 * 7 * 64 * es + 2 * 64 * 4)


def test_library_header_reader_rejects_what_the_oracle_rejects(tmp_path):
    K = np.zeros((1, 1, 4, 64), np.uint16)
    good = osnap.encode(1, 2, K, K, np.zeros((1, 1, 2, 64), np.float32))
    cases = {
        "truncated": good[:-2],
        "long": good + b"\0\0",
        "magic": b"SSAKVSN2" + good[8:],
        "version": good[:8] + struct.pack("<I", 2) + good[12:],
        "dtype": good[:12] + struct.pack("<i", 7) + good[16:],
        "n_summ": good[:40] + struct.pack("<q", 1) + good[48:],
        "reserved": good[:60] + b"\1" + good[61:],
        "short": good[:40],
    }
    for name, data in cases.items():
        with pytest.raises(ValueError):
            osnap.decode(data)
        with pytest.raises(ssa.SSAError) as e:
            ssa.ssa_snapshot_read_header(_write(tmp_path, name, data))
        assert e.value.status == ssa.SSA_ERR_IO, name
    with pytest.raises(ssa.SSAError) as e:
        ssa.ssa_snapshot_read_header(str(tmp_path / "missing.bin"))
    assert e.value.status == ssa.SSA_ERR_IO


# ---------------------------------------------------------------- argument checks (no GPU call)


class _Fake:
    """Stands in for a device tensor: only its address is passed."""

    def __init__(self, addr=1 << 20):
        self.addr = addr

    def data_ptr(self):
        return self.addr


def test_save_and_load_check_arguments_before_any_device_work(tmp_path):
    p = ssa.params(1, 8, 2, 64, 1000, 64, 4, torch.bfloat16, L_cap=1024)
    f = _Fake()
    small = torch.empty(2 * 64 * 4 - 1, dtype=torch.uint8)
    ok = torch.empty(1 << 12, dtype=torch.uint8)
    path = str(tmp_path / "x.bin")
    for kw in ({"n_tokens": 1001}, {"n_tokens": -1}):
        with pytest.raises(ssa.SSAError) as e:
            ssa.ssa_snapshot_save(p, kw["n_tokens"], f, f, f, path, staging=ok, stream=0)
        assert e.value.status == ssa.SSA_ERR_INVALID_ARG
    with pytest.raises(ssa.SSAError) as e:
        ssa.ssa_snapshot_save(p, 10, f, f, f, path, staging=small, stream=0)
    assert e.value.status == ssa.SSA_ERR_INVALID_ARG
    with pytest.raises(ssa.SSAError) as e:
        ssa.ssa_snapshot_save(p, 10, f, None, f, path, staging=ok, stream=0)
    assert e.value.status == ssa.SSA_ERR_INVALID_ARG
    bad = ssa.params(1, 8, 3, 64, 1000, 64, 4, torch.bfloat16)       # Hq not a multiple of Hkv
    with pytest.raises(ssa.SSAError) as e:
        ssa.ssa_snapshot_save(bad, 10, f, f, f, path, staging=ok, stream=0)
    assert e.value.status == ssa.SSA_ERR_INVALID_ARG
    assert not (tmp_path / "x.bin").exists()
    # load: a missing file, and files that do not match the parameters
    with pytest.raises(ssa.SSAError) as e:
        ssa.ssa_snapshot_load(p, str(tmp_path / "missing.bin"), f, f, f, staging=ok, stream=0)
    assert e.value.status == ssa.SSA_ERR_IO
    K = np.zeros((1, 2, 40, 64), np.uint16)
    summ = np.zeros((1, 2, 0, 64), np.float32)
    mism = {
        "S": osnap.encode(1, 41, K, K, summ),                                   # S 41, not 64
        "dtype": osnap.encode(2, 64, K, K, summ),                               # fp16, not bf16
        "heads": osnap.encode(1, 64, K[:, :1], K[:, :1], summ[:, :1]),           # Hkv 1
        "d": osnap.encode(1, 64, K[..., :32], K[..., :32], summ[..., :32]),      # d 32
        "cap": osnap.encode(1, 64, np.zeros((1, 2, 1025, 64), np.uint16), np.zeros((1, 2, 1025, 64), np.uint16),
                            np.zeros((1, 2, 16, 64), np.float32)),              # 1025 rows > L_cap
    }
    for name, data in mism.items():
        with pytest.raises(ssa.SSAError) as e:
            ssa.ssa_snapshot_load(p, _write(tmp_path, name + ".bin", data), f, f, f, staging=ok, stream=0)
        assert e.value.status == ssa.SSA_ERR_IO, name


def test_snapshot_symbols_and_status_text():
    L = ssa.lib()
    for name in ("ssa_snapshot_save", "ssa_snapshot_load", "ssa_snapshot_read_header"):
        assert hasattr(L, name)
    assert "snapshot" in ssa.ssa_status_string(ssa.SSA_ERR_IO)
    assert ctypes.sizeof(ssa.ssa_snapshot_header) == 64
