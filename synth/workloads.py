"""The synthetic workloads of content-routed sparse attention.

Each workload fixes the shapes, the storage type, the seed and the structure
added to the keys.  The five full-size workloads follow the sizes the
superlinear release post and the SubQ pages talk about (1M and 10M token
contexts, chunked prefill at 128K and against a 1M cache); ``tiny_*`` and
``case_*`` are small cases with the same structure.

Layouts (all row-major, contiguous):
  K, V      [B, Hkv, L, d]  -- the persistent cache, L rows per head
  Q prefill [B, Hq, n_q, d] -- query i sits at position q_pos0 + i
  Q decode  [steps, B, Hq, d] -- step s sits at position q_pos0 + s

Structure (input construction only, float64 on the host):
  * needles: per (b, kv-head) a seeded set of complete candidate spans whose
    every key gets +2*u, u = the normalised sum of the run's query rows of
    that kv-head's query heads (first draw, before any row is redrawn);
  * low rank: key row t of kv-head h gets W_h z_{t // S}, W_h a d x r matrix
    with N(0, 1/r) entries and z_j an r-vector with N(0, 1) entries that is
    constant over span j, so span means (not only single keys) differ.
The added term is one fp32 table [B*Hkv, ceil(L/S), d]; see synth_core.h for
how it enters each element.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass

import numpy as np
import torch

from . import (TID_K, TID_LOWRANK_W, TID_LOWRANK_Z, TID_NEEDLE, TID_Q, TID_V, f64_values,
               fill_, round_f32)


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str            # "prefill" or "decode"
    B: int
    Hq: int
    Hkv: int
    d: int
    L: int               # cache rows per head (valid length once every chunk is in)
    S: int               # span length
    topk: int
    dtype: torch.dtype
    n_q: int             # prefill: queries; decode: steps
    q_pos0: int          # position of the first query / step
    chunk: int           # prefill chunk (queries per attend call)
    needles: int = 0     # planted needle spans per (b, kv-head)
    lowrank: int = 0     # rank of the per-span term in K
    seed: int = 1

    @property
    def g(self) -> int:
        return self.Hq // self.Hkv

    @property
    def n_spans(self) -> int:
        return (self.L + self.S - 1) // self.S

    @property
    def q_shape(self):
        if self.kind == "decode":
            return (self.n_q, self.B, self.Hq, self.d)
        return (self.B, self.Hq, self.n_q, self.d)

    @property
    def kv_shape(self):
        return (self.B, self.Hkv, self.L, self.d)

    @property
    def last_pos(self) -> int:
        return self.q_pos0 + self.n_q - 1

    def positions(self) -> np.ndarray:
        return self.q_pos0 + np.arange(self.n_q, dtype=np.int64)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


F32, BF16, F16 = torch.float32, torch.bfloat16, torch.float16

# The five full-size workloads.
TINY_PREFILL = Workload("tiny_prefill_4k_f32", "prefill", 1, 4, 4, 64, 4096, 64, 8, F32,
                        n_q=4096, q_pos0=0, chunk=4096, needles=2, seed=1001)
DECODE_1M = Workload("decode_1m", "decode", 1, 32, 4, 128, 1 << 20, 1024, 16, BF16,
                     n_q=256, q_pos0=(1 << 20) - 256, chunk=1, needles=8, seed=1002)
PREFILL_128K = Workload("prefill_128k", "prefill", 1, 32, 8, 128, 131072, 256, 16, BF16,
                        n_q=131072, q_pos0=0, chunk=8192, lowrank=8, seed=1003)
PREFILL_1M = Workload("prefill_chunk_vs_1m", "prefill", 1, 32, 4, 128, 1 << 20, 1024, 16, BF16,
                      n_q=8192, q_pos0=(1 << 20) - 8192, chunk=8192, needles=16, seed=1004)
DECODE_10M = Workload("decode_10m", "decode", 1, 32, 4, 128, 10_000_000, 3072, 16, BF16,
                      n_q=128, q_pos0=10_000_000 - 128, chunk=1, needles=32, seed=1005)

FULL = {w.name: w for w in (TINY_PREFILL, DECODE_1M, PREFILL_128K, PREFILL_1M, DECODE_10M)}


class Inputs:
    """Lazily generated inputs of one workload.

    ``attempt`` (int32, one per query row of the full Q) redraws rows; it is
    supplied by whoever checks score margins.  Needle directions always come
    from the first draw.
    """

    def __init__(self, w: Workload, attempt: torch.Tensor | None = None):
        self.w = w
        self.attempt = attempt
        self.needle_spans = None   # int64 [B*Hkv, needles]
        self.u = None              # float64 [B*Hkv, d]
        self.bias = None           # float32 [B*Hkv, n_spans, d] (host) or None
        self._bias_dev = {}
        self._build_structure()

    # ---- structure -------------------------------------------------------
    def _build_structure(self) -> None:
        w = self.w
        nb = w.n_spans
        bias = None
        if w.needles > 0:
            q0 = self.q("cpu", first_draw=True).to(torch.float64).numpy()
            if w.kind == "decode":
                q0 = q0.transpose(1, 2, 0, 3)            # [B, Hq, steps, d]
            q0 = q0.reshape(w.B, w.Hkv, w.g * w.n_q, w.d)
            s = q0.sum(axis=2)
            u = s / np.linalg.norm(s, axis=-1, keepdims=True)
            self.u = u.reshape(w.B * w.Hkv, w.d)
            n_cand = w.last_pos // w.S                   # complete spans before the last query's span
            if w.needles > n_cand:
                raise ValueError("more needles than candidate spans")
            keys = f64_values(w.B * w.Hkv * n_cand, w.seed, TID_NEEDLE).reshape(w.B * w.Hkv, n_cand)
            self.needle_spans = np.sort(np.argsort(keys, axis=1, kind="stable")[:, : w.needles], axis=1)
            bias = np.zeros((w.B * w.Hkv, nb, w.d), np.float64)
            for bh in range(w.B * w.Hkv):
                bias[bh, self.needle_spans[bh], :] += 2.0 * self.u[bh]
        if w.lowrank > 0:
            r = w.lowrank
            W = f64_values(w.Hkv * w.d * r, w.seed, TID_LOWRANK_W).reshape(w.Hkv, w.d, r) / math.sqrt(r)
            z = f64_values(nb * r, w.seed, TID_LOWRANK_Z).reshape(nb, r)
            lr = np.einsum("hcr,jr->hjc", W, z)          # [Hkv, nb, d]
            lr = np.broadcast_to(lr[None], (w.B, w.Hkv, nb, w.d)).reshape(w.B * w.Hkv, nb, w.d)
            bias = lr if bias is None else bias + lr
        if bias is not None:
            self.bias = torch.from_numpy(np.ascontiguousarray(bias.astype(np.float32)))

    def bias_on(self, device) -> torch.Tensor | None:
        if self.bias is None:
            return None
        dev = torch.device(device)
        if dev.type == "cpu":
            return self.bias
        key = str(dev)
        if key not in self._bias_dev:
            self._bias_dev[key] = self.bias.to(dev)
        return self._bias_dev[key]

    # ---- tensors ---------------------------------------------------------
    def q(self, device="cpu", first_draw: bool = False, out: torch.Tensor | None = None) -> torch.Tensor:
        w = self.w
        if out is None:
            out = torch.empty(w.q_shape, dtype=w.dtype, device=device)
        att = None
        if self.attempt is not None and not first_draw:
            att = self.attempt.to(out.device)
        return fill_(out, w.seed, TID_Q, d=w.d, attempt=att)

    def q_rows(self, rows: np.ndarray) -> torch.Tensor:
        """Host copy of selected query rows (global row indices of the full Q)."""
        w = self.w
        rows = np.asarray(rows, dtype=np.int64)
        out = torch.empty((len(rows), w.d), dtype=w.dtype)
        # The attempt array is indexed by global row, so the full array serves
        # any sub-range fill.
        for i, r in enumerate(rows):
            fill_(out[i: i + 1], w.seed, TID_Q, e0=int(r) * w.d, d=w.d, attempt=self.attempt)
        return out

    def k(self, device="cpu", out: torch.Tensor | None = None) -> torch.Tensor:
        return self._kv(TID_K, device, out, with_bias=True)

    def v(self, device="cpu", out: torch.Tensor | None = None) -> torch.Tensor:
        return self._kv(TID_V, device, out, with_bias=False)

    def _kv(self, tid, device, out, with_bias):
        w = self.w
        if out is None:
            out = torch.empty(w.kv_shape, dtype=w.dtype, device=device)
        bias = self.bias_on(out.device) if with_bias else None
        return fill_(out, w.seed, tid, d=w.d, bias=bias, rows_per_head=w.L, S=w.S)

    def kv_rows(self, which: str, bh: int, t0: int, t1: int) -> torch.Tensor:
        """Host rows [t0, t1) of K or V for flattened (b, kv-head) index bh."""
        w = self.w
        out = torch.empty((t1 - t0, w.d), dtype=w.dtype)
        tid = TID_K if which == "k" else TID_V
        bias = self.bias if which == "k" else None
        e0 = (bh * w.L + t0) * w.d
        return fill_(out, w.seed, tid, e0=e0, d=w.d, bias=bias, rows_per_head=w.L, S=w.S)

    def probe_q(self) -> torch.Tensor:
        """Probe queries [B, Hq, d]: every head of kv-head group h gets sqrt(d) * u_h."""
        w = self.w
        if self.u is None:
            raise ValueError("workload has no needles")
        u = self.u.reshape(w.B, w.Hkv, 1, w.d)
        p = np.broadcast_to(math.sqrt(w.d) * u, (w.B, w.Hkv, w.g, w.d)).reshape(w.B, w.Hq, w.d)
        p32 = np.ascontiguousarray(p.astype(np.float32))
        if w.dtype == torch.float32:
            return torch.from_numpy(p32)
        bits = round_f32(p32, w.dtype)
        return torch.from_numpy(bits.view(np.int16)).view(w.dtype)
