"""Oracle runs on caches too large to hold on the host (the 10M-token decode).

TEST INFRASTRUCTURE, like the rest of this package: only the tests, the
package's smoke check and the benchmark's CPU legs use it.

Two helpers, both built on the oracle's own functions and on rows that the
seeded input generator regenerates on the host for any range:

* ``summaries_streamed``: the oracle's span means of a whole cache, computed
  from host regenerations of span ranges, so the 20 GB cache is never held.
* ``compact_decode_step``: one decode step's attention as a smaller problem
  (rows regenerated on the host, or read by a caller-given function).
  For one kv-head it holds only the union of its query heads' selected spans
  (ascending) followed by the causal part of the local span.  Attention over
  a token set does not depend on where the tokens sit, so the compacted
  problem has the same answer (the shift and permutation pins of the oracle
  tests check that property of the oracle).

``inp`` is the generator's ``Inputs`` object; only its workload (``inp.w``)
and its host row regenerator (``inp.kv_rows``) are used.
"""
from __future__ import annotations

import numpy as np
import torch

from . import summaries


def summaries_streamed(inp, spans_per_part: int = 128) -> np.ndarray:
    """Oracle summaries [B, Hkv, n_spans, d] of the whole cache of inp.w."""
    w = inp.w
    ns = w.n_spans
    out = np.zeros((w.B, w.Hkv, ns, w.d), np.float64)
    for bh in range(w.B * w.Hkv):
        b, h = divmod(bh, w.Hkv)
        for j0 in range(0, ns, spans_per_part):
            j1 = min(ns, j0 + spans_per_part)
            t0, t1 = j0 * w.S, min(w.L, j1 * w.S)
            Kc = inp.kv_rows("k", bh, t0, t1).reshape(1, 1, t1 - t0, w.d)
            out[b, h, j0:j1] = summaries(Kc, t1 - t0, w.S)[0, 0]
    return out


def _regenerate(inp, which: str, bh: int, parts) -> torch.Tensor:
    return torch.cat([inp.kv_rows(which, bh, a, e) for a, e in parts])


def compact_decode_step(inp, q_step: torch.Tensor, sel_step: np.ndarray, t: int, fetch=None):
    """The decode step at position t as one compacted problem per (b, kv-head).

    q_step [B, Hq, d] (host), sel_step [B*Hq, k] (the step's selections).
    Yields (rows, q [1, g, 1, d], K [1, 1, n, d], V [1, 1, n, d], pos, sel)
    where rows are the step's row indices (b * Hq + head) of the kv-head's
    query heads and (q, K, V, pos, sel) are the arguments of oracle.attend
    for the compacted cache.

    ``fetch(which, bh, parts)`` returns the host rows of the half-open row
    ranges ``parts`` of K or V ("k" / "v") of flattened kv-head bh, one range
    after the other.  By default the rows are regenerated on the host; a
    caller that holds the same generated cache elsewhere may read it there.
    """
    if fetch is None:
        def fetch(which, bh, parts):
            return _regenerate(inp, which, bh, parts)
    w = inp.w
    ell = t // w.S
    for bh in range(w.B * w.Hkv):
        b, h = divmod(bh, w.Hkv)
        rows = [b * w.Hq + hq for hq in range(h * w.g, (h + 1) * w.g)]
        sel_h = sel_step[rows]
        union = np.unique(sel_h[sel_h >= 0])
        parts = [(int(j) * w.S, (int(j) + 1) * w.S) for j in union] + [(ell * w.S, t + 1)]
        Kc = fetch("k", bh, parts).reshape(1, 1, -1, w.d)
        Vc = fetch("v", bh, parts).reshape(1, 1, -1, w.d)
        remap = {int(j): i for i, j in enumerate(union)}
        sel_c = np.full(sel_h.shape, -1, np.int32)
        for r in range(sel_h.shape[0]):
            for c in range(sel_h.shape[1]):
                if sel_h[r, c] >= 0:
                    sel_c[r, c] = remap[int(sel_h[r, c])]
        qc = q_step[b, h * w.g:(h + 1) * w.g].reshape(1, w.g, 1, w.d).contiguous()
        yield rows, qc, Kc, Vc, len(union) * w.S + (t - ell * w.S), sel_c
