"""Shared helpers of the parity tests: margin-checked inputs, the CUDA path
through the C ABI, and the oracle on the same inputs.

Selections are compared bit for bit.  The generator's query rows whose
k-th / (k+1)-th oracle score margin is below MARGIN are redrawn (attempt
counter) before any comparison, so that an fp32 score can never reorder two
spans the double-precision oracle separates.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import content_routed_sparse_build_b300 as ssa
import oracle
from synth import workloads as W

MARGIN = 1e-3
TOL = {torch.float32: 1e-5, torch.bfloat16: 2e-2, torch.float16: 2e-2}
LSE_TOL = {torch.float32: 1e-5, torch.bfloat16: 1e-3, torch.float16: 1e-3}

# What the margin check found, one entry per checked case: printed at the end
# of the run by conftest.py (and written as JSON where SSA_MARGIN_REPORT
# names a file).
MARGIN_REPORT: list[dict] = []


def report_margins(case: str, margin, redrawn: int) -> None:
    """Records a case's oracle margins (k-th minus (k+1)-th score of each
    checked row; +inf for rows with no more candidates than k) and how many
    query rows the generator redrew to reach MARGIN."""
    m = np.asarray(margin, dtype=np.float64).reshape(-1)
    ranked = m[np.isfinite(m)]
    MARGIN_REPORT.append({"case": case, "rows": int(m.size), "ranked_rows": int(ranked.size),
                          "redrawn": int(redrawn),
                          "min_margin": float(ranked.min()) if ranked.size else None})


def params_of(w: W.Workload, L: int | None = None, topk: int | None = None) -> ssa.ssa_params:
    return ssa.params(w.B, w.Hq, w.Hkv, w.d, w.L if L is None else L, w.S,
                      w.topk if topk is None else topk, w.dtype, L_cap=w.L)


# ------------------------------------------------------------------ oracle side
class OracleRun:
    """Oracle summaries / selections / outputs of a workload (host)."""

    def __init__(self, w: W.Workload, inp: W.Inputs, K: torch.Tensor | None = None):
        self.w = w
        self.inp = inp
        self.K = K if K is not None else inp.k()
        self.summ = oracle.summaries(self.K, w.L, w.S)

    def q_step(self, Q: torch.Tensor, s: int) -> torch.Tensor:
        """Decode: the [B, Hq, 1, d] query of step s."""
        return Q[s].reshape(self.w.B, self.w.Hq, 1, self.w.d).contiguous()

    def route_all(self, Q: torch.Tensor, topk: int | None = None):
        w = self.w
        k = w.topk if topk is None else topk
        if w.kind == "decode":
            sels, margins = [], []
            for s in range(w.n_q):
                sel, m = oracle.route(self.q_step(Q, s), w.q_pos0 + s, self.summ, w.Hkv, w.S, k)
                sels.append(sel)
                margins.append(m)
            return np.stack(sels), np.stack(margins)   # [steps, B*Hq, k], [steps, B*Hq]
        sel, m = oracle.route(Q, w.q_pos0, self.summ, w.Hkv, w.S, k)
        return sel, m                                   # [B*Hq*n_q, k], [B*Hq*n_q]


def margin_checked_inputs(w: W.Workload, max_rounds: int = 64):
    """Inputs whose every query row has an oracle margin >= MARGIN.

    Returns (inputs, host Q, host K, oracle run, oracle sel, oracle margins,
    number of redrawn rows).
    """
    n_rows = int(np.prod(w.q_shape[:-1]))
    attempt = torch.zeros(n_rows, dtype=torch.int32)
    inp = W.Inputs(w, attempt=attempt)
    K = inp.k()
    orc = OracleRun(w, inp, K)
    Q = inp.q()
    redrawn = 0
    for _ in range(max_rounds):
        sel, margin = orc.route_all(Q)
        bad = _bad_rows(w, margin)
        if len(bad) == 0:
            report_margins(w.name, margin, redrawn)
            return inp, Q, K, orc, sel, margin, redrawn
        redrawn += len(bad)
        attempt[bad] += 1
        Q = inp.q()
    raise RuntimeError("could not reach the score margin for %d rows" % len(bad))


def _bad_rows(w: W.Workload, margin: np.ndarray) -> np.ndarray:
    """Global Q row indices (generator order) whose margin is too small."""
    if w.kind == "decode":
        return np.nonzero(margin.reshape(-1) < MARGIN)[0]      # [steps, B*Hq] = Q row order
    # prefill: oracle rows are [B, Hq, n_q] = Q row order as well
    return np.nonzero(margin < MARGIN)[0]


# ------------------------------------------------------------------ CUDA side
class DeviceRun:
    """Runs the CUDA path of a workload through the C ABI."""

    def __init__(self, w: W.Workload, Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor,
                 topk: int | None = None, device="cuda"):
        self.w = w
        self.topk = w.topk if topk is None else topk
        self.dev = torch.device(device)
        self.Q = Q.to(self.dev)
        self.K = K.to(self.dev)
        self.V = V.to(self.dev)
        self.p_full = params_of(w, topk=self.topk)
        ns_cap = (w.L + w.S - 1) // w.S
        self.summ = torch.zeros((w.B, w.Hkv, ns_cap, w.d), dtype=torch.float32, device=self.dev)

    def summaries(self, L: int | None = None, j0: int = 0, j1: int | None = None):
        w = self.w
        L = w.L if L is None else L
        p = params_of(w, L=L, topk=self.topk)
        if j1 is None:
            j1 = (L + w.S - 1) // w.S
        ssa.ssa_build_summaries(p, self.K, j0, j1, self.summ)

    def decode(self, steps: range | None = None, want_scores: bool = False, fused: bool = False):
        """Route + attend for decode steps; returns host (sel, O, lse[, scores], err).

        fused: each step is one ssa_decode_step call (the benchmark's path)
        instead of ssa_route then ssa_attend_decode."""
        w = self.w
        p = self.p_full
        ws = ssa.workspace(p, 1, ssa.SSA_OP_DECODE, self.dev)
        steps = range(w.n_q) if steps is None else steps
        sels, outs, lses, scs = [], [], [], []
        for s in steps:
            q = self.Q[s].contiguous()
            sel = torch.empty((w.B, w.Hq, 1, self.topk), dtype=torch.int32, device=self.dev)
            sc = torch.empty(sel.shape, dtype=torch.float32, device=self.dev) if want_scores else None
            O = torch.empty((w.B, w.Hq, w.d), dtype=w.dtype, device=self.dev)
            lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=self.dev)
            if fused:
                ssa.ssa_decode_step(p, q, w.q_pos0 + s, self.summ, self.K, self.V, sel, O, lse, ws)
            else:
                ssa.ssa_route(p, q, 1, w.q_pos0 + s, self.summ, sel, sc)
                ssa.ssa_attend_decode(p, q, w.q_pos0 + s, self.K, self.V, sel, O, lse, ws)
            sels.append(sel)
            outs.append(O)
            lses.append(lse)
            if want_scores:
                scs.append(sc)
        err = ssa.ssa_workspace_error(ws)
        out = (torch.stack(sels).reshape(len(steps), -1, self.topk).cpu().numpy(),
               torch.stack(outs).reshape(len(steps), -1, w.d).cpu(),
               torch.stack(lses).reshape(len(steps), -1).cpu())
        if want_scores:
            out = out + (torch.stack(scs).reshape(len(steps), -1, self.topk).cpu(),)
        return out + (err,)

    def prefill(self, chunked: bool = True):
        """Chunked prefill of all the workload's queries; returns host (sel, O, lse, err).

        Chunk c covers queries [c*chunk, (c+1)*chunk); before routing it, the
        spans the chunk's positions complete get their summaries and the valid
        cache length moves to the chunk's end.
        """
        w = self.w
        sel = torch.empty((w.B, w.Hq, w.n_q, self.topk), dtype=torch.int32, device=self.dev)
        O = torch.empty((w.B, w.Hq, w.n_q, w.d), dtype=w.dtype, device=self.dev)
        lse = torch.empty((w.B, w.Hq, w.n_q), dtype=torch.float32, device=self.dev)
        chunk = w.chunk if chunked else w.n_q
        # spans completed before the first chunk
        self.summaries(L=w.q_pos0, j0=0, j1=w.q_pos0 // w.S) if w.q_pos0 >= w.S else None
        errs = 0
        for c0 in range(0, w.n_q, chunk):
            n = min(chunk, w.n_q - c0)
            pos0 = w.q_pos0 + c0
            L_now = pos0 + n
            j0, j1 = pos0 // w.S, (L_now + w.S - 1) // w.S
            p = params_of(w, L=L_now, topk=self.topk)
            ssa.ssa_build_summaries(p, self.K, j0, j1, self.summ)
            qc = self.Q[:, :, c0: c0 + n].contiguous()
            sc = torch.empty((w.B, w.Hq, n, self.topk), dtype=torch.int32, device=self.dev)
            oc = torch.empty((w.B, w.Hq, n, w.d), dtype=w.dtype, device=self.dev)
            lc = torch.empty((w.B, w.Hq, n), dtype=torch.float32, device=self.dev)
            ws = ssa.workspace(p, n, ssa.SSA_OP_PREFILL, self.dev)
            wsr = ssa.workspace(p, n, ssa.SSA_OP_ROUTE, self.dev)
            ssa.ssa_route(p, qc, n, pos0, self.summ, sc, None, wsr)
            ssa.ssa_attend_prefill(p, qc, n, pos0, self.K, self.V, sc, oc, lc, ws)
            errs |= ssa.ssa_workspace_error(ws)
            if wsr is not None:
                errs |= ssa.ssa_workspace_error(wsr)
            sel[:, :, c0: c0 + n] = sc
            O[:, :, c0: c0 + n] = oc
            lse[:, :, c0: c0 + n] = lc
        return (sel.reshape(-1, self.topk).cpu().numpy(), O.reshape(-1, w.d).cpu(),
                lse.reshape(-1).cpu(), errs)


def max_abs(a, b) -> float:
    a = a.double().numpy() if isinstance(a, torch.Tensor) else np.asarray(a, np.float64)
    b = b.double().numpy() if isinstance(b, torch.Tensor) else np.asarray(b, np.float64)
    return float(np.abs(a - b).max()) if a.size else 0.0


def oracle_outputs_prefill(orc: OracleRun, Q, V, sel, rows=None):
    w = orc.w
    if rows is not None:
        sel = sel[rows]
    O, lse, _ = oracle.attend(Q, orc.K, V, w.q_pos0, w.S, sel, rows=rows)
    return O, lse


def oracle_outputs_decode(orc: OracleRun, Q, V, sel, steps):
    w = orc.w
    Os, ls = [], []
    for s in steps:
        O, lse, _ = oracle.attend(orc.q_step(Q, s), orc.K, V, w.q_pos0 + s, w.S, sel[s])
        Os.append(O)
        ls.append(lse)
    return np.stack(Os), np.stack(ls)


def scale_of(w: W.Workload) -> float:
    return 1.0 / math.sqrt(w.d)
