"""Decode with incremental summary maintenance (superlinear release post,
geeks.co.kr/post/2077, "why this matters": the cache is kept and grows with
the conversation instead of being re-processed): the cache grows one token per step, and when a step's position starts a new
span, the span just completed gets its summary (one ssa_build_summaries call
over that span) before the query routes.  Selections and outputs must equal
the oracle's on the full cache, where every candidate span's summary is the
mean of its keys."""
import numpy as np
import pytest
import torch

import content_routed_sparse_build_b300 as ssa
import oracle
from synth import workloads as W

from harness import LSE_TOL, MARGIN, TOL, max_abs

pytestmark = pytest.mark.gpu


def test_decode_with_summaries_built_as_spans_complete():
    S = 256
    start = 6 * S - 3                 # three steps before span 5 completes, then into span 6
    w = W.Workload("incremental_decode", "decode", 1, 16, 2, 128, 8 * S, S, 4, torch.bfloat16,
                   n_q=12, q_pos0=start, chunk=1, needles=2, seed=91)
    attempt = torch.zeros(w.n_q * w.B * w.Hq, dtype=torch.int32)
    inp = W.Inputs(w, attempt=attempt)
    K, V = inp.k(), inp.v()
    summ_o = oracle.summaries(K, w.L, w.S)
    Q = inp.q()
    for _ in range(32):
        margins = []
        for s in range(w.n_q):
            _, m = oracle.route(Q[s].reshape(w.B, w.Hq, 1, w.d).contiguous(), w.q_pos0 + s, summ_o,
                                w.Hkv, w.S, w.topk)
            margins.append(m)
        bad = np.nonzero(np.stack(margins).reshape(-1) < MARGIN)[0]
        if len(bad) == 0:
            break
        attempt[bad] += 1
        Q = inp.q()
    Kd, Vd, Qd = K.cuda(), V.cuda(), Q.cuda()
    ns_cap = w.n_spans
    summ = torch.full((w.B, w.Hkv, ns_cap, w.d), float("nan"), dtype=torch.float32, device="cuda")
    # the spans complete before the first step
    p0 = ssa.params(w.B, w.Hq, w.Hkv, w.d, start, w.S, w.topk, w.dtype, L_cap=w.L)
    ssa.ssa_build_summaries(p0, Kd, 0, start // w.S, summ)
    built = start // w.S
    ws = ssa.workspace(ssa.params(w.B, w.Hq, w.Hkv, w.d, w.L, w.S, w.topk, w.dtype), 1, ssa.SSA_OP_DECODE)
    for s in range(w.n_q):
        pos = w.q_pos0 + s
        p = ssa.params(w.B, w.Hq, w.Hkv, w.d, pos + 1, w.S, w.topk, w.dtype, L_cap=w.L)
        ell = pos // w.S
        if ell > built:                       # span ell - 1 has just completed
            ssa.ssa_build_summaries(p, Kd, built, ell, summ)
            built = ell
        q = Qd[s].contiguous()
        sel = torch.empty((w.B, w.Hq, 1, w.topk), dtype=torch.int32, device="cuda")
        O = torch.empty((w.B, w.Hq, w.d), dtype=w.dtype, device="cuda")
        lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device="cuda")
        ssa.ssa_route(p, q, 1, pos, summ, sel)
        ssa.ssa_attend_decode(p, q, pos, Kd, Vd, sel, O, lse, ws)
        qh = Q[s].reshape(w.B, w.Hq, 1, w.d).contiguous()
        sel_o, _ = oracle.route(qh, pos, summ_o, w.Hkv, w.S, w.topk)
        assert np.array_equal(sel.reshape(-1, w.topk).cpu().numpy(), sel_o), pos
        O_o, lse_o, _ = oracle.attend(qh, K, V, pos, w.S, sel_o)
        assert max_abs(O.reshape(-1, w.d).cpu(), O_o) <= TOL[w.dtype]
        assert max_abs(lse.reshape(-1).cpu(), lse_o) <= LSE_TOL[w.dtype]
    assert built == (w.q_pos0 + w.n_q - 1) // w.S
    assert ssa.ssa_workspace_error(ws) == 0
