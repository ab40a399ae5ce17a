"""Group-shared selection (ssa_route_group) against the oracle's
route_group, and the attention it feeds against the oracle's attend.

Inputs are margin-checked per group: a group row whose k-th / (k+1)-th
summed-score margin is below 1e-3 has all of its g query heads redrawn.
"""
import numpy as np
import pytest
import torch

import content_routed_sparse_build_b300 as ssa
import oracle
from synth import workloads as W

from harness import LSE_TOL, MARGIN, TOL, DeviceRun, max_abs, params_of

pytestmark = pytest.mark.gpu

BF16, F16, F32 = torch.bfloat16, torch.float16, torch.float32


def group_checked_inputs(w: W.Workload, max_rounds: int = 64):
    """(inputs, host Q, host K, oracle summaries, group sel, margins)."""
    n_rows = int(np.prod(w.q_shape[:-1]))
    attempt = torch.zeros(n_rows, dtype=torch.int32)
    inp = W.Inputs(w, attempt=attempt)
    K = inp.k()
    summ = oracle.summaries(K, w.L, w.S)
    Q = inp.q()
    g = w.g
    for _ in range(max_rounds):
        if w.kind == "decode":
            sels, ms = [], []
            for s in range(w.n_q):
                sel, m = oracle.route_group(Q[s].reshape(w.B, w.Hq, 1, w.d).contiguous(), w.q_pos0 + s,
                                            summ, w.Hkv, w.S, w.topk)
                sels.append(sel)
                ms.append(m)
            sel, margin = np.stack(sels), np.stack(ms)          # [steps, B*Hq, k], [steps, B*Hq]
            bad = np.nonzero(margin.reshape(-1) < MARGIN)[0]     # Q row order: (step, b, h)
            heads = bad % w.Hq
            base = bad - heads
            redraw = (base[:, None] + (heads // g * g)[:, None] + np.arange(g)[None, :]).reshape(-1)
        else:
            sel, margin = oracle.route_group(Q, w.q_pos0, summ, w.Hkv, w.S, w.topk)
            bad = np.nonzero(margin < MARGIN)[0]                 # rows (b, h, i)
            i = bad % w.n_q
            bh = bad // w.n_q
            h0 = (bh % w.Hq) // g * g
            b = bh // w.Hq
            redraw = (((b * w.Hq)[:, None] + h0[:, None] + np.arange(g)[None, :]) * w.n_q
                      + i[:, None]).reshape(-1)
        if len(bad) == 0:
            return inp, Q, K, summ, sel, margin
        attempt[np.unique(redraw)] += 1
        Q = inp.q()
    raise RuntimeError("margin not reached")


DECODE_CASES = [
    W.Workload("group_decode_bf16_gqa8", "decode", 1, 32, 4, 128, 65536 + 100, 1024, 16, BF16,
               n_q=6, q_pos0=65536 + 94, chunk=1, needles=8, seed=71),
    W.Workload("group_decode_f32_d64", "decode", 2, 8, 2, 64, 6000, 128, 6, F32,
               n_q=3, q_pos0=5997, chunk=1, needles=2, seed=72),
    # the one-call group step with g = 16 and k = 40 (two-word router lists), B = 2, d = 64
    W.Workload("group_decode_f16_d64_g16_k40", "decode", 2, 16, 1, 64, 9000, 128, 40, F16,
               n_q=3, q_pos0=8997, chunk=1, needles=2, seed=75),
    # g = 4 and S = 300: items start inside 32-token tiles
    W.Workload("group_decode_bf16_g4_s300", "decode", 1, 16, 4, 128, 20000, 300, 8, BF16,
               n_q=3, q_pos0=19990, chunk=1, seed=76),
]
PREFILL_CASES = [
    W.Workload("group_prefill_bf16", "prefill", 1, 8, 2, 128, 3000, 128, 4, BF16,
               n_q=3000, q_pos0=0, chunk=1024, needles=2, seed=73),
    W.Workload("group_prefill_f16_g16", "prefill", 1, 16, 1, 64, 2100, 64, 5, F16,
               n_q=600, q_pos0=1500, chunk=600, seed=74),
]


def _decode_run(w, Q, K, V):
    """route_group + attend per step; where the fast decode path applies, the
    one-call group step runs beside them: the same selections bit for bit,
    and its own outputs (its work items are smaller, so its partials split
    the spans differently), which the tests hold to the oracle as well."""
    run = DeviceRun(w, Q, K, V)
    run.summaries()
    p = run.p_full
    ws = ssa.workspace(p, 1, ssa.SSA_OP_DECODE)
    wsg = ssa.workspace(p, 1, ssa.SSA_OP_ROUTE_GROUP)
    fused = ssa.ssa_attend_path(p, 1, ssa.SSA_OP_DECODE) == ssa.SSA_PATH_FAST
    sels, outs, lses, fouts, flses = [], [], [], [], []
    for s in range(w.n_q):
        q = run.Q[s].contiguous()
        sel = torch.empty((w.B, w.Hq, 1, w.topk), dtype=torch.int32, device="cuda")
        O = torch.empty((w.B, w.Hq, w.d), dtype=w.dtype, device="cuda")
        lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device="cuda")
        ssa.ssa_route_group(p, q, 1, w.q_pos0 + s, run.summ, sel, None, wsg)
        ssa.ssa_attend_decode(p, q, w.q_pos0 + s, run.K, run.V, sel, O, lse, ws)
        if fused:
            sel2, O2, lse2 = torch.full_like(sel, 7), torch.empty_like(O), torch.empty_like(lse)
            ssa.ssa_decode_step_group(p, q, w.q_pos0 + s, run.summ, run.K, run.V, sel2, O2, lse2, ws)
            assert torch.equal(sel2, sel), s
            fouts.append(O2.reshape(-1, w.d))
            flses.append(lse2.reshape(-1))
        sels.append(sel.reshape(-1, w.topk))
        outs.append(O.reshape(-1, w.d))
        lses.append(lse.reshape(-1))
    err = ssa.ssa_workspace_error(ws) | ssa.ssa_workspace_error(wsg)
    fused_out = (torch.stack(fouts).cpu(), torch.stack(flses).cpu()) if fused else None
    return (torch.stack(sels).cpu().numpy(), torch.stack(outs).cpu(), torch.stack(lses).cpu(), err, fused_out)


@pytest.mark.parametrize("w", DECODE_CASES, ids=lambda w: w.name)
def test_group_decode_parity(w):
    inp, Q, K, summ, sel_o, margin = group_checked_inputs(w)
    V = inp.v()
    sel_g, O_g, lse_g, err, fused = _decode_run(w, Q, K, V)
    assert err == 0
    assert np.array_equal(sel_g, sel_o)
    for s in range(w.n_q):
        q = Q[s].reshape(w.B, w.Hq, 1, w.d).contiguous()
        O_o, lse_o, _ = oracle.attend(q, K, V, w.q_pos0 + s, w.S, sel_o[s])
        assert max_abs(O_g[s], O_o) <= TOL[w.dtype]
        assert max_abs(lse_g[s], lse_o) <= LSE_TOL[w.dtype]
        if fused is not None:
            assert max_abs(fused[0][s], O_o) <= TOL[w.dtype]
            assert max_abs(fused[1][s], lse_o) <= LSE_TOL[w.dtype]


@pytest.mark.parametrize("w", PREFILL_CASES, ids=lambda w: w.name)
def test_group_prefill_parity(w):
    inp, Q, K, summ, sel_o, margin = group_checked_inputs(w)
    V = inp.v()
    run = DeviceRun(w, Q, K, V)
    sel = torch.empty((w.B, w.Hq, w.n_q, w.topk), dtype=torch.int32, device="cuda")
    O = torch.empty((w.B, w.Hq, w.n_q, w.d), dtype=w.dtype, device="cuda")
    lse = torch.empty((w.B, w.Hq, w.n_q), dtype=torch.float32, device="cuda")
    if w.q_pos0 >= w.S:
        run.summaries(L=w.q_pos0, j0=0, j1=w.q_pos0 // w.S)
    errs = 0
    for c0 in range(0, w.n_q, w.chunk):
        n = min(w.chunk, w.n_q - c0)
        pos0 = w.q_pos0 + c0
        L_now = pos0 + n
        p = params_of(w, L=L_now)
        ssa.ssa_build_summaries(p, run.K, pos0 // w.S, (L_now + w.S - 1) // w.S, run.summ)
        qc = run.Q[:, :, c0: c0 + n].contiguous()
        sc = torch.empty((w.B, w.Hq, n, w.topk), dtype=torch.int32, device="cuda")
        oc = torch.empty((w.B, w.Hq, n, w.d), dtype=w.dtype, device="cuda")
        lc = torch.empty((w.B, w.Hq, n), dtype=torch.float32, device="cuda")
        wsg = ssa.workspace(p, n, ssa.SSA_OP_ROUTE_GROUP)
        ws = ssa.workspace(p, n, ssa.SSA_OP_PREFILL)
        ssa.ssa_route_group(p, qc, n, pos0, run.summ, sc, None, wsg)
        ssa.ssa_attend_prefill(p, qc, n, pos0, run.K, run.V, sc, oc, lc, ws)
        errs |= ssa.ssa_workspace_error(ws) | ssa.ssa_workspace_error(wsg)
        sel[:, :, c0: c0 + n] = sc
        O[:, :, c0: c0 + n] = oc
        lse[:, :, c0: c0 + n] = lc
    assert errs == 0
    sel_g = sel.reshape(-1, w.topk).cpu().numpy()
    assert np.array_equal(sel_g, sel_o)
    O_o, lse_o, _ = oracle.attend(Q, K, V, w.q_pos0, w.S, sel_o)
    assert max_abs(O.reshape(-1, w.d).cpu(), O_o) <= TOL[w.dtype]
    assert max_abs(lse.reshape(-1).cpu(), lse_o) <= LSE_TOL[w.dtype]


def test_group_decode_1m_all_steps():
    """The 1M decode workload with group-shared selection: all 256 steps'
    selections, O / lse of 16 of them."""
    w = W.DECODE_1M
    inp, Q, K, summ, sel_o, margin = group_checked_inputs(w)
    V = inp.v()
    sel_g, O_g, lse_g, err, fused = _decode_run(w, Q, K, V)
    assert err == 0
    assert np.array_equal(sel_g, sel_o)
    assert fused is not None
    for s in range(0, w.n_q, 16):
        q = Q[s].reshape(w.B, w.Hq, 1, w.d).contiguous()
        O_o, lse_o, _ = oracle.attend(q, K, V, w.q_pos0 + s, w.S, sel_o[s])
        assert max_abs(O_g[s], O_o) <= TOL[w.dtype]
        assert max_abs(lse_g[s], lse_o) <= LSE_TOL[w.dtype]
        assert max_abs(fused[0][s], O_o) <= TOL[w.dtype]
        assert max_abs(fused[1][s], lse_o) <= LSE_TOL[w.dtype]
