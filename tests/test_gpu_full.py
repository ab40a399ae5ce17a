"""CUDA path vs the oracle at the full workload sizes, in the launch
configuration the benchmark times.

Selections are compared bit for bit on every row whose oracle margin was
checked; outputs on every decode step and on seeded row samples of the
prefills, within the same tolerances as the small cases:

  decode at 1M      all 256 steps (selections and outputs)
  decode at 10M     all 128 steps (selections; outputs on compacted caches)
  chunk against 1M  every selection; outputs of a seeded 1/16 of the rows
  128K prefill      chunks 0 and 15 in full, a seeded 1/16 of the rows of
                    the other chunks (selections and outputs)

Each needle workload also routes its needle probe on the GPU (one query per
head at sqrt(d) times the kv-head's needle direction, at the run's last
position): it must select min(#needles, k) needle spans, and when the oracle
separates its k-th and (k+1)-th scores by the margin, exactly the oracle's
spans.  Probes are extra queries, outside every timed run.

The 10M decode case never holds the 20 GB cache on the host: the oracle's
summaries come from host regenerations of span ranges, and each step's
outputs are checked on a compacted cache that holds only the kv-head's
selected spans (in ascending order) followed by its local span (see
oracle/streamed.py), its rows read from the generator's device fill.
"""
import numpy as np
import pytest
import torch

import content_routed_sparse_build_b300 as ssa
import oracle
from oracle import streamed
from synth import workloads as W

from harness import (LSE_TOL, MARGIN, TOL, DeviceRun, margin_checked_inputs, max_abs, oracle_outputs_decode,
                     params_of, report_margins)

pytestmark = pytest.mark.gpu


def _sample(n, k, seed):
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(n, size=min(k, n), replace=False))


def _check_probe(w, inp, sel_probe, sel_gpu):
    """The needle probe's selections [B*Hq, k] (oracle) against the planted
    needles and against the GPU's selections."""
    need = min(w.needles, w.topk)
    for bh in range(w.B * w.Hkv):
        b, h = divmod(bh, w.Hkv)
        needles = set(int(j) for j in inp.needle_spans[bh])
        for hq in range(h * w.g, (h + 1) * w.g):
            row = b * w.Hq + hq
            for sel in (sel_probe[row], sel_gpu[row]):
                hits = sum(1 for j in sel if int(j) in needles)
                assert hits == need, (bh, hq, sorted(needles), sel)


def _probe_decode(w, inp, run, summ_o):
    """Routes and attends the probe at the last position, decode path."""
    t = w.last_pos
    q = inp.probe_q()                                      # [B, Hq, d]
    q4 = q.reshape(w.B, w.Hq, 1, w.d).contiguous()
    sel_o, margin = oracle.route(q4, t, summ_o, w.Hkv, w.S, w.topk)
    p = run.p_full
    qd = q.to(run.dev)
    sel = torch.empty((w.B, w.Hq, 1, w.topk), dtype=torch.int32, device=run.dev)
    O = torch.empty((w.B, w.Hq, w.d), dtype=w.dtype, device=run.dev)
    lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=run.dev)
    ws = ssa.workspace(p, 1, ssa.SSA_OP_DECODE, run.dev)
    ssa.ssa_route(p, qd, 1, t, run.summ, sel)
    ssa.ssa_attend_decode(p, qd, t, run.K, run.V, sel, O, lse, ws)
    assert ssa.ssa_workspace_error(ws) == 0
    sel_g = sel.reshape(-1, w.topk).cpu().numpy()
    _check_probe(w, inp, sel_o, sel_g)
    ok = margin >= MARGIN
    assert np.array_equal(sel_g[ok], sel_o[ok])
    report_margins(w.name + "/probe", margin, 0)
    # outputs are compared on the rows whose selections agree (every row the
    # margin separates, and any other that happens to agree)
    same = (sel_g == sel_o).all(axis=1)
    return q4, sel_o, same, O.reshape(-1, w.d).cpu(), lse.reshape(-1).cpu(), t


def test_decode_1m_all_steps():
    """All 256 decode steps at 1M, selections and outputs; then the probe."""
    w = W.DECODE_1M
    inp, Q, K, orc, sel_o, margin, _ = margin_checked_inputs(w)
    V = inp.v()
    run = DeviceRun(w, Q, K, V)
    run.summaries()
    sel_g, O_g, lse_g, err = run.decode()
    assert err == 0
    assert np.array_equal(sel_g, sel_o)
    steps = list(range(w.n_q))
    O_o, lse_o = oracle_outputs_decode(orc, Q, V, sel_o, steps)
    assert max_abs(O_g, O_o) <= TOL[w.dtype]
    assert max_abs(lse_g, lse_o) <= LSE_TOL[w.dtype]
    # the benchmark's path: one ssa_decode_step per step
    sel_f, O_f, lse_f, err = run.decode(fused=True)
    assert err == 0
    assert np.array_equal(sel_f, sel_o)
    assert max_abs(O_f, O_o) <= TOL[w.dtype]
    assert max_abs(lse_f, lse_o) <= LSE_TOL[w.dtype]
    q4, sel_p, same, O_p, lse_p, t = _probe_decode(w, inp, run, orc.summ)
    O_po, lse_po, _ = oracle.attend(q4, K, V, t, w.S, sel_p)
    assert max_abs(O_p[same], O_po[same]) <= TOL[w.dtype]
    assert max_abs(lse_p[same], lse_po[same]) <= LSE_TOL[w.dtype]


def test_prefill_chunk_vs_1m_all_rows():
    """The 8192-query chunk against the 1M cache, as one attend call: every
    selection, O / lse of a seeded 1/16 of the rows; then the probe as a
    two-query chunk at the last two positions (tensor-core router)."""
    w = W.PREFILL_1M
    inp, Q, K, orc, sel_o, margin, _ = margin_checked_inputs(w)
    V = inp.v()
    run = DeviceRun(w, Q, K, V)
    sel_g, O_g, lse_g, err = run.prefill()
    assert err == 0
    assert np.array_equal(sel_g, sel_o), "selection mismatch in %d rows" % int(
        (sel_g != sel_o).any(axis=1).sum())
    rows = _sample(sel_o.shape[0], sel_o.shape[0] // 16, 7)
    O_o, lse_o, _ = oracle.attend(Q, K, V, w.q_pos0, w.S, sel_o[rows], rows=rows)
    assert max_abs(O_g[rows], O_o) <= TOL[w.dtype]
    assert max_abs(lse_g[rows], lse_o) <= LSE_TOL[w.dtype]
    # probe: queries at positions L-2 and L-1, both the probe vector
    pq = inp.probe_q()                                                  # [B, Hq, d]
    qp = pq.reshape(w.B, w.Hq, 1, w.d).expand(w.B, w.Hq, 2, w.d).contiguous()
    pos0 = w.L - 2
    sel_po, m_po = oracle.route(qp, pos0, orc.summ, w.Hkv, w.S, w.topk)
    p = params_of(w)
    qd = qp.to(run.dev)
    sel = torch.empty((w.B, w.Hq, 2, w.topk), dtype=torch.int32, device=run.dev)
    O = torch.empty_like(qd)
    lse = torch.empty((w.B, w.Hq, 2), dtype=torch.float32, device=run.dev)
    wsr = ssa.workspace(p, 2, ssa.SSA_OP_ROUTE, run.dev)
    ws = ssa.workspace(p, 2, ssa.SSA_OP_PREFILL, run.dev)
    ssa.ssa_route(p, qd, 2, pos0, run.summ, sel, None, wsr)
    ssa.ssa_attend_prefill(p, qd, 2, pos0, run.K, run.V, sel, O, lse, ws)
    assert ssa.ssa_workspace_error(ws) == 0
    sel_pg = sel.reshape(-1, w.topk).cpu().numpy()
    ok = m_po >= MARGIN
    assert np.array_equal(sel_pg[ok], sel_po[ok])
    for i in range(2):
        idx = [r * 2 + i for r in range(w.B * w.Hq)]
        _check_probe(w, inp, sel_po[idx], sel_pg[idx])
    report_margins(w.name + "/probe", m_po, 0)
    same = (sel_pg == sel_po).all(axis=1)
    O_po, lse_po, _ = oracle.attend(qp, K, V, pos0, w.S, sel_po)
    assert max_abs(O.reshape(-1, w.d).cpu()[same], O_po[same]) <= TOL[w.dtype]
    assert max_abs(lse.reshape(-1).cpu()[same], lse_po[same]) <= LSE_TOL[w.dtype]


def test_prefill_128k_sampled_rows():
    """The whole 128K prefill in 16 chunks of 8192; the oracle checks every
    row of the first and last chunk and a seeded 1/16 of the rows of the
    others (selections and outputs)."""
    w = W.PREFILL_128K
    n_rows = w.B * w.Hq * w.n_q
    rid = np.arange(n_rows)
    i = rid % w.n_q
    chunk = i // w.chunk
    rng = np.random.default_rng(11)
    keep = (chunk == 0) | (chunk == w.n_q // w.chunk - 1) | (rng.random(n_rows) < 1 / 16)
    rows = rid[keep]
    attempt = torch.zeros(n_rows, dtype=torch.int32)
    inp = W.Inputs(w, attempt=attempt)
    K = inp.k()
    summ = oracle.summaries(K, w.L, w.S)
    Q = inp.q()
    redrawn = 0
    for _ in range(64):
        sel_o, margin = oracle.route(Q, w.q_pos0, summ, w.Hkv, w.S, w.topk, rows=rows)
        bad = rows[margin < MARGIN]
        if len(bad) == 0:
            break
        redrawn += len(bad)
        attempt[bad] += 1
        Q = inp.q()
    else:
        raise RuntimeError("margin not reached")
    report_margins(w.name, margin, redrawn)
    V = inp.v()
    run = DeviceRun(w, Q, K, V)
    sel_g, O_g, lse_g, err = run.prefill()
    assert err == 0
    assert np.array_equal(sel_g[rows], sel_o)
    O_o, lse_o, _ = oracle.attend(Q, K, V, w.q_pos0, w.S, sel_o, rows=rows)
    assert max_abs(O_g[rows], O_o) <= TOL[w.dtype]
    assert max_abs(lse_g[rows], lse_o) <= LSE_TOL[w.dtype]


def test_decode_10m_all_steps():
    """128 decode steps against the 10M cache: every selection, and the
    outputs of every step on compacted caches; then the probe (32 needles
    per kv-head, k = 16: all 16 spans it keeps must be needles)."""
    w = W.DECODE_10M
    n_rows = w.n_q * w.B * w.Hq
    attempt = torch.zeros(n_rows, dtype=torch.int32)
    inp = W.Inputs(w, attempt=attempt)
    summ = streamed.summaries_streamed(inp)
    Q = inp.q()
    redrawn = 0
    for _ in range(64):
        sels, margins = [], []
        for s in range(w.n_q):
            q = Q[s].reshape(w.B, w.Hq, 1, w.d).contiguous()
            sel, m = oracle.route(q, w.q_pos0 + s, summ, w.Hkv, w.S, w.topk)
            sels.append(sel)
            margins.append(m)
        sel_o, margin = np.stack(sels), np.stack(margins)
        bad = np.nonzero(margin.reshape(-1) < MARGIN)[0]
        if len(bad) == 0:
            break
        redrawn += len(bad)
        attempt[bad] += 1
        Q = inp.q()
    else:
        raise RuntimeError("margin not reached")
    report_margins(w.name, margin, redrawn)
    dev = torch.device("cuda")
    Kd, Vd = inp.k(dev), inp.v(dev)
    run = DeviceRun(w, Q, Kd, Vd)
    run.summaries()
    sel_g, O_g, lse_g, err = run.decode()
    assert err == 0
    assert np.array_equal(sel_g, sel_o)
    # the benchmark's path gives the same selections and bit-identical outputs
    sel_f, O_f, lse_f, err = run.decode(fused=True)
    assert err == 0
    assert np.array_equal(sel_f, sel_o)
    assert torch.equal(O_f, O_g) and torch.equal(lse_f, lse_g)
    # the probe routes on the device cache; its outputs are checked compacted too
    q4, sel_p, same, O_p, lse_p, t_p = _probe_decode(w, inp, run, summ)
    del run
    torch.cuda.empty_cache()
    cases = [(w.q_pos0 + s, Q[s], sel_o[s], O_g[s], lse_g[s], None) for s in range(w.n_q)]
    cases.append((t_p, q4.reshape(w.B, w.Hq, w.d), sel_p, O_p, lse_p, same))
    # The compacted caches are read from the device copy of the generated
    # cache (the generator's device fill equals its host regeneration bit for
    # bit: test_gpu_synth.py), gathered on the device and copied back.
    kv = {"k": Kd, "v": Vd}

    def fetch(which, bh, parts):
        b, h = divmod(bh, w.Hkv)
        idx = torch.cat([torch.arange(a, e, dtype=torch.int64) for a, e in parts]).to(dev)
        return kv[which][b, h].index_select(0, idx).cpu()

    for t, q, sel_s, O_s, lse_s, keep in cases:
        for rows, qc, Kc, Vc, pos, sel_c in streamed.compact_decode_step(inp, q, sel_s, t, fetch):
            O_o, lse_o, _ = oracle.attend(qc, Kc, Vc, pos, w.S, sel_c)
            m = np.ones(len(rows), bool) if keep is None else keep[rows]
            assert max_abs(O_s[rows][m], O_o[m]) <= TOL[w.dtype], t
            assert max_abs(lse_s[rows][m], lse_o[m]) <= LSE_TOL[w.dtype], t
