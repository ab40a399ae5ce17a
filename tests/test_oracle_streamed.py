"""The oracle's helpers for caches too large for the host (oracle/streamed.py),
checked on small caches that do fit: summaries from regenerated span ranges
equal the oracle's summaries of the whole cache, and a decode step attended
on its compacted cache equals the same step on the whole cache."""
import numpy as np
import torch

import oracle
from oracle import streamed
from synth import workloads as W


def _case():
    return W.Workload("case_streamed", "decode", 2, 8, 2, 64, 64 * 300 + 17, 64, 6, torch.bfloat16,
                      n_q=3, q_pos0=64 * 300 + 14, chunk=1, needles=4, seed=77)


def test_summaries_streamed_equal_the_whole_cache():
    w = _case()
    inp = W.Inputs(w)
    full = oracle.summaries(inp.k(), w.L, w.S)
    # small parts so that several ranges, and a partial last span, are stitched
    part = streamed.summaries_streamed(inp, spans_per_part=37)
    assert np.array_equal(part, full)


def test_compacted_step_equals_the_whole_cache():
    w = _case()
    inp = W.Inputs(w)
    K, V, Q = inp.k(), inp.v(), inp.q()
    summ = oracle.summaries(K, w.L, w.S)
    for s in range(w.n_q):
        t = w.q_pos0 + s
        q4 = Q[s].reshape(w.B, w.Hq, 1, w.d).contiguous()
        sel, _ = oracle.route(q4, t, summ, w.Hkv, w.S, w.topk)
        O, lse, _ = oracle.attend(q4, K, V, t, w.S, sel)
        seen = set()
        for rows, qc, Kc, Vc, pos, sel_c in streamed.compact_decode_step(inp, Q[s], sel, t):
            Oc, lc, _ = oracle.attend(qc, Kc, Vc, pos, w.S, sel_c)
            # the same token set in another order: equal up to summation order
            assert np.abs(Oc - O[rows]).max() < 1e-12
            assert np.abs(lc - lse[rows]).max() < 1e-12
            seen.update(rows)
        assert seen == set(range(w.B * w.Hq))
