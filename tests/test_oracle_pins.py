"""Pins of the CPU oracle against things other than itself.

Each pin is a closed form, a library routine the definition reduces to
(numpy mean, numpy lexsort, heapq, torch SDPA in float64), an invariant, or
a planted answer.  Integer-valued inputs make every score and span mean an
exact double, so selections (and their ties) compare exactly.
"""
import heapq
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth
from synth import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _int_inputs(B, Hq, Hkv, L, d, seed, lo=-4, hi=5, dtype=torch.float32):
    rng = np.random.default_rng(seed)
    Q = rng.integers(lo, hi, (B, Hq, L, d)).astype(np.float32)
    K = rng.integers(lo, hi, (B, Hkv, L, d)).astype(np.float32)
    V = rng.integers(lo, hi, (B, Hkv, L, d)).astype(np.float32)
    f = lambda a: torch.from_numpy(a).to(dtype).contiguous()
    return f(Q), f(K), f(V)


def _expand(t, g):
    return t.repeat_interleave(g, dim=1)


# ---------------------------------------------------------------- summaries
@pytest.mark.parametrize("L,S", [(64, 8), (61, 8), (40, 4)])
def test_summaries_equal_numpy_mean(L, S):
    _, K, _ = _int_inputs(2, 2, 2, L, 8, 1)
    got = oracle.summaries(K, L, S)
    Kn = K.double().numpy()
    for j in range((L + S - 1) // S):
        ref = Kn[:, :, j * S: min((j + 1) * S, L), :].mean(axis=2)
        assert np.array_equal(got[:, :, j], ref)


def test_summaries_partial_range_and_closed_form():
    L, S, d = 32, 8, 4
    K = torch.zeros(1, 1, L, d)
    for t in range(L):
        K[0, 0, t] = torch.tensor([t, 1.0, -2.0 * t, 0.5])
    s = oracle.summaries(K, L, S, 1, 3)
    # span j: mean of t over [8j, 8j+8) = 8j + 3.5
    for j in (1, 2):
        assert np.array_equal(s[0, 0, j], [8 * j + 3.5, 1.0, -2 * (8 * j + 3.5), 0.5])
    assert not s[0, 0, 0].any() and not s[0, 0, 3].any()


def test_summaries_widen_half_types_exactly():
    x = torch.tensor([1.5, -2.25, 0.0078125, 3.0e-5], dtype=torch.float32)
    for dt in (torch.bfloat16, torch.float16):
        K = x.to(dt).reshape(1, 1, 4, 1).contiguous()
        s = oracle.summaries(K, 4, 1)
        assert np.array_equal(s[0, 0, :, 0], K.double().reshape(-1).numpy())


# ---------------------------------------------------------------- routing
def _ref_scores(Q, K, S, Hkv, q_pos0=0):
    B, Hq, n_q, d = Q.shape
    L = K.shape[2]
    ns = L // S
    summ = K.double().numpy()[:, :, : ns * S].reshape(B, Hkv, ns, S, d).mean(axis=3)
    summ = np.repeat(summ, Hq // Hkv, axis=1)                     # head h -> kv head h // g
    return np.einsum("bhqc,bhjc->bhqj", Q.double().numpy(), summ)


@pytest.mark.parametrize("Hq,Hkv,S,topk", [(4, 2, 4, 3), (2, 2, 8, 2), (6, 3, 4, 5)])
def test_route_equals_full_sort_and_heap(Hq, Hkv, S, topk):
    L, d = 64, 4
    Q, K, _ = _int_inputs(2, Hq, Hkv, L, d, 7, lo=-2, hi=3)
    summ = oracle.summaries(K, L, S)
    sel, margin = oracle.route(Q, 0, summ, Hkv, S, topk)
    sc = _ref_scores(Q, K, S, Hkv)
    B = Q.shape[0]
    ties_seen = 0
    r = 0
    for b in range(B):
        for h in range(Hq):
            for t in range(L):
                ell = t // S
                s = sc[b, h, t, :ell]
                order = np.lexsort((np.arange(ell), -s))             # score desc, index asc
                ref = sorted(order[: min(topk, ell)].tolist())
                heap = sorted(heapq.nsmallest(min(topk, ell), range(ell), key=lambda j: (-s[j], j)))
                got = sel[r][sel[r] >= 0].tolist()
                assert got == ref == heap, (b, h, t)
                assert (sel[r][len(got):] == -1).all()
                if ell > topk:
                    ss = s[order]
                    assert margin[r] == ss[topk - 1] - ss[topk]
                    ties_seen += ss[topk - 1] == ss[topk]
                else:
                    assert margin[r] == np.inf
                r += 1
    assert ties_seen > 0  # the integer inputs do exercise the tie rule


def test_route_tie_goes_to_lower_index():
    # Spans 1 and 3 hold identical keys, span 2 is better than both and span 0
    # worse: with k = 2 the second slot is a tie between 1 and 3.
    S, d = 4, 2
    K = torch.zeros(1, 1, 20, d)
    K[0, 0, 0:4] = torch.tensor([-1.0, 0.0])
    K[0, 0, 4:8] = torch.tensor([0.5, 0.25])
    K[0, 0, 8:12] = torch.tensor([2.0, 0.0])
    K[0, 0, 12:16] = torch.tensor([0.5, 0.25])
    Q = torch.tensor([1.0, 0.0]).reshape(1, 1, 1, d)
    summ = oracle.summaries(K, 20, S)
    sel, margin = oracle.route(Q, 19, summ, 1, S, 2)
    assert sel.tolist() == [[1, 2]]
    assert margin[0] == 0.0


def test_route_probe_selects_every_needle():
    for w in (W.TINY_PREFILL, W.PREFILL_1M.with_(L=64 * 1024, n_q=1024, q_pos0=63 * 1024,
                                                  chunk=1024, S=1024, Hq=8, Hkv=2)):
        w = w.with_(S=w.S) if w is W.TINY_PREFILL else w.with_(S=256, needles=16)
        inp = W.Inputs(w)
        K = inp.k()
        summ = oracle.summaries(K, w.L, w.S)
        probe = inp.probe_q().reshape(w.B, w.Hq, 1, w.d).contiguous()
        sel, margin = oracle.route(probe, w.last_pos, summ, w.Hkv, w.S, w.topk)
        for b in range(w.B):
            for h in range(w.Hq):
                bh = b * w.Hkv + h // w.g
                got = set(sel[b * w.Hq + h].tolist()) - {-1}
                assert set(inp.needle_spans[bh].tolist()) <= got


# ---------------------------------------------------------------- group-shared route
@pytest.mark.parametrize("Hq,Hkv,S,topk", [(4, 2, 4, 3), (8, 2, 8, 2), (6, 3, 4, 5)])
def test_route_group_equals_full_sort_of_summed_scores(Hq, Hkv, S, topk):
    """Group selection = the first k of a full sort of the group's summed
    scores (computed here from the summed queries, by linearity), and every
    head of a group gets the same row."""
    L, d = 64, 4
    Q, K, _ = _int_inputs(2, Hq, Hkv, L, d, 11, lo=-2, hi=3)
    summ = oracle.summaries(K, L, S)
    sel, margin = oracle.route_group(Q, 0, summ, Hkv, S, topk)
    g = Hq // Hkv
    qsum = Q.double().numpy().reshape(2, Hkv, g, L, d).sum(axis=2)       # [B, Hkv, L, d]
    sc = np.einsum("bhqc,bhjc->bhqj", qsum, summ)
    ties_seen = 0
    for b in range(2):
        for h in range(Hq):
            for t in range(L):
                r = (b * Hq + h) * L + t
                ell = t // S
                s = sc[b, h // g, t, :ell]
                order = np.lexsort((np.arange(ell), -s))
                ref = sorted(order[: min(topk, ell)].tolist())
                got = sel[r][sel[r] >= 0].tolist()
                assert got == ref, (b, h, t)
                h0 = (h // g) * g
                assert (sel[r] == sel[(b * Hq + h0) * L + t]).all()
                if ell > topk:
                    ss = s[order]
                    assert margin[r] == ss[topk - 1] - ss[topk]
                    ties_seen += ss[topk - 1] == ss[topk]
    assert ties_seen > 0


def test_route_group_one_head_per_group_is_the_per_head_route():
    L, d, S, topk = 96, 8, 8, 4
    Q, K, _ = _int_inputs(1, 3, 3, L, d, 12)
    summ = oracle.summaries(K, L, S)
    a, ma = oracle.route_group(Q, 0, summ, 3, S, topk)
    b, mb = oracle.route(Q, 0, summ, 3, S, topk)
    assert np.array_equal(a, b) and np.array_equal(ma, mb)


def test_route_group_probe_selects_every_needle():
    w = W.TINY_PREFILL.with_(Hq=8, Hkv=2, needles=2)
    inp = W.Inputs(w)
    K = inp.k()
    summ = oracle.summaries(K, w.L, w.S)
    probe = inp.probe_q().reshape(w.B, w.Hq, 1, w.d).contiguous()
    sel, _ = oracle.route_group(probe, w.last_pos, summ, w.Hkv, w.S, w.topk)
    for h in range(w.Hq):
        got = set(sel[h].tolist()) - {-1}
        assert set(inp.needle_spans[h // w.g].tolist()) <= got


def test_route_reports_missing_summary():
    Q = torch.zeros(1, 1, 1, 2)
    with pytest.raises(ValueError):
        oracle.route(Q, 100, np.zeros((1, 1, 3, 2)), 1, 4, 2)


# ---------------------------------------------------------------- attention
def _sdpa_masked(Q, K, V, mask, scale):
    g = Q.shape[1] // K.shape[1]
    q, k, v = Q.double(), _expand(K.double(), g), _expand(V.double(), g)
    O = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale)
    x = torch.einsum("bhqc,bhtc->bhqt", q, k) * scale
    lse = torch.logsumexp(x.masked_fill(~mask, -math.inf), dim=-1)
    return O, lse


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (4, 2)])
def test_all_spans_selected_equals_dense_causal(dtype, Hq, Hkv):
    B, L, d, S = 2, 96, 16, 8
    Q = synth.normal((B, Hq, L, d), dtype, 3, 1)
    K = synth.normal((B, Hkv, L, d), dtype, 3, 2)
    V = synth.normal((B, Hkv, L, d), dtype, 3, 3)
    topk = L // S
    summ = oracle.summaries(K, L, S)
    sel, _ = oracle.route(Q, 0, summ, Hkv, S, topk)
    O, lse, ws = oracle.attend(Q, K, V, 0, S, sel)
    g = Hq // Hkv
    q, k, v = Q.double(), _expand(K.double(), g), _expand(V.double(), g)
    ref = F.scaled_dot_product_attention(q, k, v, is_causal=True, scale=1 / math.sqrt(d))
    x = torch.einsum("bhqc,bhtc->bhqt", q, k) / math.sqrt(d)
    causal = torch.ones(L, L, dtype=torch.bool).tril()
    ref_lse = torch.logsumexp(x.masked_fill(~causal, -math.inf), dim=-1)
    assert np.abs(O - ref.reshape(-1, d).numpy()).max() < 1e-12
    assert np.abs(lse - ref_lse.reshape(-1).numpy()).max() < 1e-12
    assert np.abs(ws - 1.0).max() < 1e-12


@pytest.mark.parametrize("q_pos0", [0, 40])
def test_sparse_attention_equals_masked_dense(q_pos0):
    B, Hq, Hkv, L, d, S, topk = 1, 4, 2, 128, 16, 8, 3
    n_q = L - q_pos0
    Qf = synth.normal((B, Hq, L, d), torch.float32, 4, 1)
    Q = Qf[:, :, q_pos0:].contiguous()
    K = synth.normal((B, Hkv, L, d), torch.float32, 4, 2)
    V = synth.normal((B, Hkv, L, d), torch.float32, 4, 3)
    summ = oracle.summaries(K, L, S)
    sel, _ = oracle.route(Q, q_pos0, summ, Hkv, S, topk)
    O, lse, ws = oracle.attend(Q, K, V, q_pos0, S, sel)
    mask = torch.zeros(B, Hq, n_q, L, dtype=torch.bool)
    r = 0
    for b in range(B):
        for h in range(Hq):
            for i in range(n_q):
                t = q_pos0 + i
                ell = t // S
                for j in sel[r]:
                    if j >= 0:
                        mask[b, h, i, j * S:(j + 1) * S] = True
                mask[b, h, i, ell * S: t + 1] = True
                r += 1
    ref, ref_lse = _sdpa_masked(Q, K, V, mask, 1 / math.sqrt(d))
    assert np.abs(O - ref.reshape(-1, d).numpy()).max() < 1e-12
    assert np.abs(lse - ref_lse.reshape(-1).numpy()).max() < 1e-12


def test_hand_micro_closed_forms():
    with open(os.path.join(GOLDEN, "hand_micro.json")) as f:
        case = json.load(f)
    L, S, d, k = case["L"], case["S"], case["d"], case["topk"]
    K = torch.tensor(case["K"], dtype=torch.float32).reshape(1, 1, L, d)
    V = torch.tensor(case["V"], dtype=torch.float32).reshape(1, 1, L, d)
    summ = oracle.summaries(K, L, S)
    env = {"exp": math.exp, "log": math.log, "sqrt": math.sqrt}
    for c in case["cases"]:
        Q = torch.tensor(c["q"], dtype=torch.float32).reshape(1, 1, 1, d)
        sel, _ = oracle.route(Q, c["pos"], summ, 1, S, k)
        assert sel[0].tolist() == c["sel"], c
        O, lse, _ = oracle.attend(Q, K, V, c["pos"], S, sel)
        expect = [eval(e, {"__builtins__": {}}, env) for e in c["O"]]
        assert np.abs(O[0] - expect).max() < 1e-12, c
        assert abs(lse[0] - eval(c["lse"], {"__builtins__": {}}, env)) < 1e-12, c


def test_invariants_shift_permutation_causality():
    B, Hq, Hkv, L, d, S, topk = 1, 2, 1, 64, 8, 8, 2
    Q = synth.normal((B, Hq, L, d), torch.float32, 5, 1)
    K = synth.normal((B, Hkv, L, d), torch.float32, 5, 2)
    # bf16-valued V, so that V + c below is exact in fp32
    V = synth.normal((B, Hkv, L, d), torch.bfloat16, 5, 3).float()
    summ = oracle.summaries(K, L, S)
    sel, _ = oracle.route(Q, 0, summ, Hkv, S, topk)
    O, lse, _ = oracle.attend(Q, K, V, 0, S, sel)
    # (1) shifting every value row by c shifts O by c (weights sum to one)
    c = torch.arange(d, dtype=torch.float32) * 0.25 - 1.0
    O2, lse2, _ = oracle.attend(Q, K, V + c, 0, S, sel)
    assert np.abs(O2 - O - c.numpy()).max() < 1e-12 and np.array_equal(lse2, lse)
    # (2) permuting tokens inside every span changes neither selection nor output
    perm = torch.cat([torch.randperm(S, generator=torch.Generator().manual_seed(j)) + j * S
                      for j in range(L // S)])
    Kp, Vp = K[:, :, perm].contiguous(), V[:, :, perm].contiguous()
    summ_p = oracle.summaries(Kp, L, S)
    selp, _ = oracle.route(Q, 0, summ_p, Hkv, S, topk)
    rows = np.array([(h * L + t) for h in range(Hq) for t in range(L) if t % S == S - 1])
    assert np.array_equal(selp[rows], sel[rows])
    Op, _, _ = oracle.attend(Q, Kp, Vp, 0, S, selp[rows], rows=rows)
    assert np.abs(Op - O[rows]).max() < 1e-12
    # (3) keys and values after a query's position do not change its output
    t = 37
    K3, V3 = K.clone(), V.clone()
    K3[:, :, t + 1:] = 9.0
    V3[:, :, t + 1:] = -9.0
    summ3 = oracle.summaries(K3, L, S)
    rows = np.array([h * L + t for h in range(Hq)])
    sel3, _ = oracle.route(Q, 0, summ3, Hkv, S, topk, rows=rows)
    assert np.array_equal(sel3, sel[rows])
    O3, lse3, _ = oracle.attend(Q, K3, V3, 0, S, sel3, rows=rows)
    assert np.array_equal(O3, O[rows]) and np.array_equal(lse3, lse[rows])


def test_decode_row_equals_prefill_row():
    B, Hq, Hkv, L, d, S, topk = 1, 4, 2, 80, 8, 8, 3
    Q = synth.normal((B, Hq, L, d), torch.bfloat16, 6, 1)
    K = synth.normal((B, Hkv, L, d), torch.bfloat16, 6, 2)
    V = synth.normal((B, Hkv, L, d), torch.bfloat16, 6, 3)
    summ = oracle.summaries(K, L, S)
    sel, margin = oracle.route(Q, 0, summ, Hkv, S, topk)
    O, lse, _ = oracle.attend(Q, K, V, 0, S, sel)
    for p in (3, 40, 79):
        q1 = Q[:, :, p: p + 1].contiguous()
        s1, m1 = oracle.route(q1, p, summ, Hkv, S, topk)
        o1, l1, _ = oracle.attend(q1, K, V, p, S, s1)
        rows = [h * L + p for h in range(Hq)]
        assert np.array_equal(s1, sel[rows]) and np.array_equal(m1, margin[rows])
        assert np.array_equal(o1, O[rows]) and np.array_equal(l1, lse[rows])


def test_attend_rejects_non_candidate_span():
    Q = torch.zeros(1, 1, 1, 2)
    K = torch.zeros(1, 1, 16, 2)
    with pytest.raises(ValueError):
        oracle.attend(Q, K, K, 9, 4, np.array([[2]], np.int32))   # span 2 is the local span


def test_needles_raise_selection_rate():
    # Reported-style check: among real queries, needle spans are chosen more
    # often than other spans.
    w = W.TINY_PREFILL
    inp = W.Inputs(w)
    Q, K = inp.q(), inp.k()
    summ = oracle.summaries(K, w.L, w.S)
    rows = np.arange(w.B * w.Hq * w.n_q).reshape(w.B * w.Hq, w.n_q)[:, 2048:].reshape(-1)
    sel, _ = oracle.route(Q, 0, summ, w.Hkv, w.S, w.topk, rows=rows)
    sel = sel.reshape(w.B * w.Hq, -1, w.topk)
    for h in range(w.Hq):
        counts = np.bincount(sel[h][sel[h] >= 0], minlength=w.n_spans)
        nd = inp.needle_spans[h]
        other = np.setdiff1d(np.arange(32), nd)
        assert counts[nd].mean() > counts[other].mean()


# ---------------------------------------------------------------- 8-bit rows
# The quantiser (SubQ release post, quantisation plan; scheme fixed by the
# library: symmetric rows, s = max|x| / 127, q = rint(x / s) in fp32).


def test_quantize_hand_examples():
    # s = 127 / 127 = 1 exactly: codes are the nearest integers, ties to even
    x = torch.tensor([[127.0, 0.5, 1.5, 2.5, -0.5, -1.5, 3.49, -126.6]], dtype=torch.float32)
    q, s = oracle.quantize_rows(x)
    assert s.tolist() == [1.0]
    assert q.tolist() == [[127, 0, 2, 2, 0, -2, 3, -127]]
    # all-zero row: scale 0, codes 0; negative extreme maps to -127
    x = torch.tensor([[0.0, 0.0], [-4.0, 1.0]], dtype=torch.float32)
    q, s = oracle.quantize_rows(x)
    assert q.tolist() == [[0, 0], [-127, 32]]      # 1 / (4 / 127) = 31.75 -> 32
    assert s[0] == 0.0 and s[1] == np.float32(4.0) / np.float32(127.0)


def test_quantize_invariants_on_random_rows():
    g = torch.Generator().manual_seed(3)
    for dt in (torch.float32, torch.bfloat16, torch.float16):
        x = (torch.randn((64, 128), generator=g) * torch.rand((64, 1), generator=g) * 10).to(dt)
        q, s = oracle.quantize_rows(x)
        xf = x.float().numpy().astype(np.float64)
        amax = np.abs(xf).max(axis=1)
        # the largest element of every row maps to +-127
        assert (np.abs(q).max(axis=1) == 127).all()
        assert np.allclose(s, amax / 127.0, rtol=2 ** -23, atol=0)
        # reconstruction within half a step, plus the fp32 rounding of s and
        # of x / s (relative 2^-24 each, times at most 127 steps)
        err = np.abs(xf - q.astype(np.float64) * s.astype(np.float64)[:, None])
        assert (err <= (0.5 + 127 * 2.0 ** -22) * s[:, None]).all()
        # signs agree or the code is 0
        assert ((np.sign(q) == np.sign(xf)) | (q == 0)).all()


def test_quantize_is_equivariant_under_powers_of_two():
    g = torch.Generator().manual_seed(4)
    x = torch.randn((16, 64), generator=g)
    q1, s1 = oracle.quantize_rows(x)
    for k in (-3, 5):
        q2, s2 = oracle.quantize_rows(x * 2.0 ** k)
        assert np.array_equal(q1, q2)
        assert np.array_equal(s2, s1 * np.float32(2.0 ** k))


# ---------------------------------------------------------------- 4-bit rows
# The same scheme with 15 levels: s = max|x| / 7, q = rint(x / s) in [-7, 7].


def test_quantize4_hand_examples():
    # s = 7 / 7 = 1 exactly: codes are the nearest integers, ties to even
    x = torch.tensor([[7.0, 0.5, 1.5, 2.5, -0.5, -1.5, 3.49, -6.6, -3.5]], dtype=torch.float32)
    q, s = oracle.quantize_rows4(x)
    assert s.tolist() == [1.0]
    assert q.tolist() == [[7, 0, 2, 2, 0, -2, 3, -7, -4]]
    x = torch.tensor([[0.0, 0.0], [-14.0, 1.0], [2.0, -1.0]], dtype=torch.float32)
    q, s = oracle.quantize_rows4(x)
    # 1 / (14 / 7) = 0.5 -> 0 (tie to even); -1 / fp32(2 / 7) is -3.4999998
    # in fp32 (the scale rounds up), so it is no tie: -> -3
    assert q.tolist() == [[0, 0], [-7, 0], [7, -3]]
    assert np.float32(-1.0) / (np.float32(2.0) / np.float32(7.0)) > np.float32(-3.5)
    assert s[0] == 0.0 and s[1] == np.float32(2.0) and s[2] == np.float32(2.0) / np.float32(7.0)


def test_quantize4_invariants_on_random_rows():
    g = torch.Generator().manual_seed(13)
    for dt in (torch.float32, torch.bfloat16, torch.float16):
        x = (torch.randn((64, 128), generator=g) * torch.rand((64, 1), generator=g) * 10).to(dt)
        q, s = oracle.quantize_rows4(x)
        xf = x.float().numpy().astype(np.float64)
        amax = np.abs(xf).max(axis=1)
        assert (np.abs(q).max(axis=1) == 7).all()
        assert np.allclose(s, amax / 7.0, rtol=2 ** -23, atol=0)
        err = np.abs(xf - q.astype(np.float64) * s.astype(np.float64)[:, None])
        assert (err <= (0.5 + 7 * 2.0 ** -22) * s[:, None]).all()
        assert ((np.sign(q) == np.sign(xf)) | (q == 0)).all()


def test_quantize4_is_equivariant_under_powers_of_two():
    g = torch.Generator().manual_seed(14)
    x = torch.randn((16, 64), generator=g)
    q1, s1 = oracle.quantize_rows4(x)
    for k in (-3, 5):
        q2, s2 = oracle.quantize_rows4(x * 2.0 ** k)
        assert np.array_equal(q1, q2)
        assert np.array_equal(s2, s1 * np.float32(2.0 ** k))


def test_dequantized_summaries_and_attention_accept_f64():
    g = torch.Generator().manual_seed(5)
    K = torch.randn((1, 1, 32, 4), generator=g)
    q, s = oracle.quantize_rows(K)
    Kd = oracle.dequantize_rows(q, s)
    assert Kd.dtype == torch.float64
    assert np.array_equal(Kd.numpy(), q.astype(np.float64) * s.astype(np.float64)[..., None])
    summ = oracle.summaries(Kd, 32, 8)
    assert np.allclose(summ[0, 0], Kd.numpy()[0, 0].reshape(4, 8, 4).mean(axis=1), rtol=0, atol=1e-15)


def test_f64_inputs_match_their_f32_values_exactly():
    # the fp64 input path (used for dequantised caches) widens nothing: the
    # same values given as fp32 and as fp64 produce identical oracle results
    g = torch.Generator().manual_seed(6)
    B, Hq, Hkv, L, d, S, k = 1, 4, 2, 96, 8, 16, 2
    Q = torch.randn((B, Hq, L, d), generator=g)
    K = torch.randn((B, Hkv, L, d), generator=g)
    V = torch.randn((B, Hkv, L, d), generator=g)
    s32 = oracle.summaries(K, L, S)
    s64 = oracle.summaries(K.double(), L, S)
    assert np.array_equal(s32, s64)
    sel32, m32 = oracle.route(Q, 0, s32, Hkv, S, k)
    sel64, m64 = oracle.route(Q.double(), 0, s64, Hkv, S, k)
    assert np.array_equal(sel32, sel64) and np.array_equal(m32, m64)
    o32, l32, _ = oracle.attend(Q, K, V, 0, S, sel32)
    o64, l64, _ = oracle.attend(Q.double(), K.double(), V.double(), 0, S, sel32)
    assert np.array_equal(o32, o64) and np.array_equal(l32, l64)
