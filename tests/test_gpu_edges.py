"""Edge cases of the CUDA path against the oracle: exact score ties on a
large scale, the first positions of a cache, and an empty chunk.

Ties.  With integer keys and queries every summary is a multiple of 1/S and
every score is exact in fp32 as in double, so the GPU and the oracle see
the same scores and equal scores must resolve the same way (the lower span
first).  A cache whose spans repeat with a period P makes ties the rule:
every span of one residue class mod P has the same summary, so a query's
best k are the lowest spans of its best residues.  A query of zeros scores
every span 0, so its k best are spans 0 .. k-1.
"""
import numpy as np
import pytest
import torch

import content_routed_sparse_build_b300 as ssa
import oracle
from synth import workloads as W

from harness import LSE_TOL, TOL, DeviceRun, max_abs

pytestmark = pytest.mark.gpu

BF16 = torch.bfloat16


def _periodic_cache(B, Hkv, L, d, S, P, seed):
    """Integer K (values -2..2) whose span j equals span j mod P; normal V."""
    rng = np.random.default_rng(seed)
    base = rng.integers(-2, 3, (B, Hkv, P * S, d)).astype(np.float32)
    reps = -(-L // (P * S))
    K = np.tile(base, (1, 1, reps, 1))[:, :, :L]
    V = rng.standard_normal((B, Hkv, L, d)).astype(np.float32)
    return torch.from_numpy(K).to(BF16), torch.from_numpy(V).to(BF16)


def _int_queries(shape, seed):
    rng = np.random.default_rng(seed)
    return torch.from_numpy(rng.integers(-1, 2, shape).astype(np.float32)).to(BF16)


@pytest.mark.parametrize("topk", [16, 64])
def test_decode_periodic_cache_ties(topk):
    B, Hq, Hkv, d, S, P = 1, 16, 2, 128, 64, 5
    L = 64 * 300 + 17
    n = 4
    K, V = _periodic_cache(B, Hkv, L, d, S, P, seed=31)
    Q = _int_queries((n, B, Hq, d), seed=32)
    w = W.Workload("ties_decode", "decode", B, Hq, Hkv, d, L, S, topk, BF16, n_q=n, q_pos0=L - n, chunk=1)
    summ = oracle.summaries(K, L, S)
    sel_o = np.stack([oracle.route(Q[s].reshape(B, Hq, 1, d).contiguous(), w.q_pos0 + s, summ, Hkv, S, topk)[0]
                      for s in range(n)])
    run = DeviceRun(w, Q, K, V)
    run.summaries()
    for fused in (False, True):
        sel_g, O_g, lse_g, err = run.decode(fused=fused)
        assert err == 0
        assert np.array_equal(sel_g, sel_o)
    for s in range(n):
        O_o, lse_o, _ = oracle.attend(Q[s].reshape(B, Hq, 1, d).contiguous(), K, V, w.q_pos0 + s, S, sel_o[s])
        assert max_abs(O_g[s], O_o) <= TOL[BF16]
        assert max_abs(lse_g[s], lse_o) <= LSE_TOL[BF16]


def test_prefill_periodic_cache_ties():
    """The tensor-core router (k <= 16) and the span-major attention."""
    B, Hq, Hkv, d, S, P, topk = 1, 8, 2, 128, 64, 7, 16
    L = 64 * 200
    n = 512
    K, V = _periodic_cache(B, Hkv, L, d, S, P, seed=33)
    Q = _int_queries((B, Hq, n, d), seed=34)
    w = W.Workload("ties_prefill", "prefill", B, Hq, Hkv, d, L, S, topk, BF16, n_q=n, q_pos0=L - n, chunk=n)
    summ = oracle.summaries(K, L, S)
    sel_o, _ = oracle.route(Q, L - n, summ, Hkv, S, topk)
    run = DeviceRun(w, Q, K, V)
    sel_g, O_g, lse_g, err = run.prefill()
    assert err == 0
    assert np.array_equal(sel_g, sel_o)
    O_o, lse_o, _ = oracle.attend(Q, K, V, L - n, S, sel_o)
    assert max_abs(O_g, O_o) <= TOL[BF16]
    assert max_abs(lse_g, lse_o) <= LSE_TOL[BF16]


def test_zero_queries_take_the_lowest_spans():
    B, Hq, Hkv, d, S, topk = 1, 8, 2, 128, 64, 16
    L = 64 * 100 + 5
    rng = np.random.default_rng(35)
    K = torch.from_numpy(rng.standard_normal((B, Hkv, L, d)).astype(np.float32)).to(BF16)
    V = torch.from_numpy(rng.standard_normal((B, Hkv, L, d)).astype(np.float32)).to(BF16)
    # decode
    n = 3
    Qd = torch.zeros((n, B, Hq, d), dtype=BF16)
    wd = W.Workload("zero_q_decode", "decode", B, Hq, Hkv, d, L, S, topk, BF16, n_q=n, q_pos0=L - n, chunk=1)
    run = DeviceRun(wd, Qd, K, V)
    run.summaries()
    want = np.broadcast_to(np.arange(topk, dtype=np.int32), (n, B * Hq, topk))
    for fused in (False, True):
        sel_g, O_g, lse_g, err = run.decode(fused=fused)
        assert err == 0
        assert np.array_equal(sel_g, want)
    O_o, lse_o, _ = oracle.attend(Qd[0].reshape(B, Hq, 1, d).contiguous(), K, V, L - n, S, want[0])
    assert max_abs(O_g[0], O_o) <= TOL[BF16]
    # prefill chunk (tensor-core router)
    m = 256
    Qp = torch.zeros((B, Hq, m, d), dtype=BF16)
    wp = W.Workload("zero_q_prefill", "prefill", B, Hq, Hkv, d, L, S, topk, BF16, n_q=m, q_pos0=L - m, chunk=m)
    sel_p, O_p, lse_p, err = DeviceRun(wp, Qp, K, V).prefill()
    assert err == 0
    assert np.array_equal(sel_p, np.broadcast_to(np.arange(topk, dtype=np.int32), sel_p.shape))


@pytest.mark.parametrize("pos", [0, 1, 63, 64, 65, 127])
def test_first_positions(pos):
    """Decode at the start of a cache: no candidate at all (pos < S), then
    one complete span with a one-token local span (pos = S)."""
    B, Hq, Hkv, d, S, topk = 1, 8, 2, 128, 64, 4
    L = pos + 1
    rng = np.random.default_rng(36 + pos)
    K = torch.from_numpy(rng.standard_normal((B, Hkv, L, d)).astype(np.float32)).to(BF16)
    V = torch.from_numpy(rng.standard_normal((B, Hkv, L, d)).astype(np.float32)).to(BF16)
    Q = torch.from_numpy(rng.standard_normal((1, B, Hq, d)).astype(np.float32)).to(BF16)
    w = W.Workload("first_positions", "decode", B, Hq, Hkv, d, L, S, topk, BF16, n_q=1, q_pos0=pos, chunk=1)
    summ = oracle.summaries(K, L, S)
    q4 = Q[0].reshape(B, Hq, 1, d).contiguous()
    sel_o, _ = oracle.route(q4, pos, summ, Hkv, S, topk)
    O_o, lse_o, _ = oracle.attend(q4, K, V, pos, S, sel_o)
    run = DeviceRun(w, Q, K, V)
    run.summaries()
    for fused in (False, True):
        sel_g, O_g, lse_g, err = run.decode(fused=fused)
        assert err == 0
        assert np.array_equal(sel_g[0], sel_o)
        assert max_abs(O_g[0], O_o) <= TOL[BF16]
        assert max_abs(lse_g[0], lse_o) <= LSE_TOL[BF16]
    if pos == 0:
        # one token: the output is its value row
        assert max_abs(O_g[0], V[0, np.arange(Hq) // (Hq // Hkv), 0]) <= TOL[BF16]


def test_empty_chunk_is_a_no_op():
    B, Hq, Hkv, d, S, topk = 1, 8, 2, 128, 64, 4
    L = 256
    p = ssa.params(B, Hq, Hkv, d, L, S, topk, BF16)
    dev = torch.device("cuda")
    Q = torch.zeros((B, Hq, 1, d), dtype=BF16, device=dev)
    K = torch.zeros((B, Hkv, L, d), dtype=BF16, device=dev)
    summ = torch.zeros((B, Hkv, L // S, d), dtype=torch.float32, device=dev)
    sel = torch.full((B, Hq, 1, topk), 7, dtype=torch.int32, device=dev)
    O = torch.full((B, Hq, 1, d), 3.0, dtype=BF16, device=dev)
    ws = ssa.workspace(p, 1, ssa.SSA_OP_PREFILL, dev)
    ssa.ssa_route(p, Q, 0, 10, summ, sel, None, ssa.workspace(p, 1, ssa.SSA_OP_ROUTE, dev))
    ssa.ssa_attend_prefill(p, Q, 0, 10, K, K, sel, O, None, ws)
    torch.cuda.synchronize()
    assert ssa.ssa_workspace_error(ws) == 0
    assert bool((sel == 7).all()) and bool((O == 3.0).all())


@pytest.mark.parametrize("cache", ["16", "q8", "q4"])
def test_decode_step_with_mapped_host_buffers(cache):
    """The one-call steps take page-locked host Q, sel, O and lse directly
    (the route reads Q once over the link, the merge writes O in place) and
    give the same bits as with device buffers; pageable host memory is
    refused before anything is launched."""
    w = W.DECODE_1M.with_(name="host_buffers", L=1 << 18, q_pos0=(1 << 18) - 4, n_q=4)
    inp = W.Inputs(w)
    dev = torch.device("cuda")
    K, V = inp.k(dev), inp.v(dev)
    Q = inp.q()
    p = ssa.params(w.B, w.Hq, w.Hkv, w.d, w.L, w.S, w.topk, w.dtype)
    summ = torch.zeros((w.B, w.Hkv, w.n_spans, w.d), dtype=torch.float32, device=dev)
    ws = ssa.workspace(p, 1, ssa.SSA_OP_DECODE, dev)
    if cache == "q8":
        Kq, Ks, Vq, Vs = ssa.q8_cache(p, dev)
        ssa.ssa_quantize_kv(p, K, V, 0, w.L, Kq, Ks, Vq, Vs)
        ssa.ssa_build_summaries_q8(p, Kq, Ks, 0, w.n_spans, summ)

        def step(q, pos, sel, O, lse):
            ssa.ssa_decode_step_q8(p, q, pos, summ, Kq, Ks, Vq, Vs, sel, O, lse, ws)
    elif cache == "q4":
        Kq, Ks, Vq, Vs = ssa.q4_cache(p, dev)
        ssa.ssa_quantize_kv4(p, K, V, 0, w.L, Kq, Ks, Vq, Vs)
        ssa.ssa_build_summaries_q4(p, Kq, Ks, 0, w.n_spans, summ)

        def step(q, pos, sel, O, lse):
            ssa.ssa_decode_step_q4(p, q, pos, summ, Kq, Ks, Vq, Vs, sel, O, lse, ws)
    else:
        ssa.ssa_build_summaries(p, K, 0, w.n_spans, summ)

        def step(q, pos, sel, O, lse):
            ssa.ssa_decode_step(p, q, pos, summ, K, V, sel, O, lse, ws)
    for s in range(w.n_q):
        pos = w.q_pos0 + s
        qd = Q[s].to(dev)
        sel_d = torch.empty((w.B, w.Hq, 1, w.topk), dtype=torch.int32, device=dev)
        O_d = torch.empty((w.B, w.Hq, w.d), dtype=w.dtype, device=dev)
        lse_d = torch.empty((w.B, w.Hq), dtype=torch.float32, device=dev)
        step(qd, pos, sel_d, O_d, lse_d)
        qh = Q[s].contiguous().pin_memory()
        sel_h = torch.empty(sel_d.shape, dtype=torch.int32).pin_memory()
        O_h = torch.empty(O_d.shape, dtype=w.dtype).pin_memory()
        lse_h = torch.empty(lse_d.shape, dtype=torch.float32).pin_memory()
        step(qh, pos, sel_h, O_h, lse_h)
        torch.cuda.synchronize()
        assert torch.equal(sel_h, sel_d.cpu()) and torch.equal(O_h, O_d.cpu()) and torch.equal(lse_h, lse_d.cpu())
    assert ssa.ssa_workspace_error(ws) == 0
    # pageable host memory: an argument error, nothing launched
    with pytest.raises(ssa.SSAError) as e:
        step(Q[0].contiguous(), w.q_pos0, sel_d, O_d, lse_d)
    assert e.value.status == ssa.SSA_ERR_INVALID_ARG
