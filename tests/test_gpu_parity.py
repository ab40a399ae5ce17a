"""CUDA path vs the CPU oracle on the same seeded inputs (small and medium sizes).

Selections must match bit for bit; outputs within 1e-5 (fp32) or 2e-2
(bf16 / fp16) max-abs error; lse within 1e-5 / 1e-3.
"""
import numpy as np
import pytest
import torch

import content_routed_sparse_build_b300 as ssa
import oracle
from synth import workloads as W

from harness import (LSE_TOL, TOL, DeviceRun, OracleRun, margin_checked_inputs, max_abs,
                     oracle_outputs_decode, oracle_outputs_prefill)

pytestmark = pytest.mark.gpu

BF16, F16, F32 = torch.bfloat16, torch.float16, torch.float32

PREFILL_CASES = [
    W.TINY_PREFILL,
    W.TINY_PREFILL.with_(name="tiny_prefill_dense_k64", topk=64),
    W.Workload("case_prefill_bf16_gqa_b2", "prefill", 2, 8, 2, 128, 3000, 128, 4, BF16,
               n_q=3000, q_pos0=0, chunk=1024, needles=2, seed=11),
    W.Workload("case_prefill_f16_d64_tail", "prefill", 1, 4, 4, 64, 2100, 64, 6, F16,
               n_q=1076, q_pos0=1024, chunk=512, lowrank=4, seed=12),
    W.Workload("case_prefill_bf16_g16", "prefill", 1, 16, 1, 128, 2048, 256, 3, BF16,
               n_q=600, q_pos0=1448, chunk=600, needles=2, seed=13),
    # k above the tensor-core router's 16 and above one merge batch of slots
    W.Workload("case_prefill_bf16_k20", "prefill", 1, 8, 2, 128, 4096, 64, 20, BF16,
               n_q=1024, q_pos0=3072, chunk=512, needles=2, seed=14),
    # k = 64 at d = 128: 65 partial slots per row, more than two merge lanes'
    # worth, and a merge row of 16,640 bytes (two rows in flight per warp)
    W.Workload("case_prefill_bf16_d128_k64", "prefill", 1, 8, 2, 128, 80 * 64 + 17, 64, 64, BF16,
               n_q=1024, q_pos0=80 * 64 + 17 - 1024, chunk=512, needles=2, seed=15),
    # spans of 512 tokens or more: the attend kernel's layout with two Q
    # buffers for tile B and a three-slot K / V ring
    W.Workload("case_prefill_bf16_s1024", "prefill", 1, 8, 2, 128, 10 * 1024 + 300, 1024, 4, BF16,
               n_q=1024, q_pos0=10 * 1024 + 300 - 1024, chunk=1024, needles=2, seed=16),
    W.Workload("case_prefill_f16_d64_s512", "prefill", 1, 4, 4, 64, 14 * 512 + 77, 512, 6, F16,
               n_q=700, q_pos0=14 * 512 + 77 - 700, chunk=700, seed=17),
]

DECODE_CASES = [
    W.Workload("case_decode_bf16_gqa8", "decode", 1, 32, 4, 128, 65536 + 100, 1024, 16, BF16,
               n_q=6, q_pos0=65536 + 100 - 6, chunk=1, needles=8, seed=21),
    W.Workload("case_decode_f16_d64_b2", "decode", 2, 8, 8, 64, 20000, 256, 8, F16,
               n_q=4, q_pos0=20000 - 4, chunk=1, needles=3, seed=22),
    W.Workload("case_decode_f32", "decode", 1, 4, 2, 64, 4096, 64, 8, F32,
               n_q=4, q_pos0=4092, chunk=1, needles=2, seed=23),
    W.Workload("case_decode_bf16_g16_small_ell", "decode", 1, 16, 1, 128, 5000, 512, 16, BF16,
               n_q=3, q_pos0=4997, chunk=1, seed=24),
    # 16,499 candidate spans: more than the plan's bitmap covers (16,384), so
    # the union positions come from its binary-search path
    W.Workload("case_decode_bf16_many_spans", "decode", 1, 8, 1, 64, 16500 * 64, 64, 8, BF16,
               n_q=2, q_pos0=16500 * 64 - 2, chunk=1, seed=25),
    # k above 32: the decode router's 64-entry lists
    W.Workload("case_decode_bf16_k64", "decode", 1, 16, 2, 128, 300 * 256 + 50, 256, 64, BF16,
               n_q=3, q_pos0=300 * 256 + 47, chunk=1, needles=4, seed=26),
    W.Workload("case_decode_f16_d64_g16_k40", "decode", 1, 16, 1, 64, 200 * 64 + 10, 64, 40, F16,
               n_q=3, q_pos0=200 * 64 + 7, chunk=1, seed=27),
]


@pytest.mark.parametrize("w", PREFILL_CASES, ids=lambda w: w.name)
def test_prefill_parity(w):
    inp, Q, K, orc, sel_o, margin, redrawn = margin_checked_inputs(w)
    V = inp.v()
    run = DeviceRun(w, Q, K, V)
    sel_g, O_g, lse_g, err = run.prefill()
    assert err == 0
    assert np.array_equal(sel_g, sel_o), "selection mismatch in %d rows" % int(
        (sel_g != sel_o).any(axis=1).sum())
    O_o, lse_o = oracle_outputs_prefill(orc, Q, V, sel_o)
    assert max_abs(O_g, O_o) <= TOL[w.dtype]
    assert max_abs(lse_g, lse_o) <= LSE_TOL[w.dtype]


@pytest.mark.parametrize("w", DECODE_CASES, ids=lambda w: w.name)
def test_decode_parity(w):
    inp, Q, K, orc, sel_o, margin, redrawn = margin_checked_inputs(w)
    V = inp.v()
    run = DeviceRun(w, Q, K, V)
    run.summaries()
    sel_g, O_g, lse_g, err = run.decode()
    assert err == 0
    assert np.array_equal(sel_g, sel_o)
    O_o, lse_o = oracle_outputs_decode(orc, Q, V, sel_o, range(w.n_q))
    assert max_abs(O_g, O_o) <= TOL[w.dtype]
    assert max_abs(lse_g, lse_o) <= LSE_TOL[w.dtype]


@pytest.mark.parametrize("w", DECODE_CASES, ids=lambda w: w.name)
def test_decode_step_parity(w):
    """ssa_decode_step (route with the plan built in its cluster, then the
    split attention and the merge) against the oracle and against the two
    calls."""
    inp, Q, K, orc, sel_o, margin, redrawn = margin_checked_inputs(w)
    V = inp.v()
    run = DeviceRun(w, Q, K, V)
    run.summaries()
    sel_g, O_g, lse_g, err = run.decode(fused=True)
    assert err == 0
    assert np.array_equal(sel_g, sel_o)
    O_o, lse_o = oracle_outputs_decode(orc, Q, V, sel_o, range(w.n_q))
    assert max_abs(O_g, O_o) <= TOL[w.dtype]
    assert max_abs(lse_g, lse_o) <= LSE_TOL[w.dtype]
    sel_2, O_2, lse_2, err2 = run.decode()
    assert err2 == 0 and np.array_equal(sel_2, sel_g)
    if w.dtype != F32:
        # same kernels for the attention, the same merge order: identical bits
        assert torch.equal(O_2, O_g) and torch.equal(lse_2, lse_g)


def test_summaries_parity_fp32_exactish():
    w = W.Workload("case_summ", "decode", 2, 4, 2, 128, 5000, 96, 4, BF16, n_q=1, q_pos0=4999,
                   chunk=1, seed=31)
    inp = W.Inputs(w)
    K = inp.k()
    run = DeviceRun(w, inp.q(), K, K)
    run.summaries()
    ref = oracle.summaries(K, w.L, w.S)
    got = run.summ.cpu().double().numpy()
    # fp32 accumulation of at most 96 bf16 values of magnitude < 5
    assert np.abs(got - ref).max() < 1e-5


def test_exact_arithmetic_ties_match():
    """Integer keys and queries make every fp32 score exact, so GPU and oracle
    scores are equal and the frequent exact ties must resolve identically."""
    B, Hq, Hkv, d, S, L, topk = 1, 8, 2, 128, 64, 64 * 40, 5
    rng = np.random.default_rng(5)
    K = torch.from_numpy(rng.integers(-2, 3, (B, Hkv, L, d)).astype(np.float32)).to(BF16)
    for dup_src, dup_dst in ((3, 17), (5, 6), (9, 30)):
        K[:, :, dup_dst * S:(dup_dst + 1) * S] = K[:, :, dup_src * S:(dup_src + 1) * S]
    Q = torch.from_numpy(rng.integers(-1, 2, (B, Hq, L, d)).astype(np.float32)).to(BF16)
    V = torch.from_numpy(rng.standard_normal((B, Hkv, L, d)).astype(np.float32)).to(BF16)
    w = W.Workload("ties", "prefill", B, Hq, Hkv, d, L, S, topk, BF16, n_q=L, q_pos0=0, chunk=L)
    summ = oracle.summaries(K, L, S)
    sel_o, margin = oracle.route(Q, 0, summ, Hkv, S, topk)
    assert (margin == 0).sum() > 100
    run = DeviceRun(w, Q, K, V)
    sel_g, O_g, lse_g, err = run.prefill(chunked=False)
    assert err == 0
    assert np.array_equal(sel_g, sel_o)
    # decode rows take the same decisions
    pos = L - 1
    p = ssa.params(B, Hq, Hkv, d, L, S, topk, BF16)
    q = run.Q[:, :, pos].contiguous()
    sel = torch.empty((B, Hq, 1, topk), dtype=torch.int32, device="cuda")
    ssa.ssa_route(p, q, 1, pos, run.summ, sel)
    rows = [h * L + pos for h in range(Hq)]
    assert np.array_equal(sel.reshape(-1, topk).cpu().numpy(), sel_o[rows])


def test_decode_matches_prefill_rows():
    w = W.Workload("case_consistency", "prefill", 1, 8, 2, 128, 4096, 256, 4, BF16,
                   n_q=512, q_pos0=3584, chunk=512, needles=2, seed=41)
    inp, Q, K, orc, sel_o, margin, _ = margin_checked_inputs(w)
    V = inp.v()
    run = DeviceRun(w, Q, K, V)
    sel_g, O_g, lse_g, err = run.prefill()
    assert np.array_equal(sel_g, sel_o)
    p = ssa.params(w.B, w.Hq, w.Hkv, w.d, w.L, w.S, w.topk, BF16)
    ws = ssa.workspace(p, 1, ssa.SSA_OP_DECODE)
    for i in (0, 255, 511):
        pos = w.q_pos0 + i
        q = run.Q[:, :, i].contiguous()
        sel = torch.empty((1, w.Hq, 1, w.topk), dtype=torch.int32, device="cuda")
        O = torch.empty((1, w.Hq, w.d), dtype=BF16, device="cuda")
        ssa.ssa_route(p, q, 1, pos, run.summ, sel)
        ssa.ssa_attend_decode(p, q, pos, run.K, run.V, sel, O, None, ws)
        rows = [h * w.n_q + i for h in range(w.Hq)]
        assert np.array_equal(sel.reshape(-1, w.topk).cpu().numpy(), sel_g[rows])
        assert max_abs(O.reshape(-1, w.d).cpu(), O_g[rows]) <= TOL[BF16]
    assert ssa.ssa_workspace_error(ws) == 0


def test_bad_selection_is_flagged_not_faulted():
    B, Hq, Hkv, d, S, L, topk = 1, 4, 2, 128, 64, 1024, 4
    g = torch.Generator().manual_seed(0)
    Q = torch.randn(B, Hq, d, generator=g).to(BF16).cuda()
    K = torch.randn(B, Hkv, L, d, generator=g).to(BF16).cuda()
    V = torch.randn(B, Hkv, L, d, generator=g).to(BF16).cuda()
    p = ssa.params(B, Hq, Hkv, d, L, S, topk, BF16)
    ws = ssa.workspace(p, 1, ssa.SSA_OP_DECODE)
    O = torch.empty(B, Hq, d, dtype=BF16, device="cuda")
    pos = 700  # local span 10, candidates 0..9
    bad = torch.tensor([[[[1, 2, 3, -1]], [[3, 2, 4, 5]], [[1, 1, 2, -1]], [[0, 12, -1, -1]]]],
                       dtype=torch.int32, device="cuda")
    ssa.ssa_attend_decode(p, Q, pos, K, V, bad, O, None, ws)
    assert ssa.ssa_workspace_error(ws) & ssa.SSA_DEVERR_BAD_SELECTION
    assert ssa.ssa_workspace_error(ws) == 0   # reading clears the record
    good = torch.tensor([[[[1, 2, 3, -1]]] * 4], dtype=torch.int32, device="cuda").reshape(1, 4, 1, 4)
    ssa.ssa_attend_decode(p, Q, pos, K, V, good, O, None, ws)
    assert ssa.ssa_workspace_error(ws) == 0
