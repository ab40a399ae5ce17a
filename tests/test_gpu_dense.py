"""With every candidate span selected (k >= number of spans), routed
attention is dense causal attention.  The CUDA path is checked here against
PyTorch's scaled_dot_product_attention in fp32 (the library the dense
comparison line of bench.py times), for prefill and for decode.  The oracle
pins the same identity on the CPU (test_all_spans_selected_equals_dense_causal)."""
import pytest
import torch
import torch.nn.functional as F

import content_routed_sparse_build_b300 as ssa
from synth import workloads as W

from harness import TOL, max_abs

pytestmark = pytest.mark.gpu


def _dense_causal(Q, K, V, q_pos0):
    """fp32 SDPA of Q [B, Hq, n, d] at positions q_pos0.. against keys 0.. of K, V."""
    B, Hq, n, d = Q.shape
    L = q_pos0 + n
    k, v = K[:, :, :L].float(), V[:, :, :L].float()
    pos = torch.arange(q_pos0, q_pos0 + n, device=Q.device)[:, None]
    mask = torch.arange(L, device=Q.device)[None, :] <= pos
    return F.scaled_dot_product_attention(Q.float(), k, v, attn_mask=mask, enable_gqa=True)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_prefill_with_every_span_is_dense_attention(dtype):
    w = W.Workload("dense_prefill", "prefill", 1, 8, 2, 128, 2048, 128, 16, dtype,
                   n_q=1024, q_pos0=1024, chunk=1024, seed=81)
    inp = W.Inputs(w)
    Q, K, V = inp.q("cuda"), inp.k("cuda"), inp.v("cuda")
    p = ssa.params(w.B, w.Hq, w.Hkv, w.d, w.L, w.S, w.topk, dtype)
    summ = torch.zeros((w.B, w.Hkv, w.n_spans, w.d), dtype=torch.float32, device="cuda")
    ssa.ssa_build_summaries(p, K, 0, w.n_spans, summ)
    sel = torch.empty((w.B, w.Hq, w.n_q, w.topk), dtype=torch.int32, device="cuda")
    O = torch.empty_like(Q)
    ssa.ssa_route(p, Q, w.n_q, w.q_pos0, summ, sel, None, ssa.workspace(p, w.n_q, ssa.SSA_OP_ROUTE))
    ws = ssa.workspace(p, w.n_q, ssa.SSA_OP_PREFILL)
    ssa.ssa_attend_prefill(p, Q, w.n_q, w.q_pos0, K, V, sel, O, None, ws)
    assert ssa.ssa_workspace_error(ws) == 0
    # every candidate is selected: at most 15 candidates (positions < 2048, S = 128), k = 16
    assert int((sel >= 0).sum(-1).max()) <= 15
    ref = _dense_causal(Q, K, V, w.q_pos0)
    assert max_abs(O.float().cpu(), ref.cpu()) <= TOL[dtype]


def test_decode_with_every_span_is_dense_attention():
    w = W.Workload("dense_decode", "decode", 1, 32, 4, 128, 8192 + 300, 512, 16, torch.bfloat16,
                   n_q=2, q_pos0=8192 + 298, chunk=1, seed=82)
    inp = W.Inputs(w)
    Q, K, V = inp.q("cuda"), inp.k("cuda"), inp.v("cuda")
    p = ssa.params(w.B, w.Hq, w.Hkv, w.d, w.L, w.S, w.topk, w.dtype)
    summ = torch.zeros((w.B, w.Hkv, w.n_spans, w.d), dtype=torch.float32, device="cuda")
    ssa.ssa_build_summaries(p, K, 0, w.n_spans, summ)
    ws = ssa.workspace(p, 1, ssa.SSA_OP_DECODE)
    for s in range(w.n_q):
        pos = w.q_pos0 + s
        q = Q[s].contiguous()
        sel = torch.empty((w.B, w.Hq, 1, w.topk), dtype=torch.int32, device="cuda")
        O = torch.empty((w.B, w.Hq, w.d), dtype=w.dtype, device="cuda")
        ssa.ssa_route(p, q, 1, pos, summ, sel)
        ssa.ssa_attend_decode(p, q, pos, K, V, sel, O, None, ws)
        ref = _dense_causal(q.reshape(w.B, w.Hq, 1, w.d), K, V, pos)
        assert max_abs(O.float().cpu(), ref.reshape(w.B, w.Hq, w.d).cpu()) <= TOL[w.dtype]
    assert ssa.ssa_workspace_error(ws) == 0
