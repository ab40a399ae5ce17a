"""ssa_attend_decode_noalloc (library-owned scratch) against ssa_attend_decode
(caller workspace) through the C ABI.

Both run the same kernels with the same work split, and every partial lands
in a fixed slot merged in a fixed order, so the outputs must be identical
bit for bit.  Two calls in a row check that the shared block is reused
cleanly.  The file sorts last so that it also runs after every other GPU
test in one session.
"""
import pytest
import torch

import content_routed_sparse_build_b300 as ssa
from synth import workloads as W

pytestmark = pytest.mark.gpu

BF16, F16, F32 = torch.bfloat16, torch.float16, torch.float32

CASES = [
    W.Workload("noalloc_bf16_gqa8", "decode", 1, 32, 4, 128, 65536 + 100, 1024, 16, BF16,
               n_q=2, q_pos0=65536 + 98, chunk=1, needles=4, seed=61),
    W.Workload("noalloc_f16_d64_b2", "decode", 2, 8, 2, 64, 9000, 128, 8, F16,
               n_q=2, q_pos0=8998, chunk=1, seed=62),
    W.Workload("noalloc_f32_rows", "decode", 1, 4, 2, 64, 3000, 64, 4, F32,
               n_q=2, q_pos0=2998, chunk=1, seed=63),
]


def _setup(w):
    inp = W.Inputs(w)
    dev = torch.device("cuda")
    Q, K, V = inp.q().to(dev), inp.k().to(dev), inp.v().to(dev)
    p = ssa.params(w.B, w.Hq, w.Hkv, w.d, w.L, w.S, w.topk, w.dtype)
    ns = (w.L + w.S - 1) // w.S
    summ = torch.zeros((w.B, w.Hkv, ns, w.d), dtype=torch.float32, device=dev)
    ssa.ssa_build_summaries(p, K, 0, ns, summ)
    return p, Q, K, V, summ


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_noalloc_matches_workspace_entry_two_calls(w):
    assert ssa.ssa_workspace_size(ssa.params(w.B, w.Hq, w.Hkv, w.d, w.L, w.S, w.topk, w.dtype), 1,
                                  ssa.SSA_OP_DECODE) <= ssa.SSA_NOALLOC_SCRATCH_BYTES
    p, Q, K, V, summ = _setup(w)
    ws = ssa.workspace(p, 1, ssa.SSA_OP_DECODE)
    block = None
    for s in range(2):
        pos = w.q_pos0 + s
        q = Q[s].contiguous()
        sel = torch.empty((w.B, w.Hq, 1, w.topk), dtype=torch.int32, device="cuda")
        ssa.ssa_route(p, q, 1, pos, summ, sel)
        O_ws = torch.empty((w.B, w.Hq, w.d), dtype=w.dtype, device="cuda")
        lse_ws = torch.empty((w.B, w.Hq), dtype=torch.float32, device="cuda")
        O_na = torch.full_like(O_ws, float("nan"))
        lse_na = torch.full_like(lse_ws, float("nan"))
        ssa.ssa_attend_decode(p, q, pos, K, V, sel, O_ws, lse_ws, ws)
        got = ssa.ssa_attend_decode_noalloc(p, q, pos, K, V, sel, O_na, lse_na)
        if block is None:
            block = got
        assert got.data_ptr() == block.data_ptr() != 0      # the same block each call
        assert got.data_ptr() % 256 == 0
        torch.cuda.synchronize()
        assert torch.equal(O_na, O_ws), "call %d: outputs differ" % s
        assert torch.equal(lse_na, lse_ws), "call %d: lse differs" % s
        assert ssa.ssa_workspace_error(got) == 0
    assert ssa.ssa_workspace_error(ws) == 0


def test_noalloc_rejects_problems_above_its_block():
    # 16 x 64 heads x (64 + 1) partials x d = 128 in fp32: far above 8 MiB
    p = ssa.params(16, 64, 4, 128, 1 << 20, 1024, 64, BF16)
    assert ssa.ssa_workspace_size(p, 1, ssa.SSA_OP_DECODE) > ssa.SSA_NOALLOC_SCRATCH_BYTES
    t = torch.zeros(64, dtype=BF16, device="cuda")
    sel = torch.zeros(64, dtype=torch.int32, device="cuda")
    with pytest.raises(ssa.SSAError) as e:
        ssa.ssa_attend_decode_noalloc(p, t, 5, t, t, sel, t, None)
    assert e.value.status == ssa.SSA_ERR_WORKSPACE


def test_noalloc_reports_argument_errors_like_the_workspace_entry():
    t = torch.zeros(64, dtype=BF16, device="cuda")
    sel = torch.zeros(64, dtype=torch.int32, device="cuda")
    bad_heads = ssa.params(1, 6, 4, 128, 4096, 64, 4, BF16)      # Hq not a multiple of Hkv
    with pytest.raises(ssa.SSAError) as e:
        ssa.ssa_attend_decode_noalloc(bad_heads, t, 5, t, t, sel, t, None)
    assert e.value.status == ssa.SSA_ERR_INVALID_ARG
    p = ssa.params(1, 8, 4, 128, 4096, 64, 4, BF16)
    with pytest.raises(ssa.SSAError) as e:
        ssa.ssa_attend_decode_noalloc(p, t, 4096, t, t, sel, t, None)   # pos == L
    assert e.value.status == ssa.SSA_ERR_INVALID_ARG
