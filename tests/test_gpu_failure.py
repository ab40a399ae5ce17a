"""Failure detection on the device, without a fault: a bounded wait that
runs out.  The library's kernels wait on mbarriers for their bulk copies and
tensor-core work with a 2 s limit and, when a wait gives up, record
SSA_DEVERR_WAIT_TIMEOUT in the workspace and return.  Here a self-test
kernel runs that same wait on a barrier nothing completes (no copy, no
tensor memory in flight), so that the give-up path is exercised on a real
device: the status must come back to the host, and the context must stay
usable for the real path afterwards."""
import numpy as np
import pytest
import torch

import content_routed_sparse_build_b300 as ssa
from synth import workloads as W

pytestmark = pytest.mark.gpu


def _ws():
    t = torch.zeros(512, dtype=torch.uint8, device="cuda")
    off = (-t.data_ptr()) % 256
    return t[off: off + 256]


@pytest.mark.parametrize("limit_ms", [0, 20, 100])
def test_a_wait_that_runs_out_is_reported_and_the_context_stays_usable(limit_ms):
    ws = _ws()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    ssa.ssa_selftest_wait_timeout(limit_ms * 1_000_000, ws)
    b.record()
    torch.cuda.synchronize()
    assert a.elapsed_time(b) >= 0.95 * limit_ms
    assert ssa.ssa_workspace_error(ws) == ssa.SSA_DEVERR_WAIT_TIMEOUT
    assert ssa.ssa_workspace_error(ws) == 0            # the read cleared it
    # the same context runs a decode step of the real path, error-free
    w = W.DECODE_1M.with_(name="after_timeout", L=1 << 16, q_pos0=(1 << 16) - 1, n_q=1)
    inp = W.Inputs(w)
    dev = torch.device("cuda")
    K, V, Q = inp.k(dev), inp.v(dev), inp.q(dev)
    p = ssa.params(w.B, w.Hq, w.Hkv, w.d, w.L, w.S, w.topk, w.dtype)
    summ = torch.zeros((w.B, w.Hkv, w.n_spans, w.d), dtype=torch.float32, device=dev)
    ssa.ssa_build_summaries(p, K, 0, w.n_spans, summ)
    wsd = ssa.workspace(p, 1, ssa.SSA_OP_DECODE, dev)
    sel = torch.empty((w.B, w.Hq, 1, w.topk), dtype=torch.int32, device=dev)
    O = torch.empty((w.B, w.Hq, w.d), dtype=w.dtype, device=dev)
    ssa.ssa_decode_step(p, Q[0].contiguous(), w.q_pos0, summ, K, V, sel, O, None, wsd)
    assert ssa.ssa_workspace_error(wsd) == 0
    assert bool(torch.isfinite(O.float()).all())
    s = sel.cpu().numpy()
    assert ((s >= 0) & (s < w.q_pos0 // w.S)).all()
