"""Cache snapshots on the GPU: ssa_snapshot_save writes exactly the bytes
the oracle's writer produces from the same rows, ssa_snapshot_load restores
them bit for bit (and nothing else), and a session restored from the file
routes and attends exactly as the saved one.

Superlinear release post (geeks.co.kr/post/2077), "why this matters": keep
the cache, save / restore a session on disk."""
import numpy as np
import pytest
import torch

import content_routed_sparse_build_b300 as ssa
from oracle import snapshot as osnap
from synth import workloads as W

pytestmark = pytest.mark.gpu

CASES = [
    # name, workload, saved rows, staging bytes (None: the binding's 64 MiB)
    ("bf16_d128_small_staging", W.Workload("snap_bf16", "decode", 1, 16, 2, 128, 6000, 256, 8, torch.bfloat16,
                                           n_q=1, q_pos0=3999, chunk=1, needles=2, seed=71), 4000, 96 << 10),
    ("f16_d64_b2", W.Workload("snap_f16", "decode", 2, 8, 4, 64, 3000, 100, 4, torch.float16,
                              n_q=1, q_pos0=2499, chunk=1, seed=72), 2500, None),
    ("f32_d64", W.Workload("snap_f32", "decode", 1, 4, 2, 64, 2000, 64, 4, torch.float32,
                           n_q=1, q_pos0=1279, chunk=1, seed=73), 1280, 1 << 20),
]


def _words(t):
    """Raw element words of a tensor as a host numpy array."""
    w = torch.int16 if t.element_size() == 2 else torch.int32
    a = t.cpu().contiguous().view(w).numpy()
    return a.view(np.uint16 if t.element_size() == 2 else np.uint32)


@pytest.mark.parametrize("name,w,n_tok,staging_bytes", CASES, ids=[c[0] for c in CASES])
def test_snapshot_round_trip_and_restored_session(tmp_path, name, w, n_tok, staging_bytes):
    dev = torch.device("cuda")
    inp = W.Inputs(w)
    K, V = inp.k(dev), inp.v(dev)                      # [B, Hkv, L_cap, d], rows beyond n_tok are data too
    p = ssa.params(w.B, w.Hq, w.Hkv, w.d, n_tok, w.S, w.topk, w.dtype, L_cap=w.L)
    ns_cap = (w.L + w.S - 1) // w.S
    summ = torch.full((w.B, w.Hkv, ns_cap, w.d), float("nan"), dtype=torch.float32, device=dev)
    n_summ = n_tok // w.S
    ssa.ssa_build_summaries(p, K, 0, n_summ, summ)
    staging = None if staging_bytes is None else torch.empty(staging_bytes, dtype=torch.uint8, pin_memory=True)
    path = str(tmp_path / (name + ".ssakv"))
    ssa.ssa_snapshot_save(p, n_tok, K, V, summ, path, staging=staging)

    # the file is the oracle's encoding of the same rows
    want = osnap.encode(ssa.DTYPE_CODE[w.dtype], w.S, _words(K[:, :, :n_tok]), _words(V[:, :, :n_tok]),
                        summ[:, :, :n_summ].cpu().numpy())
    got = open(path, "rb").read()
    assert len(got) == len(want)
    assert got == want
    h = ssa.ssa_snapshot_read_header(path)
    assert (h.n_tokens, h.n_summ) == (n_tok, n_summ)

    # restore into fresh buffers: the saved rows come back bit for bit, the rest is untouched
    K2 = torch.full_like(K, 7.0)
    V2 = torch.full_like(V, -3.0)
    summ2 = torch.full_like(summ, 11.0)
    n = ssa.ssa_snapshot_load(p, path, K2, V2, summ2, staging=staging)
    torch.cuda.synchronize()
    assert n == n_tok
    assert torch.equal(_t(K2[:, :, :n_tok]), _t(K[:, :, :n_tok]))
    assert torch.equal(_t(V2[:, :, :n_tok]), _t(V[:, :, :n_tok]))
    assert bool((K2[:, :, n_tok:] == 7.0).all()) and bool((V2[:, :, n_tok:] == -3.0).all())
    assert torch.equal(summ2[:, :, :n_summ], summ[:, :, :n_summ])
    assert bool((summ2[:, :, n_summ:] == 11.0).all())

    # the restored session decodes the next token exactly as the saved one
    pos = n_tok - 1
    p_dec = ssa.params(w.B, w.Hq, w.Hkv, w.d, n_tok, w.S, w.topk, w.dtype, L_cap=w.L)
    q = inp.q(dev)[0].contiguous()
    outs = []
    for KK, VV, ss in ((K, V, summ), (K2, V2, summ2)):
        sel = torch.empty((w.B, w.Hq, 1, w.topk), dtype=torch.int32, device=dev)
        O = torch.empty((w.B, w.Hq, w.d), dtype=w.dtype, device=dev)
        lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=dev)
        ws = ssa.workspace(p_dec, 1, ssa.SSA_OP_DECODE)
        ssa.ssa_route(p_dec, q, 1, pos, ss, sel)
        ssa.ssa_attend_decode(p_dec, q, pos, KK, VV, sel, O, lse, ws)
        assert ssa.ssa_workspace_error(ws) == 0
        outs.append((sel, O, lse))
    assert torch.equal(outs[0][0], outs[1][0])
    assert torch.equal(_t(outs[0][1]), _t(outs[1][1]))
    assert torch.equal(outs[0][2], outs[1][2])


def _t(x):
    """Bit view, so that NaN payloads and signed zeros compare exactly."""
    return x.contiguous().view(torch.int16 if x.element_size() == 2 else torch.int32)


def test_snapshot_load_refuses_a_file_of_other_parameters(tmp_path):
    w = CASES[1][1]
    dev = torch.device("cuda")
    K = torch.zeros((w.B, w.Hkv, w.L, w.d), dtype=w.dtype, device=dev)
    summ = torch.zeros((w.B, w.Hkv, (w.L + w.S - 1) // w.S, w.d), dtype=torch.float32, device=dev)
    p = ssa.params(w.B, w.Hq, w.Hkv, w.d, 500, w.S, w.topk, w.dtype, L_cap=w.L)
    path = str(tmp_path / "a.ssakv")
    ssa.ssa_snapshot_save(p, 500, K, K, summ, path)
    other = ssa.params(w.B, w.Hq, w.Hkv, w.d, 500, w.S + 1, w.topk, w.dtype, L_cap=w.L)
    K2 = torch.full_like(K, 1.0)
    with pytest.raises(ssa.SSAError) as e:
        ssa.ssa_snapshot_load(other, path, K2, K2, summ)
    assert e.value.status == ssa.SSA_ERR_IO
    torch.cuda.synchronize()
    assert bool((K2 == 1.0).all())                     # nothing was written
