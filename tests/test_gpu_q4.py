"""The 4-bit cache against the oracle.

* ssa_quantize_kv4: codes and scales bit for bit equal to the oracle's
  4-bit fp32 quantiser; the K and V word layouts are unpacked here from
  their definition in the public header, and tokens outside the quantised
  range keep their old codes (V words gather eight tokens).
* ssa_build_summaries_q4: the mean of the dequantised keys.
* decode over the 4-bit cache: selections equal the oracle's on the
  dequantised cache (margin-checked inputs), outputs within the 16-bit
  tolerance of the oracle's exact attention over the dequantised K / V,
  and the one-call step gives the two calls' bits.

SubQ release post (geeks.co.kr/post/2077), quantisation plan: 4-bit K / V
with the summaries kept in fp32.
"""
import numpy as np
import pytest
import torch

import content_routed_sparse_build_b300 as ssa
import oracle
from synth import workloads as W

from harness import LSE_TOL, MARGIN, TOL, max_abs

pytestmark = pytest.mark.gpu

D = 128


def _shift(e):
    return 4 * (e // 2) + 16 * (e % 2)


def unpack_kq4(Kq4: torch.Tensor) -> np.ndarray:
    """[B, Hkv, L_cap / 32, 512] words -> codes [B, Hkv, L_cap, 128]: word
    [J][tok][c] holds token tok's dimensions 32 J + 8 c + e at bits
    4 (e / 2) + 16 (e % 2), each as code + 8."""
    w = Kq4.cpu().numpy().view(np.uint32)
    B, H, T, _ = w.shape
    w = w.reshape(B, H, T, 4, 32, 4)                   # [J][tok][c]
    out = np.zeros((B, H, T, 32, D), np.int8)
    for J in range(4):
        for c in range(4):
            for e in range(8):
                out[:, :, :, :, 32 * J + 8 * c + e] = ((w[:, :, :, J, :, c] >> _shift(e)) & 0xF).astype(np.int8) - 8
    return out.reshape(B, H, T * 32, D)


def unpack_vq4(Vq4: torch.Tensor) -> np.ndarray:
    """[B, Hkv, L_cap / 32, 512] words -> codes [B, Hkv, L_cap, 128]: word
    [d][c] holds dimension d of tokens 2 c + (0, 1, 8, 9, 16, 17, 24, 25)[e]."""
    w = Vq4.cpu().numpy().view(np.uint32)
    B, H, T, _ = w.shape
    w = w.reshape(B, H, T, D, 4)
    out = np.zeros((B, H, T, 32, D), np.int8)
    f = (0, 1, 8, 9, 16, 17, 24, 25)
    seen = set()
    for c in range(4):
        for e in range(8):
            tok = 2 * c + f[e]
            seen.add(tok)
            out[:, :, :, tok, :] = ((w[:, :, :, :, c] >> _shift(e)) & 0xF).astype(np.int8) - 8
    assert seen == set(range(32))
    return out.reshape(B, H, T * 32, D)


QCASES = [
    ("bf16", 1, 2, 320, 5, 300, torch.bfloat16),
    ("f16_b2", 2, 1, 96, 0, 96, torch.float16),
    ("f32_two_rows", 1, 3, 64, 31, 33, torch.float32),
]


@pytest.mark.parametrize("name,B,Hkv,L,t0,t1,dt", QCASES, ids=[c[0] for c in QCASES])
def test_quantize4_matches_oracle_bit_for_bit(name, B, Hkv, L, t0, t1, dt):
    g = torch.Generator().manual_seed(17)
    K = (torch.randn((B, Hkv, L, D), generator=g) * 3).to(dt)
    V = (torch.randn((B, Hkv, L, D), generator=g) * 0.7).to(dt)
    K[0, 0, t0] = 0                                   # an all-zero row: scale 0, codes 0
    if t1 - t0 > 1:
        K[0, 0, t0 + 1, :4] = torch.tensor([7.0, 0.5, 1.5, -2.5]).to(dt)   # ties to even
        K[0, 0, t0 + 1, 4:] = 0
    p = ssa.params(B, 8 * Hkv, Hkv, D, L, 64, 4, dt)
    Kq4, Ks, Vq4, Vs = ssa.q4_cache(p)
    for t in (Kq4, Vq4):
        t.fill_(-1)                                   # every field 0xF: code 7
    for t in (Ks, Vs):
        t.fill_(-1.0)
    ssa.ssa_quantize_kv4(p, K.cuda(), V.cuda(), t0, t1, Kq4, Ks, Vq4, Vs)
    torch.cuda.synchronize()
    qk, sk = oracle.quantize_rows4(K[:, :, t0:t1].contiguous())
    qv, sv = oracle.quantize_rows4(V[:, :, t0:t1].contiguous())
    Kq_h, Vq_h = unpack_kq4(Kq4), unpack_vq4(Vq4)
    Ks_h, Vs_h = Ks.cpu().numpy(), Vs.cpu().numpy()
    assert np.array_equal(Kq_h[:, :, t0:t1], qk)
    assert np.array_equal(Vq_h[:, :, t0:t1], qv)
    assert np.array_equal(Ks_h[:, :, t0:t1].view(np.uint32), sk.view(np.uint32))
    assert np.array_equal(Vs_h[:, :, t0:t1].view(np.uint32), sv.view(np.uint32))
    for a in (Kq_h, Vq_h):
        assert (a[:, :, :t0] == 7).all() and (a[:, :, t1:] == 7).all()
    for a in (Ks_h, Vs_h):
        assert (a[:, :, :t0] == -1).all() and (a[:, :, t1:] == -1).all()
    if t1 - t0 > 1:
        assert Kq_h[0, 0, t0].tolist() == [0] * D and Ks_h[0, 0, t0] == 0
        assert Kq_h[0, 0, t0 + 1, :4].tolist() == [7, 0, 2, -2]


def test_summaries_q4_are_means_of_the_dequantised_keys():
    B, Hkv, L, S = 1, 2, 1000 + 24, 100
    g = torch.Generator().manual_seed(18)
    K = torch.randn((B, Hkv, L, D), generator=g).to(torch.bfloat16)
    p = ssa.params(B, 8, Hkv, D, 1000, S, 4, torch.bfloat16, L_cap=L)
    Kq4, Ks, Vq4, Vs = ssa.q4_cache(p)
    ssa.ssa_quantize_kv4(p, K.cuda(), K.cuda(), 0, 1000, Kq4, Ks, Vq4, Vs)
    ns_cap = (L + S - 1) // S
    summ = torch.full((B, Hkv, ns_cap, D), float("nan"), dtype=torch.float32, device="cuda")
    ssa.ssa_build_summaries_q4(p, Kq4, Ks, 0, 10, summ)
    q, s = oracle.quantize_rows4(K.contiguous())
    ref = oracle.summaries(oracle.dequantize_rows(q, s), 1000, S, 0, 10)
    got = summ.cpu().double().numpy()
    assert np.isnan(got[:, :, 10:]).all()
    err = np.abs(got[:, :, :10] - ref[:, :, :10]).max()
    assert err <= 2e-5, err


DCASES = [
    W.Workload("q4_bf16_gqa8", "decode", 1, 32, 4, 128, 65536 + 100, 1024, 16, torch.bfloat16,
               n_q=2, q_pos0=65536 + 98, chunk=1, needles=4, seed=91),
    W.Workload("q4_f16_s300_b2", "decode", 2, 16, 2, 128, 20000 + 32, 300, 8, torch.float16,
               n_q=2, q_pos0=19990, chunk=1, needles=2, seed=92),
    W.Workload("q4_bf16_g16", "decode", 1, 32, 2, 128, 8192, 100, 12, torch.bfloat16,
               n_q=2, q_pos0=8000, chunk=1, seed=93),
    # k above 32: the router's 64-entry lists, up to 65 spans per row
    W.Workload("q4_bf16_k64", "decode", 1, 16, 2, 128, 300 * 256 + 50, 256, 64, torch.bfloat16,
               n_q=2, q_pos0=300 * 256 + 47, chunk=1, needles=4, seed=94),
]


@pytest.mark.parametrize("w", DCASES, ids=lambda w: w.name)
def test_decode_q4_matches_oracle_on_the_dequantised_cache(w):
    n_rows = int(np.prod(w.q_shape[:-1]))
    attempt = torch.zeros(n_rows, dtype=torch.int32)
    inp = W.Inputs(w, attempt=attempt)
    K, V = inp.k(), inp.v()
    qk, sk = oracle.quantize_rows4(K)
    qv, sv = oracle.quantize_rows4(V)
    Kdq, Vdq = oracle.dequantize_rows(qk, sk), oracle.dequantize_rows(qv, sv)
    summ_o = oracle.summaries(Kdq, w.L, w.S)
    Q = inp.q()
    for _ in range(32):
        margins = []
        for s in range(w.n_q):
            _, m = oracle.route(Q[s].reshape(w.B, w.Hq, 1, w.d).contiguous(), w.q_pos0 + s, summ_o,
                                w.Hkv, w.S, w.topk)
            margins.append(m)
        bad = np.nonzero(np.stack(margins).reshape(-1) < MARGIN)[0]
        if len(bad) == 0:
            break
        attempt[bad] += 1
        Q = inp.q()
    else:
        raise RuntimeError("margins not reached")
    L_cap = (w.L + 31) // 32 * 32
    Kd = torch.zeros((w.B, w.Hkv, L_cap, w.d), dtype=w.dtype, device="cuda")
    Vd = torch.zeros_like(Kd)
    Kd[:, :, :w.L] = K.cuda()
    Vd[:, :, :w.L] = V.cuda()
    p_full = ssa.params(w.B, w.Hq, w.Hkv, w.d, w.L, w.S, w.topk, w.dtype, L_cap=L_cap)
    Kq4, Ks, Vq4, Vs = ssa.q4_cache(p_full)
    Ks.fill_(float("nan"))                         # rows past L: masked, never read as numbers
    Vs.fill_(float("nan"))
    ssa.ssa_quantize_kv4(p_full, Kd, Vd, 0, w.L, Kq4, Ks, Vq4, Vs)
    ns_cap = (L_cap + w.S - 1) // w.S
    summ = torch.zeros((w.B, w.Hkv, ns_cap, w.d), dtype=torch.float32, device="cuda")
    ws = ssa.workspace(p_full, 1, ssa.SSA_OP_DECODE)
    Qd = Q.cuda()
    for s in range(w.n_q):
        pos = w.q_pos0 + s
        p = ssa.params(w.B, w.Hq, w.Hkv, w.d, pos + 1, w.S, w.topk, w.dtype, L_cap=L_cap)
        ssa.ssa_build_summaries_q4(p, Kq4, Ks, 0, pos // w.S, summ)
        q = Qd[s].contiguous()
        sel = torch.empty((w.B, w.Hq, 1, w.topk), dtype=torch.int32, device="cuda")
        O = torch.empty((w.B, w.Hq, w.d), dtype=w.dtype, device="cuda")
        lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device="cuda")
        ssa.ssa_route(p, q, 1, pos, summ, sel)
        ssa.ssa_attend_decode_q4(p, q, pos, Kq4, Ks, Vq4, Vs, sel, O, lse, ws)
        sel2, O2, lse2 = torch.empty_like(sel), torch.empty_like(O), torch.empty_like(lse)
        ssa.ssa_decode_step_q4(p, q, pos, summ, Kq4, Ks, Vq4, Vs, sel2, O2, lse2, ws)
        assert torch.equal(sel2, sel) and torch.equal(O2, O) and torch.equal(lse2, lse), pos
        qh = Q[s].reshape(w.B, w.Hq, 1, w.d).contiguous()
        sel_o, _ = oracle.route(qh, pos, summ_o, w.Hkv, w.S, w.topk)
        assert np.array_equal(sel.reshape(-1, w.topk).cpu().numpy(), sel_o), pos
        O_o, lse_o, _ = oracle.attend(qh.double(), Kdq, Vdq, pos, w.S, sel_o)
        assert max_abs(O.reshape(-1, w.d).cpu(), O_o) <= TOL[w.dtype]
        assert max_abs(lse.reshape(-1).cpu(), lse_o) <= LSE_TOL[w.dtype]
    assert ssa.ssa_workspace_error(ws) == 0


def test_q4_entry_points_reject_what_they_do_not_take():
    t = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    w32 = torch.zeros(64, dtype=torch.int32, device="cuda")
    f = torch.zeros(64, dtype=torch.float32, device="cuda")
    sel = torch.zeros(64, dtype=torch.int32, device="cuda")
    p = ssa.params(1, 8, 2, 128, 100, 64, 4, torch.bfloat16, L_cap=100)     # L_cap not a multiple of 32
    p64 = ssa.params(1, 8, 2, 64, 128, 64, 4, torch.bfloat16)               # d = 64
    for pp in (p, p64):
        for call in (lambda: ssa.ssa_quantize_kv4(pp, t, t, 0, 10, w32, f, w32, f),
                     lambda: ssa.ssa_build_summaries_q4(pp, w32, f, 0, 1, f),
                     lambda: ssa.ssa_attend_decode_q4(pp, t, 5, w32, f, w32, f, sel, t, None, None),
                     lambda: ssa.ssa_decode_step_q4(pp, t, 5, f, w32, f, w32, f, sel, t, None, None)):
            with pytest.raises(ssa.SSAError) as e:
                call()
            assert e.value.status == ssa.SSA_ERR_UNSUPPORTED
    p = ssa.params(1, 8, 2, 128, 128, 64, 4, torch.bfloat16)
    with pytest.raises(ssa.SSAError) as e:
        ssa.ssa_quantize_kv4(p, t, t, 0, 129, w32, f, w32, f)               # t_end > L
    assert e.value.status == ssa.SSA_ERR_INVALID_ARG


def test_decode_q4_1m_sampled_steps():
    """The 4-bit decode at the full 1M size, in the launch configuration the
    benchmark times: eight of the 256 steps, every head, the one-call step."""
    w = W.DECODE_1M
    steps = list(range(0, w.n_q, 32))
    n_rows = int(np.prod(w.q_shape[:-1]))
    attempt = torch.zeros(n_rows, dtype=torch.int32)
    inp = W.Inputs(w, attempt=attempt)
    dev = torch.device("cuda")
    Kd, Vd = inp.k(dev), inp.v(dev)
    p = ssa.params(w.B, w.Hq, w.Hkv, w.d, w.L, w.S, w.topk, w.dtype)
    Kq4, Ks, Vq4, Vs = ssa.q4_cache(p)
    ssa.ssa_quantize_kv4(p, Kd, Vd, 0, w.L, Kq4, Ks, Vq4, Vs)
    summ = torch.zeros((w.B, w.Hkv, w.n_spans, w.d), dtype=torch.float32, device=dev)
    ssa.ssa_build_summaries_q4(p, Kq4, Ks, 0, w.n_spans, summ)
    del Kd, Vd
    Kdq = torch.from_numpy(unpack_kq4(Kq4).astype(np.float32) * Ks.cpu().numpy()[..., None])
    Vdq = torch.from_numpy(unpack_vq4(Vq4).astype(np.float32) * Vs.cpu().numpy()[..., None])
    summ_o = oracle.summaries(Kdq, w.L, w.S)
    Q = inp.q()
    for _ in range(32):
        margins = [oracle.route(Q[s].reshape(w.B, w.Hq, 1, w.d).contiguous(), w.q_pos0 + s, summ_o,
                                w.Hkv, w.S, w.topk)[1] for s in steps]
        bad_rows = []
        for s, m in zip(steps, margins):
            for r in np.nonzero(m < MARGIN)[0]:
                bad_rows.append(s * w.B * w.Hq + int(r))
        if not bad_rows:
            break
        attempt[np.array(bad_rows)] += 1
        Q = inp.q()
    else:
        raise RuntimeError("margins not reached")
    ws = ssa.workspace(p, 1, ssa.SSA_OP_DECODE)
    Qd = Q.cuda()
    for s in steps:
        pos = w.q_pos0 + s
        q = Qd[s].contiguous()
        sel = torch.empty((w.B, w.Hq, 1, w.topk), dtype=torch.int32, device=dev)
        O = torch.empty((w.B, w.Hq, w.d), dtype=w.dtype, device=dev)
        lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=dev)
        ssa.ssa_decode_step_q4(p, q, pos, summ, Kq4, Ks, Vq4, Vs, sel, O, lse, ws)
        qh = Q[s].reshape(w.B, w.Hq, 1, w.d).contiguous()
        sel_o, _ = oracle.route(qh, pos, summ_o, w.Hkv, w.S, w.topk)
        assert np.array_equal(sel.reshape(-1, w.topk).cpu().numpy(), sel_o), pos
        O_o, lse_o, _ = oracle.attend(qh.float(), Kdq, Vdq, pos, w.S, sel_o)
        assert max_abs(O.reshape(-1, w.d).cpu(), O_o) <= TOL[w.dtype]
        assert max_abs(lse.reshape(-1).cpu(), lse_o) <= LSE_TOL[w.dtype]
    assert ssa.ssa_workspace_error(ws) == 0
