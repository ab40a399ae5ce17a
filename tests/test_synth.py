"""The seeded input generator: Philox known answers, rounding, statistics."""
import numpy as np
import pytest
import torch

import synth
from synth import workloads as W


# Known-answer vectors of Philox4x32-10 published with the generator
# (Salmon et al., SC'11, Random123 distribution): (counter, key) -> output.
KAT = [
    ([0, 0, 0, 0], [0, 0], [0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]),
    ([0xFFFFFFFF] * 4, [0xFFFFFFFF] * 2, [0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD]),
    ([0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344], [0xA4093822, 0x299F31D0],
     [0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1]),
]


@pytest.mark.parametrize("ctr,key,expect", KAT)
def test_philox_known_answers(ctr, key, expect):
    assert list(synth.philox_block(ctr, key)) == expect


def _edge_floats():
    rng = np.random.default_rng(0)
    vals = [0.0, -0.0, 1.0, -1.0, 65504.0, 65519.0, 65520.0, 1e-8, 2.0 ** -24, 2.0 ** -25,
            3 * 2.0 ** -26, 2.0 ** -14, 2.0 ** -14 * 0.999, 6.1e-5, 1.00048828125, 1.0009765625]
    x = np.concatenate([np.array(vals, np.float32), rng.standard_normal(20000).astype(np.float32) * 3,
                        (rng.standard_normal(5000) * 1e-5).astype(np.float32),
                        np.ldexp(rng.random(5000), rng.integers(-30, 16, 5000)).astype(np.float32)])
    return np.concatenate([x, -x])


def test_f16_rounding_matches_numpy():
    x = _edge_floats()
    got = synth.round_f32(x, torch.float16)
    ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_rounding_matches_torch():
    x = _edge_floats()
    got = synth.round_f32(x, torch.bfloat16)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


def test_values_are_unit_normal_like():
    x = synth.normal((1 << 20,), torch.float32, 7, 2).double().numpy()
    assert abs(x.mean()) < 5e-3
    assert abs(x.var() - 1.0) < 5e-3
    assert np.abs(x).max() <= 4.9
    # Irwin-Hall(8) fourth moment: 3 - 1.2 / 8 = 2.85 (normal: 3)
    assert abs((x ** 4).mean() - 2.85) < 0.05


def test_subrange_and_dtypes_consistent():
    full = synth.normal((3, 5, 64), torch.float32, 11, 3)
    part = torch.empty(2 * 64, dtype=torch.float32)
    synth.fill_(part, 11, 3, e0=7 * 64, d=64)
    assert torch.equal(part, full.reshape(-1)[7 * 64: 9 * 64])
    bf = synth.normal((3, 5, 64), torch.bfloat16, 11, 3)
    assert torch.equal(bf, full.to(torch.bfloat16))
    hf = synth.normal((3, 5, 64), torch.float16, 11, 3)
    assert torch.equal(hf, full.to(torch.float16))


def test_attempt_redraws_only_that_row():
    att = torch.zeros(15, dtype=torch.int32)
    att[4] = 3
    a = synth.normal((15, 64), torch.float32, 5, 1)
    b = synth.normal((15, 64), torch.float32, 5, 1, attempt=att)
    same = (a == b).all(dim=1)
    assert not same[4] and same[torch.arange(15) != 4].all()


def test_bias_is_one_fp32_add_per_element():
    L, S, d = 40, 8, 16
    bias = torch.from_numpy(np.random.default_rng(1).standard_normal((2, 5, d)).astype(np.float32))
    base = synth.normal((2, L, d), torch.float32, 9, 2)
    k = synth.normal((2, L, d), torch.float32, 9, 2, bias=bias, rows_per_head=L, S=S)
    expect = base + bias.repeat_interleave(S, dim=1)
    assert torch.equal(k, expect)


def test_needle_structure():
    w = W.TINY_PREFILL
    inp = W.Inputs(w)
    assert inp.needle_spans.shape == (w.B * w.Hkv, w.needles)
    assert (inp.needle_spans < w.last_pos // w.S).all()
    assert np.allclose(np.linalg.norm(inp.u, axis=1), 1.0)
    nz = (inp.bias.abs().sum(-1) > 0).numpy()
    for bh in range(w.B * w.Hkv):
        assert set(np.nonzero(nz[bh])[0]) == set(inp.needle_spans[bh])


def test_lowrank_structure_is_constant_per_span():
    w = W.PREFILL_128K.with_(L=2048, n_q=2048, chunk=1024, Hq=8, Hkv=2)
    inp = W.Inputs(w)
    assert inp.bias.shape == (w.Hkv, w.n_spans, w.d)
    assert inp.bias.std().item() > 0.5
