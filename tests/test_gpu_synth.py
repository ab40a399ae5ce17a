"""The seeded input generator on the device against the same generator on the
host: bit for bit, on ranges of the full-size workloads that cover the
structure added to the keys (needle spans, the per-span low-rank term, the
partial last span) and on plain ranges.  The full-size parity tests rely on
this when they read the oracle's rows of a cache too large for the host
from the device copy of the same generated cache."""
import numpy as np
import pytest
import torch

from synth import workloads as W

pytestmark = pytest.mark.gpu


def _ranges(w, inp, rng):
    out = [(0, 0, 3 * w.S), (w.B * w.Hkv - 1, w.L - 700, w.L)]
    if inp.needle_spans is not None:
        for bh in range(w.B * w.Hkv):
            j = int(inp.needle_spans[bh][rng.integers(len(inp.needle_spans[bh]))])
            out.append((bh, j * w.S, (j + 1) * w.S))
    for _ in range(4):
        bh = int(rng.integers(w.B * w.Hkv))
        t0 = int(rng.integers(w.L - 5000))
        out.append((bh, t0, t0 + 4999))
    return out


@pytest.mark.parametrize("w", [W.DECODE_10M, W.PREFILL_128K, W.DECODE_1M], ids=lambda w: w.name)
def test_device_cache_equals_host_generator(w):
    inp = W.Inputs(w)
    dev = torch.device("cuda")
    rng = np.random.default_rng(3)
    for which, fill in (("k", inp.k), ("v", inp.v)):
        X = fill(dev)
        for bh, t0, t1 in _ranges(w, inp, rng):
            b, h = divmod(bh, w.Hkv)
            got = X[b, h, t0:t1].cpu()
            ref = inp.kv_rows(which, bh, t0, t1)
            assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), (which, bh, t0, t1)
        del X
        torch.cuda.empty_cache()
    Qd = inp.q(dev).cpu()
    assert torch.equal(Qd.view(torch.int16), inp.q().view(torch.int16))
