"""The decode locality trace reproduces the statistic it stands in for: the
pages' Table 5 discussion reports that consecutive tokens share their first or
second expert 61.6-67.0% of the time at layer 15, against ~46% for
independent top-2 choices among 8 experts (1 - C(6,2)/C(8,2) = 46.4%).  The
router (the float64 oracle's) picks the chain's steered pair."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads as W


def _shares(idx):
    return float(np.mean([len(set(idx[i]) & set(idx[i - 1])) > 0 for i in range(1, len(idx))]))


def test_locality_trace_matches_table5_and_chance():
    d, E = 1024, 8
    Wg = W.randn((d, E), d ** -0.5, W._seed(W.BASE_SEED, "Wg"), "cpu", torch.bfloat16)
    x, pairs = W.decode_trace(400, Wg, T=1)
    g = oracle.gating(x[:, 0], Wg, 2)
    assert 0.60 <= _shares(g.idx) <= 0.72                     # Table 5: 61.6-67.0%
    agree = np.mean([set(g.idx[i]) == set(pairs[i, 0].tolist()) for i in range(400)])
    assert agree >= 0.95
    x0, _ = W.decode_trace(400, Wg, T=1, keep=0.0)
    g0 = oracle.gating(x0[:, 0], Wg, 2)
    assert 0.38 <= _shares(g0.idx) <= 0.54                    # independent choices: 46.4%


def test_trace_is_seeded_and_batched():
    d, E = 256, 8
    Wg = W.randn((d, E), d ** -0.5, 7, "cpu", torch.bfloat16)
    a, pa = W.decode_trace(10, Wg, T=3, seed=5)
    b, pb = W.decode_trace(10, Wg, T=3, seed=5)
    assert a.shape == (10, 3, d) and a.dtype == torch.bfloat16
    assert torch.equal(a, b) and torch.equal(pa, pb)
    # rows are RMS-normalised
    rms = a.float().pow(2).mean(dim=-1).sqrt()
    assert torch.allclose(rms, torch.ones_like(rms), atol=1e-2)
