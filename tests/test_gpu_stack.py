"""The 32-layer attention-free MoE stack at full size: T = 8192 tokens,
h0 ~ N(0,1), h <- h + MoE_l(RMSNorm(h)) for l = 0..31, each layer with its own
seeded Mixtral-shaped weights (90 GB resident in HBM).  Every layer is checked
against the oracle on a 256-token sample of the GPU's own input to that layer
(routing on every token); the run is the launch sequence bench.py times."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as W
from tests.stack_check import check_stack_layer

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

T, LAYERS, SAMPLE = 8192, 32, 256


def test_stack32_per_layer(cuda_device):
    from sparse_mixture_experts_55_b300 import build
    build.build()
    import sparse_mixture_experts_55_b300 as moe
    d, f, E, K = W.MIXTRAL["d"], W.MIXTRAL["f"], W.MIXTRAL["E"], W.MIXTRAL["K"]
    layers = [W.stack_layer_weights(l, d, f, E, device=cuda_device) for l in range(LAYERS)]
    h = W.stack_h0(T, d, device=cuda_device)
    ws = moe.Workspace(T, d, f, E, K, torch.bfloat16, cuda_device)
    toks = np.sort(np.random.default_rng(4321).choice(T, size=SAMPLE, replace=False))
    worst_y = worst_h = 0.0
    for l in range(LAYERS):
        err_y, err_h, rep = check_stack_layer(moe, h, layers[l], K, toks, ws, "bf16")
        worst_y, worst_h = max(worst_y, err_y), max(worst_h, err_h)
        print(f"layer {l:2d}: rel err y {err_y:.2e}, residual {err_h:.2e}, near-ties {rep.n_exempt_in_out}")
    print(f"stack32: worst rel err y {worst_y:.2e}, residual {worst_h:.2e}; |h|max {h.abs().max().item():.2f}")
    assert torch.isfinite(h.float()).all()
