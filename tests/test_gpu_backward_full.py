"""Backward parity at full training size (the bench's `train` workload: T=4096,
d=4096, f=14336, E=8, top-2, bf16), in the launch configuration the bench
times, on outputs the float64 oracle can compute exactly on a sample:

* weight gradients of sampled intermediate columns J: each expert's SwiGLU is
  a sum over its f columns (H[:, i] depends on column i of W1 and W3 only,
  and reaches y through row i of W2), so the gradients of W1[:, :, J],
  W3[:, :, J] and W2[:, J, :] are those of the layer restricted to the
  columns J, whose routing is the full layer's (the router does not see the
  experts).  The oracle runs that restricted layer on all 4096 tokens.
* dx on sampled tokens: a token's input gradient depends only on its own
  routing, experts and dy row, so the oracle runs the full experts on those
  tokens alone.

Tolerances as in test_gpu_backward.py (normwise 1e-2, max-abs relative to
the largest reference entry 3e-2)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

T, D, F, E, K = 4096, 4096, 14336, 8, 2
COLS = [0, 1, 777, 5000, 9001, 14335]
TOKENS = [0, 1, 1234, 4095]


@pytest.fixture(scope="module")
def run(cuda_device):
    from sparse_mixture_experts_55_b300 import build
    build.build()
    import sparse_mixture_experts_55_b300 as moe
    inp = W.prefill(T=T, device=cuda_device)
    dy = W.randn((T, D), 1.0, W.BASE_SEED + 77, cuda_device, torch.bfloat16)
    ws = moe.TrainWorkspace(T, D, F, E, K, torch.bfloat16, cuda_device)
    moe.moe_forward_train(inp.x, inp.Wg, inp.W1, inp.W3, inp.W2, K, ws)
    g = moe.moe_backward(inp.x, inp.Wg, inp.W1, inp.W3, inp.W2, dy, K, ws)
    torch.cuda.synchronize()
    assert moe.moe_read_status(ws) == 0
    return inp, dy, g


def _err(gpu, ref):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    return (float(np.linalg.norm(gpu - ref) / np.linalg.norm(ref)),
            float(np.abs(gpu - ref).max() / np.abs(ref).max()))


def test_weight_gradients_on_sampled_columns(run):
    inp, dy, g = run
    cols = torch.tensor(COLS)
    x = inp.x.cpu()
    Wg = inp.Wg.cpu()
    # every token's selection is decided far from a tie (fp32 and fp64 routing agree)
    gap, _ = oracle.logit_gaps(oracle.router_logits(oracle.f64(x), oracle.f64(Wg)), K)
    assert gap.min() > 1e-5, gap.min()
    W1 = inp.W1[:, :, cols.to(inp.W1.device)].cpu()
    W3 = inp.W3[:, :, cols.to(inp.W3.device)].cpu()
    W2 = inp.W2[:, cols.to(inp.W2.device), :].cpu()
    ref = oracle.moe_layer_backward(x, Wg, W1, W3, W2, K, dy.cpu())
    c = cols.to(g.dW1.device)
    for name, gpu, r in (("dW1", g.dW1[:, :, c], ref.dW1), ("dW3", g.dW3[:, :, c], ref.dW3),
                         ("dW2", g.dW2[:, c, :], ref.dW2)):
        nrm, linf = _err(gpu.cpu().numpy(), r)
        print(f"\n{name} on columns {COLS}: normwise {nrm:.2e}, max {linf:.2e}")
        assert nrm <= 1e-2 and linf <= 3e-2, (name, nrm, linf)


def test_input_gradient_on_sampled_tokens(run):
    inp, dy, g = run
    t = torch.tensor(TOKENS)
    ref = oracle.moe_layer_backward(inp.x.cpu()[t], inp.Wg.cpu(), inp.W1.cpu(), inp.W3.cpu(), inp.W2.cpu(), K,
                                    dy.cpu()[t])
    nrm, linf = _err(g.dx.cpu()[t].numpy(), ref.dx)
    print(f"\ndx on tokens {TOKENS}: normwise {nrm:.2e}, max {linf:.2e}")
    assert nrm <= 1e-2 and linf <= 3e-2, (nrm, linf)
