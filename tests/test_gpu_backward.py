"""GPU parity of the training path (moe_forward_train + moe_backward, bf16
layer, fp32 gradients) against the float64 oracle's chain-rule gradients
(oracle.moe_layer_backward, itself pinned by finite differences).

Tolerance: every gradient G is compared normwise,
    ||G_gpu - G_ref||_F / ||G_ref||_F <= 1e-2,
and elementwise against the largest reference magnitude,
    max |G_gpu - G_ref| / max |G_ref| <= 3e-2.
The GPU path rounds five operands to bf16 (unit roundoff u = 2^-9): the gate-
scaled output gradient dY, the saved pre-activations a and b, H, and the
pre-activation gradients da | db, each feeding fp32-accumulated products.
Independent roundings of relative size <= u add up to a normwise relative
error of a few u ~ 0.2-0.6 %; 1e-2 leaves a factor of about two.  The router
gradient dL/dl = <dy, P_k> - G_k <dy, sum_j P_j> involves cancellation, which
the normwise measure (over all tokens) absorbs.  Routing must agree exactly:
the cases are seeded so that no token's K-th/(K+1)-th logit gap lies within
1e-3 (asserted), where fp32 and fp64 routing could differ.

Cases span several 128 x 256 tiles with ragged M and N tails in every
product, CTA-pair and multicast forms of the forward, top-1 and top-2, empty
experts (whose weight gradients must be zeros, or untouched when
accumulating), the split down projection of tiny batches, and T = 0.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests import parity

pytestmark = pytest.mark.gpu

NORM_TOL = 1e-2
LINF_TOL = 3e-2


@pytest.fixture(scope="module")
def moe(cuda_device):
    from sparse_mixture_experts_55_b300 import build
    build.build()
    import sparse_mixture_experts_55_b300 as m
    return m


def _np(t):
    return t.detach().cpu().numpy().astype(np.float64)


def _case(T, d, f, E, K, seed):
    Wg, W1, W3, W2 = W.mixtral_weights(d, f, E, seed=seed, device="cpu")
    x = W.rms_rows(T, d, seed * 7 + 1, "cpu", torch.bfloat16)
    dy = W.randn((T, d), 1.0, seed * 7 + 2, "cpu", torch.bfloat16)
    return x, Wg, W1, W3, W2, dy


def _errors(g, ref):
    g = np.asarray(g, np.float64)
    ref = np.asarray(ref, np.float64)
    nref = np.linalg.norm(ref)
    if nref == 0.0:
        return float(np.abs(g).max(initial=0.0)), float(np.abs(g).max(initial=0.0))
    return float(np.linalg.norm(g - ref) / nref), float(np.abs(g - ref).max() / np.abs(ref).max())


def _run(moe, x, Wg, W1, W3, W2, dy, K, flags=0, grads=None, fwd_flags=0):
    dev = torch.device("cuda:0")
    T, d = x.shape
    E, _, f = W1.shape
    xs, Wgs, W1s, W3s, W2s, dys = (t.to(dev) for t in (x, Wg, W1, W3, W2, dy))
    ws = moe.TrainWorkspace(T, d, f, E, K, torch.bfloat16, dev)
    y = moe.moe_forward_train(xs, Wgs, W1s, W3s, W2s, K, ws, flags=fwd_flags)
    g = moe.moe_backward(xs, Wgs, W1s, W3s, W2s, dys, K, ws, grads=grads, flags=flags)
    torch.cuda.synchronize()
    assert moe.moe_read_status(ws) == 0
    return y, g, ws


def _check(moe, T, d, f, E, K, seed, fwd_flags=0):
    x, Wg, W1, W3, W2, dy = _case(T, d, f, E, K, seed)
    dev = torch.device("cuda:0")
    # routing must match the oracle's exactly (no near-tie tokens in these seeds)
    ref_fwd = oracle.moe_layer(x, Wg, W1, W3, W2, K)
    idx, gate, *_ = moe.moe_route(x.to(dev), Wg.to(dev), K)
    rep = parity.check_routing(idx.cpu().numpy(), gate.cpu().numpy(), ref_fwd.gating, K)
    assert rep.n_mismatch == 0 and rep.n_exempt_in_out == 0, rep
    y, g, _ = _run(moe, x, Wg, W1, W3, W2, dy, K, fwd_flags=fwd_flags)
    # the training forward computes the same layer as moe_forward, bit for bit
    # where moe_forward does not split the gate/up contraction (it does for
    # at most four rows per touched expert; the training forward never does)
    assert parity.rel_linf(_np(y.float()), ref_fwd.y) <= parity.TOL["bf16"]
    if T * K > 4 * min(T * K, E):
        y_plain = moe.moe_forward(*(t.to(dev) for t in (x, Wg, W1, W3, W2)), K, flags=fwd_flags)
        assert torch.equal(y, y_plain)
    ref = oracle.moe_layer_backward(x, Wg, W1, W3, W2, K, dy)
    report = {}
    for name, gg, rr in (("dx", g.dx, ref.dx), ("dWg", g.dWg, ref.dWg), ("dW1", g.dW1, ref.dW1),
                         ("dW3", g.dW3, ref.dW3), ("dW2", g.dW2, ref.dW2)):
        report[name] = _errors(_np(gg), rr)
    print(f"\nbackward T={T} d={d} f={f} E={E} K={K}: " +
          ", ".join(f"{k} {v[0]:.2e}/{v[1]:.2e}" for k, v in report.items()))
    for name, (nrm, linf) in report.items():
        assert nrm <= NORM_TOL and linf <= LINF_TOL, (name, nrm, linf)
    # experts no token chose have exactly zero weight gradients
    used = np.zeros(E, bool)
    used[np.unique(ref_fwd.gating.idx)] = True
    for e in np.nonzero(~used)[0]:
        assert not g.dW1[e].any() and not g.dW3[e].any() and not g.dW2[e].any()
    return x, Wg, W1, W3, W2, dy, g


@pytest.mark.parametrize("T,d,f,E,K,seed", [
    (300, 256, 512, 8, 2, 11),     # multicast-pair forward, several tiles per product
    (257, 192, 320, 8, 2, 15),     # ragged M and N tails in every product
    (600, 256, 512, 4, 1, 13),     # top-1: zero router gradient
    (3, 256, 512, 8, 2, 14),       # empty experts, split down projection
    (129, 128, 256, 32, 2, 13),    # many experts, most segments one tile
    (1100, 128, 384, 4, 2, 33),    # several m-tiles per expert
])
def test_backward_parity(moe, T, d, f, E, K, seed):
    _check(moe, T, d, f, E, K, seed)


def test_backward_parity_pair_form(moe):
    # CTA-pair MMAs in the forward (odd tile counts: phantom halves never stored)
    _check(moe, 1100, 128, 384, 4, 2, 33, fwd_flags=moe.MOE_GEMM_PAIR_MMA)


def test_backward_deterministic_and_accumulate(moe):
    T, d, f, E, K = 257, 192, 320, 8, 2
    x, Wg, W1, W3, W2, dy = _case(T, d, f, E, K, 15)
    _, g1, _ = _run(moe, x, Wg, W1, W3, W2, dy, K)
    _, g2, _ = _run(moe, x, Wg, W1, W3, W2, dy, K)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)
    # accumulate: the result is added to what the buffers held
    base = [torch.randn_like(t) for t in g1]
    acc = [t.clone() for t in base]
    _, g3, _ = _run(moe, x, Wg, W1, W3, W2, dy, K, flags=moe.MOE_ACCUMULATE, grads=type(g1)(*acc))
    for b0, g, s in zip(base, g1, g3):
        torch.testing.assert_close(s, b0 + g, rtol=1e-6, atol=1e-6)


def test_backward_accumulate_leaves_empty_experts(moe):
    T, d, f, E, K = 3, 256, 512, 8, 2
    x, Wg, W1, W3, W2, dy = _case(T, d, f, E, K, 14)
    _, g0, _ = _run(moe, x, Wg, W1, W3, W2, dy, K)
    base = [torch.full_like(t, 0.5) for t in g0]
    _, g1, _ = _run(moe, x, Wg, W1, W3, W2, dy, K, flags=moe.MOE_ACCUMULATE, grads=type(g0)(*[t.clone() for t in base]))
    idx = oracle.gating(x, Wg, K).idx
    for e in set(range(E)) - set(np.unique(idx).tolist()):
        assert torch.all(g1.dW1[e] == 0.5) and torch.all(g1.dW2[e] == 0.5)


def test_backward_empty_batch(moe, cuda_device):
    d, f, E, K = 128, 256, 4, 2
    Wg, W1, W3, W2 = (t.to(cuda_device) for t in W.mixtral_weights(d, f, E, seed=5, device="cpu"))
    x = torch.empty(0, d, dtype=torch.bfloat16, device=cuda_device)
    ws = moe.TrainWorkspace(0, d, f, E, K, torch.bfloat16, cuda_device)
    grads = moe.LayerGrads(torch.empty(0, d, device=cuda_device), torch.ones(d, E, device=cuda_device),
                           torch.ones(E, d, f, device=cuda_device), torch.ones(E, d, f, device=cuda_device),
                           torch.ones(E, f, d, device=cuda_device))
    moe.moe_backward(x, Wg, W1, W3, W2, x, K, ws, grads=grads)
    torch.cuda.synchronize()
    for t in grads[1:]:
        assert not t.any()


def test_forced_timeout_is_reported_and_the_next_call_is_correct(moe):
    # The dH product's MMA thread waits on a barrier nothing signals; after
    # about a second the wait gives up, the CTAs drain their copies, free
    # TMEM and exit, and the status word reads MOE_ERR_DEVICE_TIMEOUT.  The
    # context stays usable: a clean call on the same workspace is correct.
    T, d, f, E, K = 300, 256, 512, 8, 2
    x, Wg, W1, W3, W2, dy = _case(T, d, f, E, K, 11)
    dev = torch.device("cuda:0")
    xs, Wgs, W1s, W3s, W2s, dys = (t.to(dev) for t in (x, Wg, W1, W3, W2, dy))
    ws = moe.TrainWorkspace(T, d, f, E, K, torch.bfloat16, dev)
    moe.moe_forward_train(xs, Wgs, W1s, W3s, W2s, K, ws)
    moe.moe_backward(xs, Wgs, W1s, W3s, W2s, dys, K, ws, flags=moe.MOE_DEBUG_FORCE_TIMEOUT)
    torch.cuda.synchronize()
    assert moe.moe_read_status(ws) == moe._lib.MOE_ERR_DEVICE_TIMEOUT
    moe.moe_forward_train(xs, Wgs, W1s, W3s, W2s, K, ws)  # clears the status word
    g = moe.moe_backward(xs, Wgs, W1s, W3s, W2s, dys, K, ws)
    torch.cuda.synchronize()
    assert moe.moe_read_status(ws) == 0
    ref = oracle.moe_layer_backward(x, Wg, W1, W3, W2, K, dy)
    for gg, rr in ((g.dx, ref.dx), (g.dW1, ref.dW1), (g.dW2, ref.dW2)):
        assert _errors(_np(gg), rr)[0] <= NORM_TOL
