"""Pins for the oracle's backward pass (moe_oracle.moe_layer_backward).

| part                     | pinned by                                                      |
|--------------------------|----------------------------------------------------------------|
| every gradient           | central finite differences of L = <dy, y> through the pinned   |
|                          | forward oracle, on tiny float64 inputs with no logit near-ties  |
| dsilu                    | finite differences of the pinned SiLU; torch.autograd of         |
|                          | torch.nn.functional.silu                                        |
| K = n = 1                | no router gradient (the single gate is the constant 1)          |
| router path              | dlogits sum to zero per token (softmax), zero off the kept set  |

Planted mistakes at the end are each caught.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import oracle.moe_oracle as OM
import workloads as W


def _case(T=6, d=8, f=12, E=4, K=2, seed=3):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d))
    Wg = rng.standard_normal((d, E)) / np.sqrt(d)
    W1 = rng.standard_normal((E, d, f)) / np.sqrt(d)
    W3 = rng.standard_normal((E, d, f)) / np.sqrt(d)
    W2 = rng.standard_normal((E, f, d)) / np.sqrt(f)
    dy = rng.standard_normal((T, d))
    # no near-ties: the selected set must not change under the perturbation
    gap_io, gap_12 = OM.logit_gaps(OM.router_logits(x, Wg), K)
    assert gap_io.min() > 1e-3 and (K < 2 or gap_12.min() > 1e-3)
    return x, Wg, W1, W3, W2, dy


def _loss(x, Wg, W1, W3, W2, K, dy):
    return float(np.sum(oracle.moe_layer(x, Wg, W1, W3, W2, K).y * dy))


def _fd(fun, arr, idx, eps=1e-6):
    old = arr[idx]
    arr[idx] = old + eps
    lp = fun()
    arr[idx] = old - eps
    lm = fun()
    arr[idx] = old
    return (lp - lm) / (2 * eps)


@pytest.mark.parametrize("K,E", [(2, 4), (1, 3), (2, 2)])
def test_gradients_match_finite_differences(K, E):
    x, Wg, W1, W3, W2, dy = _case(E=E, K=K, seed=10 + E + K)
    gr = oracle.moe_layer_backward(x, Wg, W1, W3, W2, K, dy)
    fun = lambda: _loss(x, Wg, W1, W3, W2, K, dy)
    rng = np.random.default_rng(0)
    for name, arr, grad in (("x", x, gr.dx), ("Wg", Wg, gr.dWg), ("W1", W1, gr.dW1), ("W3", W3, gr.dW3),
                            ("W2", W2, gr.dW2)):
        for _ in range(12):
            idx = tuple(int(rng.integers(0, n)) for n in arr.shape)
            num = _fd(fun, arr, idx)
            assert abs(num - grad[idx]) <= 1e-6 * (1 + abs(num)), (name, idx, num, grad[idx])


def test_dsilu_against_finite_differences_and_autograd():
    z = np.linspace(-8, 8, 101)
    fd = (oracle.silu(z + 1e-6) - oracle.silu(z - 1e-6)) / 2e-6
    assert np.abs(fd - oracle.dsilu(z)).max() < 1e-8
    zt = torch.tensor(z, requires_grad=True)
    torch.nn.functional.silu(zt).sum().backward()
    assert np.abs(zt.grad.numpy() - oracle.dsilu(z)).max() < 1e-12


def test_single_expert_has_no_router_gradient():
    x, Wg, W1, W3, W2, dy = _case(E=1, K=1, seed=5)
    gr = oracle.moe_layer_backward(x, Wg, W1, W3, W2, 1, dy)
    assert np.all(gr.dWg == 0) and np.all(gr.dlogits == 0)


def test_router_gradient_structure():
    x, Wg, W1, W3, W2, dy = _case(T=20, E=6, K=2, seed=8)
    gr = oracle.moe_layer_backward(x, Wg, W1, W3, W2, 2, dy)
    g = oracle.gating(x, Wg, 2)
    assert np.abs(gr.dlogits.sum(axis=1)).max() < 1e-12            # softmax: sums to zero
    kept = np.zeros_like(g.G, dtype=bool)
    np.put_along_axis(kept, g.idx.astype(np.int64), True, axis=1)
    assert np.all(gr.dlogits[~kept] == 0)


# ---------------------------------------------------------------------------
# planted mistakes
# ---------------------------------------------------------------------------
def _dsilu_missing_term(z):
    sg = 1.0 / (1.0 + np.exp(-z))
    return sg


def _softmax_backward_sign(G, dG):
    return G * (dG + np.sum(G * dG, axis=1, keepdims=True))


def _softmax_backward_no_centering(G, dG):
    return G * dG


PLANTS = {"dsilu_missing_term": ("dsilu", _dsilu_missing_term),
          "softmax_backward_sign": ("softmax_backward", _softmax_backward_sign),
          "softmax_backward_not_centred": ("softmax_backward", _softmax_backward_no_centering)}


@pytest.mark.parametrize("name", sorted(PLANTS))
def test_planted_backward_mistake_is_caught(name, monkeypatch):
    attr, fn = PLANTS[name]
    monkeypatch.setattr(OM, attr, fn)
    with pytest.raises(AssertionError):
        test_gradients_match_finite_differences(2, 4)


def test_weight_gradients_separate_over_columns_and_dx_over_tokens():
    # The full-size GPU check samples these: restricting every expert to a set
    # J of intermediate columns leaves the routing and the gradients of the
    # kept weights unchanged, and a token subset keeps its dx rows.
    x, Wg, W1, W3, W2, dy = _case(T=9, d=8, f=12, E=4, K=2, seed=8)
    full = oracle.moe_layer_backward(x, Wg, W1, W3, W2, 2, dy)
    J = [0, 5, 11]
    part = oracle.moe_layer_backward(x, Wg, W1[:, :, J], W3[:, :, J], W2[:, J, :], 2, dy)
    np.testing.assert_allclose(part.dW1, full.dW1[:, :, J], rtol=0, atol=1e-12)
    np.testing.assert_allclose(part.dW3, full.dW3[:, :, J], rtol=0, atol=1e-12)
    np.testing.assert_allclose(part.dW2, full.dW2[:, J, :], rtol=0, atol=1e-12)
    S = [1, 4, 8]
    sub = oracle.moe_layer_backward(x[S], Wg, W1, W3, W2, 2, dy[S])
    np.testing.assert_allclose(sub.dx, full.dx[S], rtol=0, atol=1e-12)
