"""Pins for the float64 oracle: each check ties it to something other than itself.

| oracle part            | pinned by                                                        |
|------------------------|------------------------------------------------------------------|
| gating (TopK+softmax)  | closed form g = (3/4, 1/4) for logits (0, ln 3, ...); invariants  |
|                        | g >= 0, sum 1, exactly K non-zero, g1 >= g2; brute-force rank    |
|                        | definition of TopK; hand-derived worked example                  |
| routed == dense        | brute-force all-expert evaluation with zero weights off the top-K |
| SwiGLU expert          | torch.nn.functional (linear, silu) library evaluation; K = n = 1 |
|                        | reduces the layer to a plain SwiGLU FFN; hand example            |
| combine                | linearity in W2; token-permutation equivariance; expert          |
|                        | relabelling invariance; hand example                             |
| permutation            | brute force via Python's sorted() on (expert, token, slot)       |
| tie-break              | exact rational arithmetic (fractions.Fraction) on tie tokens     |
| RMSNorm                | closed form on a 3-4-5 row; torch.nn.functional.rms_norm         |
| shapes / params        | 3*4096*14336 = 176,160,768 per expert; 45.1B over 32 layers      |
| logit_gaps             | hand-built rows with known order statistics (exact ties too);    |
|                        | the gap as min over the kept logits minus max over the rest      |
| moe_layer_tokens       | the full layer's rows at the same tokens (unsorted, repeated)    |
| moe_block (pre-norm)   | hand-derived two-token block example (tests/golden)              |

The mutation tests at the end plant plausible mistakes in the oracle (on the
CPU) and check that at least one pin fails for each.
"""
from __future__ import annotations

import json
import math
import pathlib
import re
from fractions import Fraction

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import oracle.moe_oracle as OM
import workloads as W

GOLDEN = pathlib.Path(__file__).resolve().parent / "golden"


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------
def _ln3(v):
    if isinstance(v, str):
        return {"ln3": math.log(3.0), "-ln3": -math.log(3.0)}[v]
    return float(v)


def _load_hand():
    h = json.loads((GOLDEN / "hand_example.json").read_text())
    conv = lambda a: np.vectorize(_ln3, otypes=[np.float64])(np.array(a, dtype=object))
    Wg = conv(h["Wg"]).T                      # listed per expert -> [d, n]
    return h, conv(h["x"]), Wg, conv(h["W1"]), conv(h["W3"]), conv(h["W2"])


def _tiny(E=8, K=2, T=64, d=64, f=128, seed=W.BASE_SEED):
    return W.tiny_fp32(T=T, d=d, f=f, E=E, K=K, seed=seed)


# ---------------------------------------------------------------------------
# pins (plain functions so the mutation tests can rerun them)
# ---------------------------------------------------------------------------
def pin_gate_closed_form():
    # one-hot token picks row 0 of Wg: logits (0, ln 3, -1, -2)
    x = np.array([[1.0, 0.0]])
    Wg = np.array([[0.0, math.log(3.0), -1.0, -2.0], [5.0, 5.0, 5.0, 5.0]])
    g = oracle.gating(x, Wg, 2)
    assert list(g.idx[0]) == [1, 0]
    assert abs(g.gate[0, 0] - 0.75) < 1e-15 and abs(g.gate[0, 1] - 0.25) < 1e-15
    assert np.allclose(g.G[0], [0.25, 0.75, 0.0, 0.0], rtol=0, atol=1e-15)


def pin_gate_invariants():
    for E, K in [(8, 2), (8, 1), (4, 2), (1, 1), (3, 3)]:
        inp = _tiny(E=E, K=K)
        g = oracle.gating(inp.x, inp.Wg, K)
        assert (g.G >= 0).all()
        assert np.allclose(g.G.sum(axis=1), 1.0, rtol=0, atol=1e-14)
        assert ((g.G > 0).sum(axis=1) == K).all()
        for t in range(g.G.shape[0]):
            assert len(set(g.idx[t].tolist())) == K
            assert set(np.nonzero(g.G[t])[0].tolist()) == set(g.idx[t].tolist())
        if K >= 2:
            assert (g.gate[:, 0] >= g.gate[:, 1]).all()


def pin_topk_bruteforce():
    rng = np.random.default_rng(7)
    for E, K in [(8, 2), (8, 1), (5, 3), (2, 2)]:
        logits = rng.integers(-3, 4, size=(300, E)).astype(np.float64)  # many ties
        idx = oracle.topk_indices(logits, K)
        for t in range(logits.shape[0]):
            l = logits[t]
            # rank(i) = #experts ahead of i: larger logit, or equal logit and lower index
            rank = [sum(1 for j in range(E) if l[j] > l[i] or (l[j] == l[i] and j < i)) for i in range(E)]
            want = [i for r in range(K) for i in range(E) if rank[i] == r]
            assert idx[t].tolist() == want


def pin_routed_equals_dense():
    for E, K in [(8, 2), (8, 1), (4, 3)]:
        inp = _tiny(E=E, K=K)
        a = oracle.moe_layer(inp.x, inp.Wg, inp.W1, inp.W3, inp.W2, K).y
        b = oracle.moe_layer_dense(inp.x, inp.Wg, inp.W1, inp.W3, inp.W2, K).y
        assert np.abs(a - b).max() <= 1e-12 * max(1.0, np.abs(b).max())


def _swiglu_torch(x, W1, W3, W2):
    x = torch.as_tensor(x, dtype=torch.float64)
    W1, W3, W2 = (torch.as_tensor(np.asarray(w, dtype=np.float64)) for w in (W1, W3, W2))
    h = F.silu(F.linear(x, W1.T)) * F.linear(x, W3.T)
    return F.linear(h, W2.T).numpy()


def pin_expert_library():
    inp = _tiny(E=8, K=2)
    x = oracle.f64(inp.x)
    for e in (0, 5):
        got = oracle.expert(x, inp.W1[e], inp.W3[e], inp.W2[e])
        want = _swiglu_torch(x, oracle.f64(inp.W1[e]), oracle.f64(inp.W3[e]), oracle.f64(inp.W2[e]))
        assert np.abs(got - want).max() <= 1e-12 * np.abs(want).max()


def pin_silu_library():
    z = np.linspace(-60, 60, 2001)
    want = F.silu(torch.as_tensor(z)).numpy()
    assert np.allclose(oracle.silu(z), want, rtol=1e-14, atol=1e-300)
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    assert abs(oracle.silu(np.array([math.log(3.0)]))[0] - 0.75 * math.log(3.0)) < 1e-15


def pin_k1_reduces_to_swiglu():
    inp = _tiny(E=1, K=1)
    y = oracle.moe_layer(inp.x, inp.Wg, inp.W1, inp.W3, inp.W2, 1).y
    want = _swiglu_torch(oracle.f64(inp.x), oracle.f64(inp.W1[0]), oracle.f64(inp.W3[0]), oracle.f64(inp.W2[0]))
    assert np.abs(y - want).max() <= 1e-12 * np.abs(want).max()


def pin_hand_example():
    h, x, Wg, W1, W3, W2 = _load_hand()
    r = oracle.moe_layer(x, Wg, W1, W3, W2, h["K"])
    assert r.gating.idx.tolist() == h["expected_idx"]
    assert np.allclose(r.gating.gate, h["expected_gate"], rtol=0, atol=1e-15)
    want = np.array(h["expected_y_over_ln3"]) * math.log(3.0)
    assert np.allclose(r.y, want, rtol=0, atol=1e-12)
    rd = oracle.moe_layer_dense(x, Wg, W1, W3, W2, h["K"])
    assert np.allclose(rd.y, want, rtol=0, atol=1e-12)


def pin_linearity_and_equivariance():
    inp = _tiny()
    K = inp.K
    base = oracle.moe_layer(inp.x, inp.Wg, inp.W1, inp.W3, inp.W2, K)
    # scaling W2 by c scales y by c
    y2 = oracle.moe_layer(inp.x, inp.Wg, inp.W1, inp.W3, oracle.f64(inp.W2) * 2.5, K).y
    assert np.allclose(y2, 2.5 * base.y, rtol=1e-13, atol=1e-13)
    # permuting tokens permutes outputs
    perm = np.random.default_rng(3).permutation(inp.x.shape[0])
    yp = oracle.moe_layer(oracle.f64(inp.x)[perm], inp.Wg, inp.W1, inp.W3, inp.W2, K).y
    assert np.allclose(yp, base.y[perm], rtol=0, atol=1e-13)
    # relabelling experts (columns of Wg with the banks) leaves y unchanged
    gap_io, gap_12 = oracle.logit_gaps(base.gating.logits, K)
    assert gap_io.min() > 1e-9 and gap_12.min() > 1e-9
    sigma = np.random.default_rng(4).permutation(inp.Wg.shape[1])
    yr = oracle.moe_layer(inp.x, oracle.f64(inp.Wg)[:, sigma], oracle.f64(inp.W1)[sigma],
                          oracle.f64(inp.W3)[sigma], oracle.f64(inp.W2)[sigma], K)
    assert np.allclose(yr.y, base.y, rtol=0, atol=1e-13)
    assert (sigma[yr.gating.idx] == base.gating.idx).all()


def pin_permutation_bruteforce():
    rng = np.random.default_rng(11)
    for T, E, K in [(50, 8, 2), (33, 4, 1), (1, 8, 2), (200, 8, 2), (17, 3, 3)]:
        idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
        p = oracle.permutation(idx, E)
        pairs = sorted((int(idx[t, k]), t, k) for t in range(T) for k in range(K))
        assert p.perm_tok.tolist() == [t for _, t, _ in pairs]
        assert p.perm_k.tolist() == [k for _, _, k in pairs]
        assert p.counts.tolist() == [sum(1 for e, _, _ in pairs if e == j) for j in range(E)]
        assert p.offsets[0] == 0 and p.offsets[-1] == T * K
        for t in range(T):
            for k in range(K):
                r = p.pos[t, k]
                assert p.perm_tok[r] == t and p.perm_k[r] == k
                assert p.offsets[idx[t, k]] <= r < p.offsets[idx[t, k] + 1]


def pin_rmsnorm():
    h = np.array([[3.0, 4.0], [0.0, 0.0], [1.0, -1.0]])
    got = oracle.rmsnorm(h, eps=1e-5)
    assert np.allclose(got[0], np.array([3.0, 4.0]) / math.sqrt(12.5 + 1e-5), rtol=1e-15)
    assert (got[1] == 0).all()
    z = np.random.default_rng(5).standard_normal((16, 64))
    want = F.rms_norm(torch.as_tensor(z), (64,), eps=1e-5).numpy()
    assert np.allclose(oracle.rmsnorm(z, eps=1e-5), want, rtol=1e-13, atol=1e-14)


def pin_tie_tokens_exact():
    inp = W.skew(T=400, d=512, f=8, E=8, K=2, n_tie=40, weights=(None, None, None, None))
    x = inp.x.float().numpy()
    Wg = inp.Wg.float().numpy()
    g = oracle.gating(inp.x, inp.Wg, 2)
    for t, pat in zip(inp.meta["tie_tokens"], inp.meta["tie_patterns"]):
        nz = np.nonzero(x[t])[0]
        exact = [sum(Fraction(float(x[t, j])) * Fraction(float(Wg[j, e])) for j in nz) for e in range(8)]
        assert exact == [Fraction(v) for v in W.TIE_PATTERNS[pat]]
        assert tuple(g.idx[t].tolist()) == W.TIE_EXPECTED[pat]
        assert g.logits[t].tolist() == [float(v) for v in exact]


def pin_param_accounting():
    c = W.param_counts(4096, 14336, 8, layers=32)
    assert c["per_expert"] == 176_160_768
    assert abs(c["per_layer_experts"] - 1.409e9) < 1e6
    assert abs(c["all_layers_experts"] - 45.1e9) < 0.01e9
    assert c["router_all_layers"] == 32 * 4096 * 8
    # the generators produce those shapes (small stand-in with the same rule)
    Wg, W1, W3, W2 = W.mixtral_weights(d=64, f=96, E=8, device="cpu")
    assert W1.numel() + W3.numel() + W2.numel() == 8 * W.param_counts(64, 96, 8)["per_expert"]
    assert Wg.shape == (64, 8) and W1.shape == (8, 64, 96) and W2.shape == (8, 96, 64)


def pin_logit_gaps():
    # hand-built rows: (sorted values) -> (K-th minus (K+1)-th, 1st minus 2nd)
    rows = np.array([[1.0, 2.0, 4.0, 0.5, 3.0],     # 4 > 3 > 2 > 1 > .5
                     [5.0, 3.0, 3.0, 1.0, -2.0],    # tie between the 2nd and 3rd
                     [2.0, 2.0, 1.0, 0.0, 0.0],     # tie between the 1st and 2nd
                     [-1.0, -1.0, -1.0, -1.0, -1.0],
                     [0.0, 10.0, -10.0, 7.5, 7.25]])
    gio, g12 = oracle.logit_gaps(rows, 2)
    assert gio.tolist() == [1.0, 0.0, 1.0, 0.0, 0.25]
    assert g12.tolist() == [1.0, 2.0, 0.0, 0.0, 2.5]
    gio1, g121 = oracle.logit_gaps(rows, 1)
    assert gio1.tolist() == [1.0, 2.0, 0.0, 0.0, 2.5]
    assert np.isinf(g121).all()
    gio3, _ = oracle.logit_gaps(rows, 3)
    assert gio3.tolist() == [1.0, 2.0, 1.0, 0.0, 7.25]
    # K = n: nothing is left out, so the gap is undefined
    assert np.isinf(oracle.logit_gaps(rows[:, :2], 2)[0]).all()
    # a second characterisation: the smallest kept logit minus the largest
    # logit left out, and the two kept logits' difference, with the kept set
    # from the (pinned) TopK
    rng = np.random.default_rng(13)
    for E, K in [(8, 2), (8, 1), (5, 3)]:
        logits = rng.integers(-4, 5, size=(400, E)).astype(np.float64) / 4.0
        idx = oracle.topk_indices(logits, K)
        gio, g12 = oracle.logit_gaps(logits, K)
        for t in range(logits.shape[0]):
            kept = set(idx[t].tolist())
            want = min(logits[t, i] for i in kept) - max(logits[t, j] for j in range(E) if j not in kept)
            assert gio[t] == want
            if K >= 2:
                assert g12[t] == logits[t, idx[t, 0]] - logits[t, idx[t, 1]]


def pin_layer_tokens_restriction():
    inp = _tiny()
    full = oracle.moe_layer(inp.x, inp.Wg, inp.W1, inp.W3, inp.W2, inp.K)
    for tokens in ([5, 0, 63, 5, 17], [63], list(range(64))[::-3]):
        sub = oracle.moe_layer_tokens(inp.x, inp.Wg, inp.W1, inp.W3, inp.W2, inp.K, tokens)
        assert sub.y.shape == (len(tokens), full.y.shape[1])
        assert np.abs(sub.y - full.y[tokens]).max() <= 1e-13 * np.abs(full.y).max()
        assert (sub.gating.idx == full.gating.idx[tokens]).all()
        assert np.allclose(sub.gating.gate, full.gating.gate[tokens], rtol=0, atol=1e-15)


_LN3_TERM = re.compile(r"^\s*([+-]?\s*[0-9.]+)?\s*(\*\s*ln3)?\s*$")


def _ln3_expr(v) -> float:
    """Value of a golden-file entry: a number, or a sum of terms 'c' and 'c*ln3'."""
    if not isinstance(v, str):
        return float(v)
    total = 0.0
    for term in re.findall(r"[+-]?[^+-]+", v.replace(" ", "")):
        m = _LN3_TERM.match(term)
        assert m, f"bad golden term {term!r}"
        coef = float(m.group(1).replace(" ", "")) if m.group(1) not in (None, "+", "-") else \
            (-1.0 if m.group(1) == "-" else 1.0)
        total += coef * (math.log(3.0) if m.group(2) else 1.0)
    return total


def pin_block_hand_example():
    b = json.loads((GOLDEN / "block_example.json").read_text())
    conv = lambda a: np.vectorize(_ln3_expr, otypes=[np.float64])(np.array(a, dtype=object))
    h, Wg, W1, W3, W2 = (conv(b[k]) for k in ("h", "Wg", "W1", "W3", "W2"))
    assert np.allclose(oracle.rmsnorm(h, eps=b["eps"]), conv(b["expected_xnorm"]), rtol=0, atol=1e-15)
    g = oracle.gating(oracle.rmsnorm(h, eps=b["eps"]), Wg, b["K"])
    assert g.idx.tolist() == b["expected_idx"]
    assert np.allclose(g.gate, b["expected_gate"], rtol=0, atol=1e-15)
    out = oracle.moe_block(h, Wg, W1, W3, W2, b["K"], eps=b["eps"])
    assert np.allclose(out, conv(b["expected_out"]), rtol=0, atol=1e-13)


PINS = [pin_gate_closed_form, pin_gate_invariants, pin_topk_bruteforce, pin_routed_equals_dense,
        pin_expert_library, pin_silu_library, pin_k1_reduces_to_swiglu, pin_hand_example,
        pin_linearity_and_equivariance, pin_permutation_bruteforce, pin_rmsnorm,
        pin_tie_tokens_exact, pin_param_accounting, pin_logit_gaps, pin_layer_tokens_restriction,
        pin_block_hand_example]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin()


# ---------------------------------------------------------------------------
# mutation tests: a plausible mistake planted in the oracle must fail a pin
# ---------------------------------------------------------------------------
def _silu_wrong_sign(z):
    return z / (1.0 + np.exp(z))


def _expert_swapped_branches(x, W1e, W3e, W2e):
    x = OM.f64(x)
    return (OM.silu(x @ OM.f64(W3e)) * (x @ OM.f64(W1e))) @ OM.f64(W2e)


def _expert_dropped_gate_branch(x, W1e, W3e, W2e):
    x = OM.f64(x)
    return (OM.silu(x @ OM.f64(W1e))) @ OM.f64(W2e)


def _expert_transposed_down(x, W1e, W3e, W2e):
    x = OM.f64(x)
    W2e = OM.f64(W2e)
    W2t = W2e.T if W2e.shape[0] == W2e.shape[1] else W2e[::-1]
    return (OM.silu(x @ OM.f64(W1e)) * (x @ OM.f64(W3e))) @ W2t


def _topk_higher_index_wins(logits, K):
    T, E = logits.shape
    order = np.lexsort((-np.broadcast_to(np.arange(E), (T, E)), -logits), axis=1)
    return order[:, :K].astype(np.int32)


def _topk_smallest(logits, K):
    return np.argsort(logits, axis=1, kind="stable")[:, :K].astype(np.int32)


def _mask_nothing(logits, idx):
    return logits.copy()


def _softmax_no_max_shift_wrong(v):
    e = np.exp(v)
    return e / e.sum(axis=-1, keepdims=True) * 0.999


def _router_transposed(x, Wg):
    Wg = OM.f64(Wg)
    return OM.f64(x) @ (Wg[::-1] if Wg.shape[0] > 1 else Wg)


def _perm_unstable(idx, E):
    p = _ORIG["permutation"](idx, E)
    # reverse the order inside every expert segment
    for e in range(E):
        a, b = int(p.offsets[e]), int(p.offsets[e + 1])
        p.perm_tok[a:b] = p.perm_tok[a:b][::-1].copy()
        p.perm_k[a:b] = p.perm_k[a:b][::-1].copy()
    return p


def _rmsnorm_no_sqrt(h, eps=1e-5):
    h = OM.f64(h)
    return h / (np.mean(h * h, axis=1, keepdims=True) + eps)


def _moe_layer_swapped_gates(x, Wg, W1, W3, W2, K):
    r = _ORIG["moe_layer"](x, Wg, W1, W3, W2, K)
    x64 = OM.f64(x)
    g = r.gating
    y = np.zeros_like(r.y)
    for t in range(x64.shape[0]):
        for k in range(K):
            e = int(g.idx[t, k])
            y[t] += g.gate[t, K - 1 - k] * OM.expert(x64[t:t + 1], W1[e], W3[e], W2[e])[0]
    return OM.LayerResult(y, g)


def _gaps_first_minus_third(logits, K):
    s = -np.sort(-logits, axis=1)
    T, E = logits.shape
    gap_in_out = s[:, 0] - s[:, K] if E > K else np.full(T, np.inf)
    gap_12 = s[:, 0] - s[:, 1] if (K >= 2 and E >= 2) else np.full(T, np.inf)
    return gap_in_out, gap_12


def _gaps_off_by_one(logits, K):
    s = -np.sort(-logits, axis=1)
    T, E = logits.shape
    gap_in_out = s[:, K] - s[:, K + 1] if E > K + 1 else np.full(T, np.inf)
    gap_12 = s[:, 0] - s[:, 1] if (K >= 2 and E >= 2) else np.full(T, np.inf)
    return gap_in_out, gap_12


def _layer_tokens_first_n(x, Wg, W1, W3, W2, K, tokens):
    return OM.moe_layer(OM.f64(x)[:len(tokens)], Wg, W1, W3, W2, K)


def _layer_tokens_sorted(x, Wg, W1, W3, W2, K, tokens):
    return OM.moe_layer(OM.f64(x)[np.sort(np.asarray(tokens))], Wg, W1, W3, W2, K)


def _block_residual_before_norm(h, Wg, W1, W3, W2, K, eps=1e-5):
    # post-norm: the residual sum is normalised instead of the block input
    h64 = OM.f64(h)
    return OM.rmsnorm(h64 + OM.moe_layer(h64, Wg, W1, W3, W2, K).y, eps)


def _block_residual_of_normed(h, Wg, W1, W3, W2, K, eps=1e-5):
    n = OM.rmsnorm(OM.f64(h), eps)
    return n + OM.moe_layer(n, Wg, W1, W3, W2, K).y


def _block_no_norm(h, Wg, W1, W3, W2, K, eps=1e-5):
    h64 = OM.f64(h)
    return h64 + OM.moe_layer(h64, Wg, W1, W3, W2, K).y


_ORIG = {name: getattr(OM, name) for name in
         ("silu", "expert", "topk_indices", "topk_mask", "softmax", "router_logits", "permutation",
          "rmsnorm", "moe_layer", "logit_gaps", "moe_layer_tokens", "moe_block")}

MUTANTS = {
    "silu_wrong_sign": ("silu", _silu_wrong_sign),
    "expert_swapped_branches": ("expert", _expert_swapped_branches),
    "expert_dropped_gate_branch": ("expert", _expert_dropped_gate_branch),
    "expert_transposed_down": ("expert", _expert_transposed_down),
    "topk_higher_index_wins": ("topk_indices", _topk_higher_index_wins),
    "topk_smallest": ("topk_indices", _topk_smallest),
    "mask_nothing": ("topk_mask", _mask_nothing),
    "softmax_bad_norm": ("softmax", _softmax_no_max_shift_wrong),
    "router_rows_reversed": ("router_logits", _router_transposed),
    "permutation_unstable": ("permutation", _perm_unstable),
    "rmsnorm_no_sqrt": ("rmsnorm", _rmsnorm_no_sqrt),
    "combine_gates_swapped": ("moe_layer", _moe_layer_swapped_gates),
    "gaps_first_minus_third": ("logit_gaps", _gaps_first_minus_third),
    "gaps_off_by_one": ("logit_gaps", _gaps_off_by_one),
    "layer_tokens_first_n": ("moe_layer_tokens", _layer_tokens_first_n),
    "layer_tokens_sorted": ("moe_layer_tokens", _layer_tokens_sorted),
    "block_residual_before_norm": ("moe_block", _block_residual_before_norm),
    "block_residual_of_normed": ("moe_block", _block_residual_of_normed),
    "block_no_norm": ("moe_block", _block_no_norm),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(OM, attr, fn)
    monkeypatch.setattr(oracle, attr, fn)
    caught = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin()
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {name}"
