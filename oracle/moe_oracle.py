"""Float64 CPU oracle for the Mixtral sparse mixture-of-experts feed-forward layer.

TEST INFRASTRUCTURE.  Only the test suite, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import this
module.  It imports nothing from the CUDA library and the library imports
nothing from here; the two share only the seeded input generators.

It is the plain definition, written out, on float64 copies of exactly the
tensors handed to the GPU (bf16 or fp32 values upcast without change).  NumPy
matmul, exp, and a sort are used as library steps; there is no blocking,
fusion or reordering beyond what the definition states.

Sources (Mixtral of Experts, arXiv 2401.04088, as summarised on the web pages):
  [GU-3.4]    paper-graph-ui summary, section 3.4 "MoE Layer Formulation":
              the gating function G(x) = Softmax(TopK(x . W_g)), the
              element-wise TopK definition (-inf off the top-K) and the output
              combination y = sum_i G(x)_i . E_i(x); only the selected experts
              compute.
  [GU-SWIGLU] same page, "Expert Network Structure (SwiGLU)":
              E_i(x) = W_3,i (SiLU(W_1,i x) (.) W_2,i x), SiLU(z) = z sigma(z).
  [GU-TOPK]   same page, "Top-K Gating Mechanism and Routing": the three-step
              Top-2 procedure (pick the two largest, mask the rest to -inf,
              softmax); no router bias.
  [GU-ARCH]   same page, "Architectural Inheritance from Mistral 7B",
              layer-normalisation paragraph: RMSNorm before the MoE block
              (pre-norm); section 3 information flow: the MoE sum is added to
              the residual stream.
  [GU-INFRA]  same page, "Inference and Deployment Infrastructure": the inputs
              of all experts are packed into one matrix, i.e. tokens are
              grouped by expert.
  [XYZ-M]     xyznot reading guide, "Method (with the key equations)": n = 8
              experts E_0..E_{n-1}, K = 2, y = sum_{i<n} G(x)_i SwiGLU_i(x).

Readings where the pages are silent or disagree:
  * TopK ties: the lower expert index ranks first (for every position).
  * slot order: slot 0 holds the larger logit, slot 1 the smaller.
  * weight naming: the pages write the expert in column-vector form with
    W_1, W_2 the two up projections and W_3 the down projection.  This code
    uses row-vector form x . W with W1 (SiLU branch) and W3 (linear branch) of
    shape [E, d, f] and W2 (down) of shape [E, f, d]:
    E_i(x) = (SiLU(x W1[i]) (.) (x W3[i])) W2[i].  Same function after
    renaming and transposition.
  * RMSNorm: unit gain, eps = 1e-5 (neither is given).

Every function is pinned by ``tests/test_oracle.py`` against closed forms,
library routines, brute force and a hand-derived worked example.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


def f64(a) -> np.ndarray:
    """Exact float64 copy of a NumPy array or torch tensor (bf16/fp16/fp32/fp64)."""
    if hasattr(a, "detach"):
        import torch
        a = a.detach().to("cpu", torch.float64).numpy()
    return np.asarray(a, dtype=np.float64)


# ---------------------------------------------------------------------------
# Router  [GU-3.4 gating function; GU-TOPK; XYZ-M]
# ---------------------------------------------------------------------------
def router_logits(x, Wg) -> np.ndarray:
    """l = x . W_g for every token; W_g is [d, n]; no bias term [GU-TOPK]."""
    return f64(x) @ f64(Wg)


def topk_indices(logits: np.ndarray, K: int) -> np.ndarray:
    """Indices of the K largest logits of each token, largest first [GU-TOPK step 1].

    Ordering key per expert i: (-l_i, i), so equal logits rank by lower index."""
    T, E = logits.shape
    expert_ids = np.broadcast_to(np.arange(E), (T, E))
    order = np.lexsort((expert_ids, -logits), axis=1)   # primary key: -l, then index
    return order[:, :K].astype(np.int32)


def topk_mask(logits: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """TopK(l): l_i for the selected experts, -inf elsewhere [GU-3.4 TopK definition; GU-TOPK step 2]."""
    masked = np.full_like(logits, -np.inf)
    rows = np.arange(logits.shape[0])[:, None]
    masked[rows, idx] = logits[rows, idx]
    return masked


def softmax(v: np.ndarray) -> np.ndarray:
    """Softmax over the last axis, exp(-inf) = 0 [GU-TOPK step 3]."""
    m = v.max(axis=-1, keepdims=True)
    e = np.exp(v - m)
    return e / e.sum(axis=-1, keepdims=True)


@dataclass
class Gating:
    logits: np.ndarray   # [T, n]  float64
    idx: np.ndarray      # [T, K]  int32, slot 0 = larger logit
    gate: np.ndarray     # [T, K]  float64, G(x) at idx
    G: np.ndarray        # [T, n]  float64 dense gate vector (zeros off the top-K)


def gating(x, Wg, K: int) -> Gating:
    """G(x) = Softmax(TopK(x . W_g)) [GU-3.4]."""
    logits = router_logits(x, Wg)
    idx = topk_indices(logits, K)
    G = softmax(topk_mask(logits, idx))
    gate = np.take_along_axis(G, idx.astype(np.int64), axis=1)
    return Gating(logits, idx, gate, G)


# ---------------------------------------------------------------------------
# Experts  [GU-SWIGLU]
# ---------------------------------------------------------------------------
def silu(z: np.ndarray) -> np.ndarray:
    """SiLU(z) = z . sigma(z) = z / (1 + exp(-z))."""
    return z / (1.0 + np.exp(-z))


def expert(x, W1e, W3e, W2e) -> np.ndarray:
    """E_i(x) = (SiLU(x W1[i]) (.) (x W3[i])) W2[i], row-vector form."""
    x = f64(x)
    return (silu(x @ f64(W1e)) * (x @ f64(W3e))) @ f64(W2e)


# ---------------------------------------------------------------------------
# Layer  [GU-3.4 output combination; XYZ-M]
# ---------------------------------------------------------------------------
@dataclass
class LayerResult:
    y: np.ndarray        # [T, d] float64
    gating: Gating


def moe_layer(x, Wg, W1, W3, W2, K: int) -> LayerResult:
    """y = sum_i G(x)_i . E_i(x), evaluating each expert only on the tokens
    that selected it (the other experts perform no computation) [GU-3.4]."""
    x64 = f64(x)
    g = gating(x64, Wg, K)
    E = g.G.shape[1]
    d_out = W2.shape[2]
    y = np.zeros((x64.shape[0], d_out))
    for e in range(E):
        rows = np.nonzero((g.idx == e).any(axis=1))[0]
        if rows.size == 0:
            continue
        y[rows] += g.G[rows, e][:, None] * expert(x64[rows], W1[e], W3[e], W2[e])
    return LayerResult(y, g)


def moe_layer_dense(x, Wg, W1, W3, W2, K: int) -> LayerResult:
    """Brute force: every expert on every token, y = sum_{i<n} G(x)_i . E_i(x),
    with G zero off the top-K [GU-3.4; XYZ-M].  Tiny inputs only."""
    x64 = f64(x)
    g = gating(x64, Wg, K)
    y = np.zeros((x64.shape[0], W2.shape[2]))
    for e in range(g.G.shape[1]):
        y += g.G[:, e][:, None] * expert(x64, W1[e], W3[e], W2[e])
    return LayerResult(y, g)


def moe_layer_tokens(x, Wg, W1, W3, W2, K: int, tokens) -> LayerResult:
    """The layer on a subset of tokens.  Each token's output depends on that
    token alone [GU-3.4: the router and the experts act per token], so this is
    the full layer's output restricted to ``tokens``."""
    tokens = np.asarray(tokens, dtype=np.int64)
    return moe_layer(f64(x)[tokens], Wg, W1, W3, W2, K)


# ---------------------------------------------------------------------------
# Grouping tokens by expert  [GU-INFRA; GU-3.4 sparse execution]
# ---------------------------------------------------------------------------
@dataclass
class Permutation:
    counts: np.ndarray     # [n]     int64, tokens per expert
    offsets: np.ndarray    # [n+1]   int64, exclusive prefix sum of counts
    perm_tok: np.ndarray   # [T*K]   int32, token id of each grouped row
    perm_k: np.ndarray     # [T*K]   int32, which slot (0..K-1) of that token
    pos: np.ndarray        # [T, K]  int32, grouped row of (token, slot)


def permutation(idx: np.ndarray, E: int) -> Permutation:
    """Stable counting sort of the flat (token, slot) list, taken in t*K + k
    order and keyed by the expert idx[t, k]: within one expert, rows keep
    ascending (token, slot) order."""
    idx = np.asarray(idx)
    T, K = idx.shape
    counts = np.zeros(E, dtype=np.int64)
    for e in range(E):
        counts[e] = int((idx == e).sum())
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    cursor = offsets[:-1].copy()
    perm_tok = np.empty(T * K, dtype=np.int32)
    perm_k = np.empty(T * K, dtype=np.int32)
    pos = np.empty((T, K), dtype=np.int32)
    for t in range(T):
        for k in range(K):
            e = int(idx[t, k])
            r = cursor[e]
            cursor[e] += 1
            perm_tok[r] = t
            perm_k[r] = k
            pos[t, k] = r
    return Permutation(counts, offsets, perm_tok, perm_k, pos)


# ---------------------------------------------------------------------------
# Transformer-block wrapper for the attention-free stack  [GU-ARCH]
# ---------------------------------------------------------------------------
RMS_EPS = 1e-5


def rmsnorm(h, eps: float = RMS_EPS) -> np.ndarray:
    """RMSNorm with unit gain: h / sqrt(mean(h^2) + eps), per row."""
    h = f64(h)
    return h / np.sqrt(np.mean(h * h, axis=1, keepdims=True) + eps)


def moe_block(h, Wg, W1, W3, W2, K: int, eps: float = RMS_EPS) -> np.ndarray:
    """One pre-norm MoE half-block: h + MoE(RMSNorm(h))."""
    h64 = f64(h)
    return h64 + moe_layer(rmsnorm(h64, eps), Wg, W1, W3, W2, K).y


# ---------------------------------------------------------------------------
# Backward pass  [GU section 3 information flow and "Top-K Gating Mechanism
# and Routing": gradients flow only through the selected experts and their
# logits; the choice of experts itself is piecewise constant]
# ---------------------------------------------------------------------------
@dataclass
class LayerGrads:
    dx: np.ndarray       # [T, d]
    dWg: np.ndarray      # [d, n]
    dW1: np.ndarray      # [n, d, f]
    dW3: np.ndarray      # [n, d, f]
    dW2: np.ndarray      # [n, f, d]
    dlogits: np.ndarray  # [T, n]


def dsilu(z: np.ndarray) -> np.ndarray:
    """d/dz SiLU(z) = sigma(z) (1 + z (1 - sigma(z)))."""
    sg = 1.0 / (1.0 + np.exp(-z))
    return sg * (1.0 + z * (1.0 - sg))


def softmax_backward(G: np.ndarray, dG: np.ndarray) -> np.ndarray:
    """Gradient of the logits for G = softmax over the kept logits (zero
    elsewhere): dl_i = G_i (dG_i - sum_j G_j dG_j), zero off the kept set."""
    return G * (dG - np.sum(G * dG, axis=1, keepdims=True))


def moe_layer_backward(x, Wg, W1, W3, W2, K: int, dy) -> LayerGrads:
    """Gradients of L = <dy, y> for y = moe_layer(x, ...), by the chain rule
    through y = sum_i G_i E_i(x): each selected expert's SwiGLU, the gates
    G = softmax over the kept logits (zero elsewhere), and the router
    l = x W_g.  The selected set is held fixed (it has no gradient)."""
    x64 = f64(x)
    dy64 = f64(dy)
    Wg64 = f64(Wg)
    g = gating(x64, Wg64, K)
    T, d = x64.shape
    E = g.G.shape[1]
    f = W1.shape[2]
    dx = np.zeros((T, d))
    dW1 = np.zeros((E, d, f))
    dW3 = np.zeros((E, d, f))
    dW2 = np.zeros((E, f, d))
    dG = np.zeros((T, E))
    for e in range(E):
        rows = np.nonzero((g.idx == e).any(axis=1))[0]
        if rows.size == 0:
            continue
        W1e, W3e, W2e = f64(W1[e]), f64(W3[e]), f64(W2[e])
        xe = x64[rows]
        a = xe @ W1e
        b = xe @ W3e
        s = silu(a)
        H = s * b
        ye = H @ W2e                                   # E_e(x) on its tokens
        dG[rows, e] = np.sum(dy64[rows] * ye, axis=1)  # dL/dG_e
        dye = g.G[rows, e][:, None] * dy64[rows]       # dL/dE_e(x)
        dW2[e] = H.T @ dye
        dH = dye @ W2e.T
        da = dH * b * dsilu(a)
        db = dH * s
        dW1[e] = xe.T @ da
        dW3[e] = xe.T @ db
        dx[rows] += da @ W1e.T + db @ W3e.T
    dl = softmax_backward(g.G, dG)
    dx += dl @ Wg64.T
    return LayerGrads(dx, x64.T @ dl, dW1, dW3, dW2, dl)


# ---------------------------------------------------------------------------
# Near-tie bookkeeping for parity checks (float64 logits)
# ---------------------------------------------------------------------------
def logit_gaps(logits: np.ndarray, K: int):
    """Per token: gap between the K-th and (K+1)-th largest logit, and between
    the 1st and 2nd (for K = 2).  Both are +inf where undefined."""
    s = -np.sort(-logits, axis=1)
    T, E = logits.shape
    gap_in_out = s[:, K - 1] - s[:, K] if E > K else np.full(T, np.inf)
    gap_12 = s[:, 0] - s[:, 1] if (K >= 2 and E >= 2) else np.full(T, np.inf)
    return gap_in_out, gap_12
