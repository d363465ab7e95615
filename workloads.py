"""Seeded synthetic inputs for the Mixtral-shaped sparse-MoE feed-forward layer.

This module holds random-number recipes and tensor shapes only: no routing,
expert or combine arithmetic lives here.  The CUDA path's tests and benchmark
and the float64 oracle both take their inputs from these functions, so the two
sides always see the same bits.

Conventions
  * every tensor comes from its own ``torch.Generator`` seeded from
    ``(base seed, tensor tag)``, drawn as fp32 ``torch.randn`` and then rounded
    to the target dtype (round-to-nearest-even);
  * ``N(0, 1/d)`` means variance 1/d, ``N(0, 0.02)`` means standard deviation
    0.02 (the usual initialisation convention);
  * "RMS-normalised rows" means ``z / sqrt(mean(z^2) + 1e-5)`` per row of
    ``z ~ N(0, 1)`` in fp32, then rounded;
  * large weight banks can be drawn directly on a CUDA device (Philox); small
    cases are drawn on the CPU.

Shapes are Mixtral's (model dimension 4096, expert hidden dimension 14336,
8 experts, top-2), from the Mixtral of Experts summary pages ("Expert Network
Structure (SwiGLU)" and the router description in "3.4 MoE Layer Formulation").
"""
from __future__ import annotations

import json
import math
import pathlib
from dataclasses import dataclass, field

import torch

BASE_SEED = 55
MIXTRAL = dict(d=4096, f=14336, E=8, K=2)
GOLDEN_DIR = pathlib.Path(__file__).resolve().parent / "tests" / "golden"

# Tensor tags: one generator stream per tensor so subsets can be regenerated.
_TAG = {"x": 1, "Wg": 2, "W1": 3, "W3": 4, "W2": 5, "tie": 6, "h0": 7, "trace": 8}


def _seed(seed: int, tag: str, sub: int = 0) -> int:
    return (int(seed) * 1_000_003 + _TAG[tag] * 10_007 + int(sub)) % (2**62)


def randn(shape, std: float, seed: int, device="cpu", dtype=torch.float32) -> torch.Tensor:
    """N(0, std^2) drawn in fp32 from a generator seeded with ``seed``, then cast."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    t = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def rms_rows(T: int, d: int, seed: int, device="cpu", dtype=torch.bfloat16, eps=1e-5) -> torch.Tensor:
    """Rows of N(0,1) scaled to unit root-mean-square, then cast."""
    z = randn((T, d), 1.0, seed, device)
    z.mul_(torch.rsqrt(z.pow(2).mean(dim=1, keepdim=True) + eps))
    return z.to(dtype)


@dataclass
class MoEInputs:
    """One MoE layer's inputs: x [T,d], Wg [d,E], W1/W3 [E,d,f], W2 [E,f,d], top-K."""
    x: torch.Tensor
    Wg: torch.Tensor
    W1: torch.Tensor
    W3: torch.Tensor
    W2: torch.Tensor
    K: int
    meta: dict = field(default_factory=dict)

    @property
    def shape(self):
        T, d = self.x.shape
        E, _, f = self.W1.shape
        return T, d, f, E, self.K

    def to(self, device):
        return MoEInputs(self.x.to(device), self.Wg.to(device), self.W1.to(device),
                         self.W3.to(device), self.W2.to(device), self.K, dict(self.meta))


def param_counts(d: int, f: int, E: int, layers: int = 1) -> dict:
    """Parameter counts implied by the tensor shapes this module produces."""
    per_expert = 3 * d * f          # W1[e], W3[e]: d*f each; W2[e]: f*d
    return {"per_expert": per_expert, "per_layer_experts": E * per_expert,
            "all_layers_experts": layers * E * per_expert, "router_per_layer": d * E,
            "router_all_layers": layers * d * E}


# ---------------------------------------------------------------------------
# config "tiny_fp32": T=64, d=64, f=128, E=8, K=2, fp32
# ---------------------------------------------------------------------------
def tiny_fp32(T=64, d=64, f=128, E=8, K=2, seed=BASE_SEED, device="cpu") -> MoEInputs:
    """x ~ N(0,1); Wg ~ N(0,1/d); W1, W3 ~ N(0,1/d); W2 ~ N(0,1/f); all fp32, one seed."""
    return MoEInputs(
        x=randn((T, d), 1.0, _seed(seed, "x"), device),
        Wg=randn((d, E), d ** -0.5, _seed(seed, "Wg"), device),
        W1=randn((E, d, f), d ** -0.5, _seed(seed, "W1"), device),
        W3=randn((E, d, f), d ** -0.5, _seed(seed, "W3"), device),
        W2=randn((E, f, d), f ** -0.5, _seed(seed, "W2"), device),
        K=K, meta={"config": "tiny_fp32", "seed": seed})


# ---------------------------------------------------------------------------
# Mixtral-shaped weights (shared by prefill, decode and skew)
# ---------------------------------------------------------------------------
W13_STD = 0.02
W2_STD = 0.02 / math.sqrt(2 * 32)


def mixtral_weights(d=4096, f=14336, E=8, seed=BASE_SEED, device="cpu", dtype=torch.bfloat16):
    """Wg ~ N(0,1/d); W1, W3 ~ N(0, std 0.02); W2 ~ N(0, std 0.02/sqrt(2*32)).

    Expert banks are drawn one expert at a time (bounded fp32 scratch)."""
    Wg = randn((d, E), d ** -0.5, _seed(seed, "Wg"), device, dtype)
    W1 = torch.empty((E, d, f), dtype=dtype, device=device)
    W3 = torch.empty((E, d, f), dtype=dtype, device=device)
    W2 = torch.empty((E, f, d), dtype=dtype, device=device)
    for e in range(E):
        W1[e] = randn((d, f), W13_STD, _seed(seed, "W1", e), device, dtype)
        W3[e] = randn((d, f), W13_STD, _seed(seed, "W3", e), device, dtype)
        W2[e] = randn((f, d), W2_STD, _seed(seed, "W2", e), device, dtype)
    return Wg, W1, W3, W2


def prefill(T=4096, d=4096, f=14336, E=8, K=2, seed=BASE_SEED, device="cpu",
            dtype=torch.bfloat16, weights=None) -> MoEInputs:
    """Mixtral prefill layer: RMS-normalised rows, near-uniform routing."""
    Wg, W1, W3, W2 = weights if weights is not None else mixtral_weights(d, f, E, seed, device, dtype)
    x = rms_rows(T, d, _seed(seed, "x", 0), device, dtype)
    return MoEInputs(x, Wg, W1, W3, W2, K, {"config": "prefill", "seed": seed})


def decode(T: int, d=4096, f=14336, E=8, K=2, seed=BASE_SEED, device="cpu",
           dtype=torch.bfloat16, weights=None) -> MoEInputs:
    """Decode batch of T tokens: prefill weights (same seed), independent x seed per T."""
    Wg, W1, W3, W2 = weights if weights is not None else mixtral_weights(d, f, E, seed, device, dtype)
    x = rms_rows(T, d, _seed(seed, "x", 1000 + T), device, dtype)
    return MoEInputs(x, Wg, W1, W3, W2, K, {"config": f"decode{T}", "seed": seed})


# ---------------------------------------------------------------------------
# config "skew": Zipf(1.2) expert loads through a constant bias feature, plus
# tokens whose logits tie exactly.
# ---------------------------------------------------------------------------
ZIPF_S = 1.2
TIE_FRACTION = 0.01
# Designed logit vectors for the tie tokens, all multiples of 1/32 (exact in
# bf16 and fp32).  Expected (slot 0, slot 1) under "lower index wins ties":
#   P0: unique top-1 = 3, 2nd/3rd tie between 1 and 5       -> (3, 1)
#   P1: unique top-1 = 0, 2nd/3rd tie between 6 and 7       -> (0, 6)
#   P2: three-way tie for the top between 2, 4 and 6        -> (2, 4)
#   P3: tie for the top between 5 and 7, third lower        -> (5, 7)
TIE_PATTERNS = [
    [-1.0, 1.0, -0.5, 2.0, -1.5, 1.0, -2.0, 0.0],
    [1.5, -1.0, 0.0, -0.25, -1.0, 0.0, 0.5, 0.5],
    [0.0, -1.0, 1.0, -1.0, 1.0, 0.25, 1.0, -2.0],
    [-0.5, 0.0, 0.75, -1.0, 0.0, 1.25, 0.5, 1.25],
]
TIE_EXPECTED = [(3, 1), (0, 6), (2, 4), (5, 7)]


def zipf_shares(E=8, s=ZIPF_S):
    w = [(k + 1) ** -s for k in range(E)]
    tot = sum(w)
    return [v / tot for v in w]


def skew_bias(d: int, E: int) -> list:
    """Per-expert logit bias (multiples of 1/32) read from the committed fixture."""
    data = json.loads((GOLDEN_DIR / "skew_bias.json").read_text())
    key = f"d{d}_E{E}"
    if key not in data["beta"]:
        raise KeyError(f"no calibrated skew bias for {key}; run tests/golden/make_skew_bias.py")
    return data["beta"][key]


def skew_features(d: int):
    """Feature columns reserved in the skew config: bias feature, then tie features."""
    return {"bias": d - 1, "tie": [d - 2 - j for j in range(len(TIE_PATTERNS))]}


def skew(T=16384, d=4096, f=14336, E=8, K=2, seed=BASE_SEED, device="cpu", dtype=torch.bfloat16,
         weights=None, beta=None, n_tie=None) -> MoEInputs:
    """Skewed routing through a constant bias feature; ~1% exactly tied tokens.

    * every normal token: RMS-normalised row, tie features zeroed, bias feature = 1;
    * Wg: N(0,1/d), bias row = beta, tie row j = TIE_PATTERNS[j] - beta;
    * tie token: zeros except bias feature = 1 and tie feature j = 1, so its
      logits are exactly TIE_PATTERNS[j] in any summation order.
    The expert banks are the prefill banks (same seed) unless given."""
    assert E == 8 and K == 2, "tie patterns are written for 8 experts, top-2"
    if beta is None:
        beta = skew_bias(d, E)
    beta_t = torch.tensor(beta, dtype=torch.float32)
    if weights is None:
        _, W1, W3, W2 = mixtral_weights(d, f, E, seed, device, dtype)
    else:
        _, W1, W3, W2 = weights
    feats = skew_features(d)
    Wg = randn((d, E), d ** -0.5, _seed(seed, "Wg", 77), "cpu", torch.float32)
    Wg[feats["bias"]] = beta_t
    for j, r in enumerate(feats["tie"]):
        Wg[r] = torch.tensor(TIE_PATTERNS[j], dtype=torch.float32) - beta_t
    Wg = Wg.to(dtype).to(device)

    x = rms_rows(T, d, _seed(seed, "x", 77), device, torch.float32)
    x[:, feats["tie"]] = 0.0
    x[:, feats["bias"]] = 1.0
    if n_tie is None:
        n_tie = int(round(TIE_FRACTION * T))
    g = torch.Generator(device="cpu")
    g.manual_seed(_seed(seed, "tie"))
    tie_tok = torch.randperm(T, generator=g)[:n_tie].sort().values
    tie_pat = torch.arange(n_tie) % len(TIE_PATTERNS)
    if n_tie:
        tt = tie_tok.to(device)
        x[tt] = 0.0
        x[tt, feats["bias"]] = 1.0
        cols = torch.tensor(feats["tie"], device=device)[tie_pat.to(device)]
        x[tt, cols] = 1.0
    x = x.to(dtype)
    return MoEInputs(x, Wg, W1, W3, W2, K, {
        "config": "skew", "seed": seed, "beta": list(beta), "tie_tokens": tie_tok.tolist(),
        "tie_patterns": tie_pat.tolist()})


# ---------------------------------------------------------------------------
# config "stack32": 32 attention-free layers h <- h + MoE_l(RMSNorm(h))
# ---------------------------------------------------------------------------
def stack_layer_seed(l: int, seed=BASE_SEED) -> int:
    return seed + 1000 + l


def stack_h0(T=8192, d=4096, seed=BASE_SEED, device="cpu", dtype=torch.bfloat16):
    """h0 ~ N(0,1)."""
    return randn((T, d), 1.0, _seed(seed, "h0"), device, dtype)


def stack_layer_weights(l: int, d=4096, f=14336, E=8, seed=BASE_SEED, device="cpu", dtype=torch.bfloat16):
    return mixtral_weights(d, f, E, stack_layer_seed(l, seed), device, dtype)


# ---------------------------------------------------------------------------
# decode traces with temporal locality (expert cache)
# ---------------------------------------------------------------------------
# The pages' routing analysis (Table 5) reports that consecutive tokens share
# their first or second expert 61.6-67.0% of the time at layer 15, against
# ~46% for independent choices (1 - C(6,2)/C(8,2) = 46.4% for 8 experts, top
# 2).  A chain that keeps the previous step's expert pair with probability
# `keep` and otherwise draws a uniform pair shares one with probability
# keep + (1 - keep) * 0.464; keep = 0.35 gives 65%.
TRACE_KEEP = 0.35
TRACE_STEER = 5.0


def decode_trace(steps: int, Wg: torch.Tensor, T: int = 1, keep: float = TRACE_KEEP, seed=BASE_SEED,
                 device="cpu", dtype=torch.bfloat16, steer: float = TRACE_STEER):
    """Token rows for `steps` decode steps of T tokens each ([steps, T, d]).

    Each of the T token streams walks a Markov chain over expert pairs
    (above); its token at a step is z + steer * (u_a + u_b), RMS-normalised,
    with z ~ N(0, I) and u_e = Wg[:, e] / |Wg[:, e]|^2, which raises the
    logits of experts a and b by about `steer` over N(0, 1) noise, so the
    router mostly picks the chain's pair.  Returns (x, pairs) with pairs
    [steps, T, 2] the chain's intended experts (the router decides the
    actual ones)."""
    d, E = Wg.shape
    g = torch.Generator(device="cpu")
    g.manual_seed(_seed(seed, "trace", T))
    pairs = torch.empty((steps, T, 2), dtype=torch.long)
    for t in range(T):
        cur = torch.randperm(E, generator=g)[:2]
        for i in range(steps):
            if i > 0 and torch.rand((), generator=g).item() >= keep:
                cur = torch.randperm(E, generator=g)[:2]
            pairs[i, t] = cur
    W = Wg.detach().to("cpu", torch.float32)
    U = W / (W * W).sum(dim=0, keepdim=True)
    z = randn((steps * T, d), 1.0, _seed(seed, "trace", 10_000 + T), "cpu")
    flat = pairs.reshape(-1, 2)
    x = z + steer * (U[:, flat[:, 0]].T + U[:, flat[:, 1]].T)
    x = x * torch.rsqrt(x.pow(2).mean(dim=1, keepdim=True) + 1e-5)
    return x.reshape(steps, T, d).to(device=device, dtype=dtype), pairs
