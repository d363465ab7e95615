"""Write skew_bias.json: the per-expert logit bias of the skewed-routing config.

The skewed config wants expert loads (shares of all top-2 assignments) to
follow Zipf(s = 1.2) over 8 experts.  The router has no bias term, so the bias
rides on a constant input feature whose W_g row holds it.  This script
calibrates that row on a held-out token sample with the float64 oracle's
router (logits, top-2 with lower-index ties) and stores it, quantised to
multiples of 1/32 so it is exact in bf16.  It calls only the oracle and the
seeded input generators.

    python tests/golden/make_skew_bias.py
"""
from __future__ import annotations

import json
import pathlib
import sys

import numpy as np

ROOT = pathlib.Path(__file__).resolve().parents[2]
sys.path.insert(0, str(ROOT))

import oracle  # noqa: E402
import workloads as W  # noqa: E402

OUT = pathlib.Path(__file__).resolve().parent / "skew_bias.json"
HELD_OUT_SEED = 5501
SAMPLE_T = 16384


def shares_for(base_logits: np.ndarray, beta: np.ndarray, K: int) -> np.ndarray:
    idx = oracle.topk_indices(base_logits + beta[None, :], K)
    E = base_logits.shape[1]
    return np.bincount(idx.ravel(), minlength=E) / idx.size


def calibrate(d: int, f: int, E: int = 8, K: int = 2, iters: int = 300):
    zero = [0.0] * E
    # Held-out tokens with the bias row set to zero, no tie tokens: the base
    # logits are then exactly x . W_g without the bias feature's contribution.
    inp = W.skew(T=SAMPLE_T, d=d, f=8, E=E, K=K, seed=HELD_OUT_SEED, beta=zero, n_tie=0,
                 weights=(None, None, None, None))
    # Use the real config's W_g (same construction, base seed) for the logits.
    ref = W.skew(T=8, d=d, f=8, E=E, K=K, beta=zero, n_tie=0, weights=(None, None, None, None))
    base = oracle.router_logits(inp.x, ref.Wg)
    target = np.array(W.zipf_shares(E))
    beta = np.zeros(E)
    for _ in range(iters):
        s = shares_for(base, beta, K)
        beta += 0.5 * (np.log(target) - np.log(np.maximum(s, 1e-6)))
        beta -= beta.mean()
    beta_q = np.round(beta * 32.0) / 32.0
    beta_q = np.clip(beta_q, -4.0, 4.0)
    realised = shares_for(base, beta_q, K)
    return beta_q, realised, target


def main():
    data = {"_about": __doc__.strip().splitlines()[0], "zipf_s": W.ZIPF_S,
            "sample_tokens": SAMPLE_T, "held_out_seed": HELD_OUT_SEED, "beta": {}, "realised_shares": {},
            "target_shares": {}}
    for d in (4096, 512):
        beta, realised, target = calibrate(d, 8)
        key = f"d{d}_E8"
        data["beta"][key] = [float(b) for b in beta]
        data["realised_shares"][key] = [round(float(s), 4) for s in realised]
        data["target_shares"][key] = [round(float(s), 4) for s in target]
        print(key, "beta", beta.tolist())
        print("  realised", np.round(realised, 4).tolist())
        print("  target  ", np.round(target, 4).tolist())
    OUT.write_text(json.dumps(data, indent=1) + "\n")
    print("wrote", OUT)


if __name__ == "__main__":
    main()
