"""Comparison helpers: CUDA path vs the float64 oracle.

Criteria
  * expert indices: bit-exact, except tokens whose oracle gap between the K-th
    and (K+1)-th logit is in (0, 1e-3) (counted, reported, exempt) and tokens
    whose top-1/top-2 gap is below 1e-3 (compared as a set).  Exact ties (gap
    exactly 0 by construction) are NOT exempt: they test the lower-index rule.
  * grouping (perm_tok, offsets, pos): bit-exact against the oracle's stable
    counting sort applied to the GPU's own indices, always; and against the
    oracle's own grouping when no token is exempt.
  * outputs: max|y_gpu - y_ref| / (max|y_ref| + 1e-6) <= 2e-2 (bf16) or 1e-4 (fp32).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

import oracle

TOL = {"bf16": 2e-2, "f32": 1e-4}
NEAR_TIE = 1e-3


def rel_linf(y_gpu, y_ref) -> float:
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    return float(np.abs(y_gpu - y_ref).max() / (np.abs(y_ref).max() + 1e-6)) if y_ref.size else 0.0


@dataclass
class RoutingReport:
    n_tokens: int
    n_exempt_in_out: int
    n_set_compared: int
    n_mismatch: int
    gate_max_abs_err: float


def check_routing(idx_gpu, gate_gpu, g: "oracle.Gating", K: int) -> RoutingReport:
    """Compare GPU indices/gates with the oracle's gating on the same tokens."""
    idx_gpu = np.asarray(idx_gpu)
    gate_gpu = np.asarray(gate_gpu, dtype=np.float64)
    gap_io, gap_12 = oracle.logit_gaps(g.logits, K)
    exempt = (gap_io > 0) & (gap_io < NEAR_TIE)
    set_cmp = (~exempt) & (gap_12 < NEAR_TIE) if K >= 2 else np.zeros_like(exempt)
    mism = 0
    for t in range(idx_gpu.shape[0]):
        if exempt[t]:
            continue
        if set_cmp[t]:
            if set(idx_gpu[t].tolist()) != set(g.idx[t].tolist()):
                mism += 1
        elif idx_gpu[t].tolist() != g.idx[t].tolist():
            mism += 1
    ok = ~exempt & ~set_cmp
    gerr = float(np.abs(gate_gpu[ok] - g.gate[ok]).max()) if ok.any() else 0.0
    return RoutingReport(int(idx_gpu.shape[0]), int(exempt.sum()), int(set_cmp.sum()), mism, gerr)


def check_grouping(idx_gpu, perm_gpu, offsets_gpu, pos_gpu, E: int) -> None:
    """GPU grouping must equal the oracle's stable sort of the GPU's own indices."""
    p = oracle.permutation(np.asarray(idx_gpu), E)
    assert np.array_equal(np.asarray(offsets_gpu), p.offsets), "offsets differ"
    assert np.array_equal(np.asarray(perm_gpu), p.perm_tok), "perm_tok differs"
    assert np.array_equal(np.asarray(pos_gpu), p.pos), "pos differs"


def gate_invariants(idx_gpu, gate_gpu, E: int, K: int) -> None:
    idx_gpu = np.asarray(idx_gpu)
    gate_gpu = np.asarray(gate_gpu, dtype=np.float64)
    assert (idx_gpu >= 0).all() and (idx_gpu < E).all()
    for t in range(idx_gpu.shape[0]):
        assert len(set(idx_gpu[t].tolist())) == K
    assert (gate_gpu >= 0).all()
    assert np.abs(gate_gpu.sum(axis=1) - 1.0).max() <= 2e-7
    if K == 2:
        assert (gate_gpu[:, 0] >= gate_gpu[:, 1]).all()


def half_ulp(v, dtype: str) -> np.ndarray:
    """Half a unit in the last place of each value as stored in ``dtype``
    (bf16: 8 significant bits, fp32: 24), i.e. the largest error of one
    round-to-nearest into that type."""
    bits = {"bf16": 8, "f32": 24}[dtype]
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - bits), 0.0)


def residual_rel_err(h_new, h_prev, y_ref, dtype: str) -> float:
    """Error of a residual update h_new = round(h_prev + y) against the oracle's
    y, relative to max|y_ref| like rel_linf, after removing the one rounding
    of the sum into the storage type (which the MoE output is not charged for)."""
    h_new = np.asarray(h_new, dtype=np.float64)
    dev = np.abs(h_new - np.asarray(h_prev, dtype=np.float64) - np.asarray(y_ref, dtype=np.float64))
    excess = np.maximum(dev - half_ulp(h_new, dtype), 0.0)
    return float(excess.max() / (np.abs(y_ref).max() + 1e-6)) if dev.size else 0.0
