"""Per-layer check of the attention-free MoE stack h <- h + MoE_l(RMSNorm(h)),
teacher-forced: each layer is compared with the oracle on the GPU's own input
to that layer, so errors do not compound across layers."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from tests import parity


def _np(t):
    return t.detach().cpu().numpy()


def check_stack_layer(moe, h, weights, K, toks, ws, tol_key: str, eps: float = 1e-5):
    """Advance h by one block with moe_block_forward and check, on the sample
    ``toks``: RMSNorm against the oracle; routing of every token (bit-exact
    indices outside near-ties, stable grouping); the layer output y of
    moe_forward on the normalised input against the oracle; the residual
    update against h_prev + y_oracle up to one rounding into the storage
    type; and that the block call equals the two-call sequence bit for bit.
    Returns (rel err of y, rel err of the residual update, routing report)."""
    Wg, W1, W3, W2 = weights
    T, d = h.shape
    E = Wg.shape[1]
    toks_t = torch.as_tensor(toks, device=h.device)
    h_prev = h.clone()
    xn = moe.moe_rmsnorm(h_prev, eps=eps)
    # RMSNorm: within one rounding of the storage type, plus the fp32 error of
    # the row's mean of squares (per-thread partial sums over d/256 terms and a
    # tree over 256 threads: well under 4e-6 relative for d <= 4096)
    xn_s = oracle.f64(xn[toks_t])
    ref_n = oracle.rmsnorm(h_prev[toks_t], eps)
    assert (np.abs(xn_s - ref_n) <= parity.half_ulp(ref_n, tol_key) + 4e-6 * np.abs(ref_n)).all()
    # routing of every token, on the GPU's normalised input
    idx, gate, perm, offs, pos = moe.moe_route(xn, Wg, K)
    g = oracle.gating(xn.cpu(), Wg.cpu(), K)
    rep = parity.check_routing(_np(idx), _np(gate), g, K)
    assert rep.n_mismatch == 0, rep
    parity.gate_invariants(_np(idx), _np(gate), E, K)
    parity.check_grouping(_np(idx), _np(perm), _np(offs), _np(pos), E)
    # the layer output on the sample
    y = moe.moe_forward(xn, Wg, W1, W3, W2, K, workspace=ws)
    y_ref = oracle.moe_layer(xn_s, Wg, W1, W3, W2, K).y
    err_y = parity.rel_linf(_np(y[toks_t].float()), y_ref)
    assert err_y <= parity.TOL[tol_key], err_y
    # the block (RMSNorm + MoE accumulated into h) and the residual update
    moe.moe_block_forward(h, Wg, W1, W3, W2, K, eps=eps, workspace=ws)
    assert moe.moe_read_status(ws) == 0
    h_two = h_prev.clone()
    moe.moe_forward(xn, Wg, W1, W3, W2, K, y=h_two, workspace=ws, flags=moe.MOE_ACCUMULATE)
    assert torch.equal(h, h_two)
    err_h = parity.residual_rel_err(_np(h[toks_t].float()), _np(h_prev[toks_t].float()), y_ref, tol_key)
    assert err_h <= parity.TOL[tol_key], err_h
    return err_y, err_h, rep
