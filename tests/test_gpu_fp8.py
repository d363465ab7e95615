"""GPU parity of the e4m3-weight variant against the float64 oracle
(oracle/fp8_oracle.py): weight quantisation bit for bit; the layer within the
bf16 bar on ragged shapes, both GEMM forms, decode sizes with split down
projections, top-1, and at full Mixtral size for a one-token decode.  All
calls go through the C ABI."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import oracle.fp8_oracle as F8
import workloads as W
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe(cuda_device):
    from sparse_mixture_experts_55_b300 import build
    build.build()
    import sparse_mixture_experts_55_b300 as m
    return m


def _np(t):
    return t.detach().cpu().numpy()


def _codes(Wq, N, K):
    """The tiled e4m3 codes as an [E, N, K] uint8 array (padding dropped)."""
    E, nt, kt = Wq.shape[:3]
    return _np(Wq.view(torch.uint8).permute(0, 1, 3, 2, 4).reshape(E, nt * 128, kt * 128)[:, :N, :K])


@pytest.mark.parametrize("E,K,N", [(3, 64, 96), (2, 200, 72), (1, 4096, 128)])
def test_weight_quantisation_bit_exact(moe, E, K, N):
    Wb = W.randn((E, K, N), 0.02, 77 + K, "cpu", torch.bfloat16)
    Wb[0, :, 5] = 0                                   # an all-zero column: scale 1
    Wq, s = moe.quantize_weights_fp8(Wb.cuda())
    q_ref, s_ref = F8.quantize_weight_columns(Wb)
    assert np.array_equal(_np(s), s_ref)
    assert np.array_equal(_codes(Wq, N, K), q_ref)
    # the tiles' padding past N and K holds zero codes
    full = _np(Wq.view(torch.uint8).permute(0, 1, 3, 2, 4).reshape(E, Wq.shape[1] * 128, Wq.shape[2] * 128))
    assert not full[:, N:, :].any() and not full[:, :, K:].any()


def _fp8_case(T, d, f, E, K, seed):
    Wg, W1, W3, W2 = W.mixtral_weights(d, f, E, seed=seed, device="cpu")
    x = W.rms_rows(T, d, seed * 7 + 1, "cpu", torch.bfloat16)
    return x, Wg, W1, W3, W2


def _check_fp8_layer(moe, T, d, f, E, K, seed, tol=2e-2):
    x, Wg, W1, W3, W2 = _fp8_case(T, d, f, E, K, seed)
    dev = torch.device("cuda:0")
    q1, s1 = moe.quantize_weights_fp8(W1.to(dev))
    q3, s3 = moe.quantize_weights_fp8(W3.to(dev))
    q2, s2 = moe.quantize_weights_fp8(W2.to(dev))
    ws = moe.Workspace(T, d, f, E, K, torch.float8_e4m3fn, dev)
    y = moe.moe_forward_fp8(x.to(dev), Wg.to(dev), q1, s1, q3, s3, q2, s2, K, workspace=ws)
    assert moe.moe_read_status(ws) == 0
    # the oracle quantises the bf16 banks itself
    r1, t1 = F8.quantize_weight_columns(W1)
    r3, t3 = F8.quantize_weight_columns(W3)
    r2, t2 = F8.quantize_weight_columns(W2)
    ref = F8.moe_layer_fp8(x, Wg, r1, t1, r3, t3, r2, t2, K)
    g = oracle.gating(x, Wg, K)
    idx, gate, perm, offs, pos = moe.moe_route(x.to(dev), Wg.to(dev), K)
    rep = parity.check_routing(_np(idx), _np(gate), g, K)
    assert rep.n_mismatch == 0, rep
    err = parity.rel_linf(_np(y.float()), ref.y)
    bf = oracle.moe_layer(x, Wg, W1, W3, W2, K).y
    qerr = parity.rel_linf(_np(y.float()), bf)
    print(f"\nfp8 T={T} d={d} f={f} E={E} K={K}: rel err vs fp8 oracle {err:.2e}, vs bf16-weight oracle {qerr:.2e}")
    assert err <= tol, err
    # deterministic
    y2 = moe.moe_forward_fp8(x.to(dev), Wg.to(dev), q1, s1, q3, s3, q2, s2, K, workspace=ws)
    assert torch.equal(y, y2)
    return err


@pytest.mark.parametrize("T,d,f,E,K", [
    (300, 512, 1024, 8, 2),     # multicast-pair tiles
    (1100, 512, 1024, 4, 2),    # CTA-pair tiles, odd tile counts (phantom halves)
    (257, 528, 1040, 8, 2),     # ragged K (k-block tails) and N (odd n-tile count)
    (600, 256, 512, 4, 1),      # top-1
    (1, 512, 1024, 8, 2),       # decode: split down projection
    (8, 1024, 1536, 8, 2),
    (129, 256, 384, 32, 2),     # many experts, empty segments
])
def test_fp8_layer_parity(moe, T, d, f, E, K):
    _check_fp8_layer(moe, T, d, f, E, K, seed=300 + T)


def test_fp8_full_size_decode_one_token(moe, cuda_device):
    """Mixtral-sized weights, one token: the oracle quantises and evaluates
    only the two experts the token selects."""
    Wg, W1, W3, W2 = W.mixtral_weights(device=cuda_device)
    inp = W.decode(1, device=cuda_device, weights=(Wg, W1, W3, W2))
    q1, s1 = moe.quantize_weights_fp8(W1)
    q3, s3 = moe.quantize_weights_fp8(W3)
    q2, s2 = moe.quantize_weights_fp8(W2)
    y = moe.moe_forward_fp8(inp.x, Wg, q1, s1, q3, s3, q2, s2, 2)
    g = oracle.gating(inp.x.cpu(), Wg.cpu(), 2)
    sel = sorted(set(g.idx[0].tolist()))
    # sub-banks of the selected experts, router columns restricted to them
    sub = lambda B: B[sel].cpu()
    r1, t1 = F8.quantize_weight_columns(sub(W1))
    r3, t3 = F8.quantize_weight_columns(sub(W3))
    r2, t2 = F8.quantize_weight_columns(sub(W2))
    # the codes the GPU made for those experts are the oracle's, bit for bit
    assert np.array_equal(_codes(q1[sel], 14336, 4096), r1)
    Wg_sub = Wg.cpu()[:, sel]
    ref = F8.moe_layer_fp8(inp.x.cpu(), Wg_sub, r1, t1, r3, t3, r2, t2, 2)
    err = parity.rel_linf(_np(y.float()), ref.y)
    print(f"\nfp8 full-size T=1: experts {sel}, rel err {err:.2e}")
    assert err <= 2e-2


def test_fp8_full_size_prefill_every_expert(moe, cuda_device):
    """The bench's prefill_fp8 workload (T=4096, Mixtral sizes), checked so
    that every expert's e4m3 banks meet the oracle: for each expert, the most
    common expert pair containing it, and two tokens that chose that pair.
    Such a token's output depends only on the two experts of its pair
    (activation and H scales are per row), and with the router restricted to
    those two columns it keeps the same pair and gates, so the oracle
    quantises and evaluates the pair's two experts only (each expert's banks
    quantised once)."""
    Wg, W1, W3, W2 = W.mixtral_weights(device=cuda_device)
    inp = W.prefill(device=cuda_device, weights=(Wg, W1, W3, W2))
    q = [t for B in (W1, W3, W2) for t in moe.quantize_weights_fp8(B)]
    y = moe.moe_forward_fp8(inp.x, Wg, *q, 2)
    x = inp.x.cpu()
    g = oracle.gating(x, Wg.cpu(), 2)
    gap, _ = oracle.logit_gaps(oracle.router_logits(oracle.f64(x), oracle.f64(Wg.cpu())), 2)
    pairs = [tuple(sorted(r)) if gap[t] > 1e-4 else None for t, r in enumerate(g.idx.tolist())]
    chosen = []
    for e in range(8):
        with_e = [p for p in pairs if p and e in p]
        pe = max(set(with_e), key=with_e.count)
        if pe not in chosen:
            chosen.append(pe)
    assert set(e for p in chosen for e in p) == set(range(8))
    cache = {}

    def banks_of(e):
        if e not in cache:
            cache[e] = [F8.quantize_weight_columns(B[[e]].cpu()) for B in (W1, W3, W2)]
        return cache[e]

    worst = 0.0
    for a, b in chosen:
        toks = [t for t, p in enumerate(pairs) if p == (a, b)][::7][:2]
        ba, bb = banks_of(a), banks_of(b)
        banks = [np.concatenate([ba[i][j], bb[i][j]]) for i in range(3) for j in range(2)]
        ref = F8.moe_layer_fp8(x[toks], Wg.cpu()[:, [a, b]], *banks, 2)
        err = parity.rel_linf(_np(y[toks].float()), ref.y)
        worst = max(worst, err)
        assert err <= 2e-2, (a, b, err)
    print(f"\nfp8 full-size prefill: pairs {chosen}, worst rel err {worst:.2e}")


def test_fp8_full_size_decode32_sampled_tokens(moe, cuda_device):
    """The decode32_fp8 workload (32 tokens, split GEMMs), checked on the
    tokens that chose the most common expert pair, as in the prefill case."""
    Wg, W1, W3, W2 = W.mixtral_weights(device=cuda_device)
    inp = W.decode(32, device=cuda_device, weights=(Wg, W1, W3, W2))
    q = [t for B in (W1, W3, W2) for t in moe.quantize_weights_fp8(B)]
    y = moe.moe_forward_fp8(inp.x, Wg, *q, 2)
    x = inp.x.cpu()
    g = oracle.gating(x, Wg.cpu(), 2)
    pairs = [tuple(sorted(r)) for r in g.idx.tolist()]
    gap, _ = oracle.logit_gaps(oracle.router_logits(oracle.f64(x), oracle.f64(Wg.cpu())), 2)
    pairs = [p if gap[t] > 1e-4 else None for t, p in enumerate(pairs)]
    a, b = max(set(p for p in pairs if p), key=pairs.count)
    toks = [t for t, p in enumerate(pairs) if p == (a, b)]
    banks = [t for B in (W1, W3, W2) for t in F8.quantize_weight_columns(B[[a, b]].cpu())]
    ref = F8.moe_layer_fp8(x[toks], Wg.cpu()[:, [a, b]], *banks, 2)
    err = parity.rel_linf(_np(y[toks].float()), ref.y)
    print(f"\nfp8 full-size decode T=32: experts {[a, b]}, tokens {toks}, rel err {err:.2e}")
    assert err <= 2e-2


@pytest.mark.parametrize("T,d,f,E,K", [(1100, 512, 1024, 4, 2), (700, 256, 384, 2, 1)])
def test_fp8_gemm_forms_agree_bit_for_bit(moe, T, d, f, E, K):
    x, Wg, W1, W3, W2 = _fp8_case(T, d, f, E, K, seed=60 + T)
    dev = torch.device("cuda:0")
    q = [t for W_ in (W1, W3, W2) for t in moe.quantize_weights_fp8(W_.to(dev))]
    outs = [moe.moe_forward_fp8(x.to(dev), Wg.to(dev), *q, K, flags=fl)
            for fl in (moe.MOE_GEMM_MULTICAST_PAIRS, moe.MOE_GEMM_PAIR_MMA, moe.MOE_GEMM_QUAD)]
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
