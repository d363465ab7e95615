"""GPU checks of the decode-time expert cache (moe_forward_cached): over a
locality trace the cached layer equals moe_forward bit for bit at every step
(the same kernels, reading expert e from its slot), and the cache's decisions
(loads, hits, misses, maps) equal the oracle LRU policy's on the needed sets
the GPU routing produced; the cached layer's output is also compared with the
float64 oracle directly at every step.  A step that needs more experts than
there are slots is refused without changing the state."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from oracle.cache_oracle import LRUCache
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe(cuda_device):
    from sparse_mixture_experts_55_b300 import build
    build.build()
    import sparse_mixture_experts_55_b300 as m
    return m


@pytest.mark.parametrize("T,C,steps,keep", [(1, 3, 24, 0.35), (1, 2, 16, 0.0), (2, 4, 12, 0.35), (1, 8, 10, 0.35)])
def test_cached_forward_equals_forward_and_policy_matches_oracle(moe, cuda_device, T, C, steps, keep):
    d, f, E, K = 256, 512, 8, 2
    Wg, W1, W3, W2 = (t.to(cuda_device) for t in W.mixtral_weights(d, f, E, seed=21, device="cpu"))
    xs, _ = W.decode_trace(steps, Wg, T=T, keep=keep, seed=21, device=cuda_device)
    cache = moe.ExpertCache(W1, W3, W2, C, cuda_device)
    ref = LRUCache(E, C)
    ws = moe.Workspace(T, d, f, E, K, torch.bfloat16, cuda_device)
    for i in range(steps):
        x = xs[i].contiguous()
        y = cache.forward(x, Wg, K, workspace=ws)
        y_ref = moe.moe_forward(x, Wg, W1, W3, W2, K)
        torch.cuda.synchronize()
        assert torch.equal(y, y_ref), i
        y64 = oracle.moe_layer(x.cpu(), Wg.cpu(), W1.cpu(), W3.cpu(), W2.cpu(), K).y
        assert parity.rel_linf(y.float().cpu().numpy(), y64) <= parity.TOL["bf16"], i
        idx, *_ = moe.moe_route(x, Wg, K)
        ref.plan(sorted(set(idx.flatten().tolist())))
        st = cache.state
        assert list(st.slot_of)[:E] == ref.slot_of and list(st.expert_in)[:C] == ref.expert_in, i
        assert (st.hits, st.misses) == (ref.hits, ref.misses)
    assert cache.state.bytes_loaded == ref.misses * 3 * d * f * 2
    assert moe.moe_read_status(ws) == 0


def test_step_needing_more_experts_than_slots_is_refused(moe, cuda_device):
    d, f, E, K = 256, 512, 8, 2
    Wg, W1, W3, W2 = (t.to(cuda_device) for t in W.mixtral_weights(d, f, E, seed=22, device="cpu"))
    x = W.rms_rows(64, d, 5, cuda_device)  # 64 tokens reach more than 2 experts
    cache = moe.ExpertCache(W1, W3, W2, 2, cuda_device)
    with pytest.raises(moe.MoEError) as ei:
        cache.forward(x, Wg, K)
    assert ei.value.code == moe._lib.MOE_ERR_UNSUPPORTED
    assert cache.state.step == 0 and cache.state.misses == 0 and cache.state.bytes_loaded == 0


def test_cached_forward_at_full_size(moe, cuda_device):
    # Mixtral-sized banks (2.8 GB in pinned host memory), 2 of 8 experts on
    # the GPU, six decode steps of the bench's locality trace: bit for bit
    # moe_forward, decisions as the oracle policy's.
    Wg, W1, W3, W2 = W.mixtral_weights(device=cuda_device)
    E, K, C = 8, 2, 2
    xs, _ = W.decode_trace(6, Wg, T=1, seed=W.BASE_SEED, device=cuda_device)
    cache = moe.ExpertCache(W1, W3, W2, C, cuda_device)
    ref = LRUCache(E, C)
    for i in range(xs.shape[0]):
        y = cache.forward(xs[i], Wg, K)
        assert torch.equal(y, moe.moe_forward(xs[i], Wg, W1, W3, W2, K)), i
        if i < 2:  # the oracle on the token directly (two steps keep the host work bounded)
            y64 = oracle.moe_layer_tokens(xs[i].cpu(), Wg.cpu(), W1, W3, W2, K, [0]).y
            assert parity.rel_linf(y.float().cpu().numpy(), y64) <= parity.TOL["bf16"], i
        idx, *_ = moe.moe_route(xs[i], Wg, K)
        ref.plan(sorted(set(idx.flatten().tolist())))
        assert list(cache.state.slot_of)[:E] == ref.slot_of, i
    assert (cache.state.hits, cache.state.misses) == (ref.hits, ref.misses)
    assert cache.state.bytes_loaded == ref.misses * 3 * 4096 * 14336 * 2
