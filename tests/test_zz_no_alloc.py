"""moe_route_noalloc: routing for callers that cannot allocate device memory.

Plugin hosts without a scratch buffer, code running during a global-mode
graph capture, and allocation-free serving loops cannot pass the library a
workspace.  moe_route_noalloc serves them from a fixed scratch array inside
the library.  This test calls it through the C ABI twice in a row (different
sizes, so the second call runs on the first call's leftovers) and checks that
its results equal moe_route's bit for bit; it also checks the size limit and
that a device-side error (a NaN router input under MOE_DEBUG_CHECKS) reaches
the caller through moe_route_noalloc_status, and that the next call clears
it.  The file is named so that pytest collects it last.
"""
from __future__ import annotations

import ctypes

import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


def _call_noalloc(lib, x, Wg, K, flags=0):
    T, d = x.shape
    E = Wg.shape[1]
    dev = x.device
    idx = torch.full((T, K), -7, dtype=torch.int32, device=dev)
    gate = torch.full((T, K), -7.0, dtype=torch.float32, device=dev)
    perm = torch.full((T * K,), -7, dtype=torch.int32, device=dev)
    offs = torch.full((E + 1,), -7, dtype=torch.int32, device=dev)
    pos = torch.full((T, K), -7, dtype=torch.int32, device=dev)
    vp = ctypes.c_void_p
    rc = lib.moe_route_noalloc(vp(x.data_ptr()), vp(Wg.data_ptr()), T, d, E, K, 0 if x.dtype == torch.bfloat16 else 1,
                               vp(idx.data_ptr()), vp(gate.data_ptr()), vp(perm.data_ptr()), vp(offs.data_ptr()),
                               vp(pos.data_ptr()), flags, vp(torch.cuda.current_stream(dev).cuda_stream))
    return rc, (idx, gate, perm, offs, pos)


def test_route_noalloc_matches_route_on_consecutive_calls(cuda_device):
    from sparse_mixture_experts_55_b300 import _lib, build
    build.build()
    import sparse_mixture_experts_55_b300 as moe
    lib = _lib.load()
    dev = cuda_device
    cases = [
        (2000, 4096, 8, 2, torch.bfloat16, 21),
        (16384, 4096, 8, 2, torch.bfloat16, 22),   # the size limit, after a smaller call
        (300, 512, 32, 1, torch.float32, 23),
        (16384, 512, 32, 2, torch.bfloat16, 24),   # the limit with the most experts
    ]
    for T, d, E, K, dt, seed in cases:
        x = W.rms_rows(T, d, seed, "cpu", dt).to(dev)
        Wg = W.randn((d, E), d ** -0.5, seed + 100, "cpu", dt).to(dev)
        rc, got = _call_noalloc(lib, x, Wg, K)
        assert rc == 0, _lib.status_string(rc)
        want = moe.moe_route(x, Wg, K)
        torch.cuda.synchronize(dev)
        for name, a, b in zip(("idx", "gate", "perm_tok", "offsets", "pos"), got, want):
            assert torch.equal(a, b), f"{name} differs at T={T} E={E} K={K}"
    # beyond the fixed scratch: rejected before anything is launched
    T = 16385
    x = torch.zeros((T, 64), dtype=torch.bfloat16, device=dev)
    Wg = torch.zeros((64, 8), dtype=torch.bfloat16, device=dev)
    rc, _ = _call_noalloc(lib, x, Wg, 2)
    assert rc == _lib.MOE_ERR_UNSUPPORTED


def test_route_noalloc_reports_device_errors(cuda_device):
    from sparse_mixture_experts_55_b300 import _lib, build
    build.build()
    lib = _lib.load()
    dev = cuda_device
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    T, d, E, K = 64, 512, 8, 2
    x = W.rms_rows(T, d, 31, "cpu", torch.bfloat16).to(dev)
    Wg = W.randn((d, E), d ** -0.5, 131, "cpu", torch.bfloat16).to(dev)
    rc, _ = _call_noalloc(lib, x, Wg, K, flags=_lib.MOE_DEBUG_CHECKS)
    assert rc == 0
    assert lib.moe_route_noalloc_status(stream) == _lib.MOE_OK
    x_bad = x.clone()
    x_bad[5, 7] = float("nan")
    rc, (idx, _, _, offs, _) = _call_noalloc(lib, x_bad, Wg, K, flags=_lib.MOE_DEBUG_CHECKS)
    assert rc == 0
    assert lib.moe_route_noalloc_status(stream) == _lib.MOE_ERR_NONFINITE
    # the routing of the finite tokens is still valid
    assert int(offs[-1]) == T * K and bool(((idx >= 0) & (idx < E)).all())
    # the next call starts from a clear status word
    rc, _ = _call_noalloc(lib, x, Wg, K, flags=_lib.MOE_DEBUG_CHECKS)
    assert rc == 0
    assert lib.moe_route_noalloc_status(stream) == _lib.MOE_OK
    # unknown flags are rejected before anything runs
    rc, _ = _call_noalloc(lib, x, Wg, K, flags=0x40)
    assert rc == _lib.MOE_ERR_INVALID_ARG
