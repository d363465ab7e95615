"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/moe.h declares, sizes workspaces, and rejects bad
arguments before touching the device."""
from __future__ import annotations

import ctypes
import pathlib
import re

import pytest

from sparse_mixture_experts_55_b300 import _lib

ROOT = pathlib.Path(__file__).resolve().parents[1]


def _header_functions():
    text = (ROOT / "include" / "moe.h").read_text()
    return sorted(set(re.findall(r"^MOE_API\s+[\w\s\*]*?\b(moe_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    from sparse_mixture_experts_55_b300 import build
    build.build()
    return _lib.load()


def test_header_declares_the_boundary():
    names = _header_functions()
    assert names == sorted(["moe_workspace_bytes", "moe_forward", "moe_forward_stamped", "moe_block_forward",
                            "moe_block_forward_stamped", "moe_route",
                            "moe_quantize_weights_fp8", "moe_fp8_weight_bytes", "moe_forward_fp8",
                            "moe_forward_fp8_stamped",
                            "moe_train_workspace_bytes", "moe_forward_train", "moe_backward", "moe_backward_timed",
                            "moe_expert_cache_init", "moe_expert_cache_plan", "moe_forward_cached",
                            "moe_forward_launches",
                            "moe_route_noalloc", "moe_route_noalloc_status", "moe_rmsnorm",
                            "moe_read_status", "moe_status_string", "moe_version"])


def test_exports_every_declared_symbol(lib):
    for name in _header_functions():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, name


def test_status_strings_and_version(lib):
    assert lib.moe_version() >= 100
    for code in range(8):
        assert lib.moe_status_string(code).decode() not in ("", "unknown status")
    assert lib.moe_status_string(99).decode() == "unknown status"


def test_workspace_bytes(lib):
    mix = lib.moe_workspace_bytes(4096, 4096, 14336, 8, 2, _lib.MOE_BF16)
    # grouped rows: 8192 tokens*slots + 8 * 127 pad rows, rounded to 128 -> 9216;
    # padded X_perm and H, compact fp32 expert outputs, the block's normalised
    # input, and the expert GEMMs' tail-split scratch (one 2 x 128 x 256 fp32
    # pair of tiles per four SMs and one more)
    R, TK = 9216, 8192
    tail = (148 // 4 + 1) * 2 * 128 * 256 * 4
    lower = R * 4096 * 2 + R * 14336 * 2 + TK * 4096 * 4 + 4096 * 4096 * 2 + tail
    assert lower <= mix <= lower + 2 * 1024 * 1024
    assert lib.moe_workspace_bytes(0, 64, 128, 8, 2, _lib.MOE_F32) > 0
    # invalid shapes -> 0
    assert lib.moe_workspace_bytes(16, 60, 128, 8, 2, _lib.MOE_BF16) == 0   # d not a multiple of 8
    assert lib.moe_workspace_bytes(16, 64, 128, 8, 3, _lib.MOE_BF16) == 0   # K > 2
    assert lib.moe_workspace_bytes(16, 64, 128, 1, 2, _lib.MOE_BF16) == 0   # K > E
    assert lib.moe_workspace_bytes(16, 64, 128, 33, 2, _lib.MOE_BF16) == 0  # E > 32
    assert lib.moe_workspace_bytes(16, 64, 128, 8, 2, 7) == 0               # dtype
    assert lib.moe_workspace_bytes(-1, 64, 128, 8, 2, 0) == 0


def _fwd(lib, **kw):
    a = dict(x=0x1000, Wg=0x2000, W1=0x3000, W3=0x4000, W2=0x5000, y=0x100000, T=16, d=64, f=128, E=8, K=2,
             dtype=_lib.MOE_BF16, ws=0x200000, ws_bytes=1 << 40, flags=0, stream=0)
    a.update(kw)
    vp = ctypes.c_void_p
    return lib.moe_forward(vp(a["x"]), vp(a["Wg"]), vp(a["W1"]), vp(a["W3"]), vp(a["W2"]), vp(a["y"]), a["T"],
                           a["d"], a["f"], a["E"], a["K"], a["dtype"], vp(a["ws"]), a["ws_bytes"], a["flags"],
                           vp(a["stream"]))


@pytest.mark.parametrize("kw,code", [
    (dict(K=3), _lib.MOE_ERR_UNSUPPORTED),
    (dict(K=0), _lib.MOE_ERR_INVALID_ARG),
    (dict(E=1, K=2), _lib.MOE_ERR_INVALID_ARG),
    (dict(E=40), _lib.MOE_ERR_UNSUPPORTED),
    (dict(d=60), _lib.MOE_ERR_INVALID_ARG),
    (dict(f=130), _lib.MOE_ERR_INVALID_ARG),
    (dict(T=-1), _lib.MOE_ERR_INVALID_ARG),
    (dict(dtype=5), _lib.MOE_ERR_UNSUPPORTED),
    (dict(x=0), _lib.MOE_ERR_INVALID_ARG),
    (dict(W2=0), _lib.MOE_ERR_INVALID_ARG),
    (dict(W1=0x3008), _lib.MOE_ERR_INVALID_ARG),                   # misaligned
    (dict(y=0x1000 + 16 * 64 * 2 - 16), _lib.MOE_ERR_INVALID_ARG),  # y overlaps x
    (dict(flags=0x80), _lib.MOE_ERR_INVALID_ARG),
    (dict(flags=0x18), _lib.MOE_ERR_INVALID_ARG),                  # two GEMM forms at once
    (dict(ws=0), _lib.MOE_ERR_WORKSPACE),
    (dict(ws=0x200008), _lib.MOE_ERR_WORKSPACE),
    (dict(ws_bytes=1024), _lib.MOE_ERR_WORKSPACE),
])
def test_forward_rejects_bad_arguments_on_host(lib, kw, code):
    # The pointers are never dereferenced: validation happens before any CUDA call.
    assert _fwd(lib, **kw) == code


def test_forced_timeout_flag_is_bf16_only(lib):
    assert _fwd(lib, flags=_lib.MOE_DEBUG_FORCE_TIMEOUT, dtype=_lib.MOE_F32) == _lib.MOE_ERR_UNSUPPORTED
    # accepted for bf16: the call goes on to the workspace check
    assert _fwd(lib, flags=_lib.MOE_DEBUG_FORCE_TIMEOUT, ws_bytes=1) == _lib.MOE_ERR_WORKSPACE


def test_fp32_multiple_of_4_is_accepted_by_shape_check(lib):
    # d = 60 is fine for fp32 (16-byte rows); with a 1-byte workspace the call
    # stops at the workspace check, after the shape checks passed.
    assert _fwd(lib, d=60, dtype=_lib.MOE_F32, ws_bytes=1) == _lib.MOE_ERR_WORKSPACE


def test_route_and_rmsnorm_reject_bad_arguments(lib):
    vp = ctypes.c_void_p
    assert lib.moe_route(vp(0x1000), vp(0x2000), 16, 64, 8, 3, 0, vp(16), vp(16), vp(16), vp(16), vp(0),
                         vp(0x200000), 1 << 40, vp(0)) == _lib.MOE_ERR_UNSUPPORTED
    assert lib.moe_route(vp(0x1000), vp(0x2000), 16, 64, 8, 2, 0, vp(0), vp(16), vp(16), vp(16), vp(0),
                         vp(0x200000), 1 << 40, vp(0)) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_rmsnorm(vp(0x1000), vp(0x1000), 4, 64, 0.0, 0, vp(0)) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_rmsnorm(vp(0x1000), vp(0x1000), 4, 64, 1e-5, 9, vp(0)) == _lib.MOE_ERR_UNSUPPORTED
    assert lib.moe_rmsnorm(vp(0), vp(0), 0, 64, 1e-5, 0, vp(0)) == _lib.MOE_OK   # empty input: no-op
    assert lib.moe_read_status(vp(0), vp(0)) == _lib.MOE_ERR_WORKSPACE


def test_binding_has_no_fallback(monkeypatch, tmp_path):
    """With the shared library missing the binding raises instead of computing anything."""
    monkeypatch.setattr(_lib, "LIB_PATH", tmp_path / "libmoe.so")
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        _lib.load()


def test_block_forward_rejects_bad_arguments(lib):
    vp = ctypes.c_void_p
    f32 = ctypes.c_float

    def blk(h=0x1000, T=16, K=2, eps=1e-5, ws=0x200000, ws_bytes=1 << 40, flags=0):
        return lib.moe_block_forward(vp(h), vp(0x2000), vp(0x3000), vp(0x4000), vp(0x5000), T, 64, 128, 8, K,
                                     _lib.MOE_BF16, f32(eps), vp(ws), ws_bytes, flags, vp(0))

    assert blk(K=3) == _lib.MOE_ERR_UNSUPPORTED
    assert blk(eps=0.0) == _lib.MOE_ERR_INVALID_ARG
    assert blk(flags=_lib.MOE_ACCUMULATE) == _lib.MOE_ERR_INVALID_ARG   # accumulation is implied
    assert blk(h=0) == _lib.MOE_ERR_INVALID_ARG
    assert blk(h=0x1008) == _lib.MOE_ERR_INVALID_ARG
    assert blk(ws=0) == _lib.MOE_ERR_WORKSPACE
    assert blk(ws_bytes=64) == _lib.MOE_ERR_WORKSPACE
    assert blk(h=0x200000 + 256) == _lib.MOE_ERR_INVALID_ARG            # h inside the workspace
    assert blk(h=0, T=0) == _lib.MOE_OK                                  # empty input: no-op


def test_fp8_entry_points_reject_bad_arguments(lib):
    vp = ctypes.c_void_p

    def fwd8(d=64, f=128, x=0x1000, w=0x3000, s=0x9000, ws=0x200000, ws_bytes=1 << 40, flags=0, K=2):
        return lib.moe_forward_fp8(vp(x), vp(0x2000), vp(w), vp(s), vp(0x4000), vp(s), vp(0x5000), vp(s),
                                   vp(0x100000), 16, d, f, 8, K, vp(ws), ws_bytes, flags, vp(0))

    assert fwd8(d=72) == _lib.MOE_ERR_INVALID_ARG          # e4m3 rows need multiples of 16
    assert fwd8(f=136) == _lib.MOE_ERR_INVALID_ARG
    assert fwd8(K=3) == _lib.MOE_ERR_UNSUPPORTED
    assert fwd8(w=0) == _lib.MOE_ERR_INVALID_ARG
    assert fwd8(s=0) == _lib.MOE_ERR_INVALID_ARG
    assert fwd8(w=0x3008) == _lib.MOE_ERR_INVALID_ARG      # misaligned
    assert fwd8(flags=0x80) == _lib.MOE_ERR_INVALID_ARG
    assert fwd8(ws=0) == _lib.MOE_ERR_WORKSPACE
    assert fwd8(ws_bytes=64) == _lib.MOE_ERR_WORKSPACE
    # the bf16 entry point does not take the e4m3 dtype
    assert _fwd(lib, dtype=_lib.MOE_FP8_E4M3) == _lib.MOE_ERR_UNSUPPORTED
    assert lib.moe_workspace_bytes(16, 64, 128, 8, 2, _lib.MOE_FP8_E4M3) > 0
    assert lib.moe_workspace_bytes(16, 72, 128, 8, 2, _lib.MOE_FP8_E4M3) == 0
    assert lib.moe_quantize_weights_fp8(vp(0), 8, 64, 64, vp(0x1000), vp(0x2000), vp(0)) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_quantize_weights_fp8(vp(0x1000), 0, 64, 64, vp(0x900000), vp(0x2000), vp(0)) == \
        _lib.MOE_ERR_INVALID_ARG
    # codes overlapping the bank
    assert lib.moe_quantize_weights_fp8(vp(0x1000), 1, 64, 64, vp(0x1000 + 64), vp(0x90000), vp(0)) == \
        _lib.MOE_ERR_INVALID_ARG


def test_training_entry_points_reject_bad_arguments(lib):
    vp = ctypes.c_void_p
    # sizes: bf16 with d and f multiples of 64 only
    assert lib.moe_train_workspace_bytes(16, 128, 256, 8, 2, _lib.MOE_BF16) > lib.moe_workspace_bytes(
        16, 128, 256, 8, 2, _lib.MOE_BF16)
    assert lib.moe_train_workspace_bytes(16, 136, 256, 8, 2, _lib.MOE_BF16) == 0
    assert lib.moe_train_workspace_bytes(16, 128, 264, 8, 2, _lib.MOE_BF16) == 0
    assert lib.moe_train_workspace_bytes(16, 128, 256, 8, 2, _lib.MOE_F32) == 0
    assert lib.moe_train_workspace_bytes(16, 128, 256, 8, 2, _lib.MOE_FP8_E4M3) == 0
    assert lib.moe_train_workspace_bytes(0, 128, 256, 8, 2, _lib.MOE_BF16) > 0
    # the training forward checks like moe_forward, plus the training sizes
    args = [vp(0x1000), vp(0x2000), vp(0x3000), vp(0x4000), vp(0x5000), vp(0x100000), 16, 128, 256, 8, 2,
            _lib.MOE_BF16, vp(0x200000), 1 << 40, 0, vp(0)]
    bad = list(args); bad[8] = 264
    assert lib.moe_forward_train(*bad) == _lib.MOE_ERR_UNSUPPORTED
    bad = list(args); bad[11] = _lib.MOE_F32
    assert lib.moe_forward_train(*bad) == _lib.MOE_ERR_UNSUPPORTED
    bad = list(args); bad[0] = vp(0)
    assert lib.moe_forward_train(*bad) == _lib.MOE_ERR_INVALID_ARG
    bad = list(args); bad[13] = 64
    assert lib.moe_forward_train(*bad) == _lib.MOE_ERR_WORKSPACE

    E, d, f = 8, 128, 256
    wb = E * d * f * 4

    def bwd(T=16, dx=0x10_000000, dWg=0x20_000000, dW1=0x30_000000, dW3=0x40_000000, dW2=0x50_000000, x=0x1000,
            dy=0x8000, ws=0x60_000000, ws_bytes=1 << 40, flags=0, dt=_lib.MOE_BF16, dd=d):
        return lib.moe_backward(vp(x), vp(0x2000), vp(0x3000), vp(0x4000), vp(0x5000), vp(dy), vp(dx), vp(dWg),
                                vp(dW1), vp(dW3), vp(dW2), T, dd, f, E, 2, dt, vp(ws), ws_bytes, flags, vp(0))

    assert bwd(dt=_lib.MOE_F32) == _lib.MOE_ERR_UNSUPPORTED
    assert bwd(dd=192 + 8) == _lib.MOE_ERR_UNSUPPORTED
    assert bwd(flags=0x8) == _lib.MOE_ERR_INVALID_ARG       # no GEMM form flags
    assert bwd(flags=0x40) == _lib.MOE_ERR_INVALID_ARG
    assert bwd(dW1=0) == _lib.MOE_ERR_INVALID_ARG
    assert bwd(dx=0) == _lib.MOE_ERR_INVALID_ARG
    assert bwd(dy=0x8008) == _lib.MOE_ERR_INVALID_ARG      # misaligned
    assert bwd(dW3=0x30_000000 + wb // 2) == _lib.MOE_ERR_INVALID_ARG   # dW3 overlaps dW1
    assert bwd(dx=0x50_000000 + 64) == _lib.MOE_ERR_INVALID_ARG        # dx overlaps dW2
    assert bwd(ws=0) == _lib.MOE_ERR_WORKSPACE
    assert bwd(ws_bytes=64) == _lib.MOE_ERR_WORKSPACE


def test_cached_forward_rejects_bad_arguments(lib):
    vp = ctypes.c_void_p
    st = _lib.ExpertCacheState()
    assert lib.moe_expert_cache_init(ctypes.byref(st), 8, 4) == 0

    def fwd(E=8, dt=_lib.MOE_BF16, w1h=0x3000, w1d=0x30_000000, flags=0, ws=0x60_000000, ws_bytes=1 << 40, cache=True):
        return lib.moe_forward_cached(vp(0x1000), vp(0x2000), vp(w1h), vp(0x4000), vp(0x5000), vp(w1d),
                                      vp(0x40_000000), vp(0x50_000000), ctypes.byref(st) if cache else None,
                                      vp(0x100000), 4, 128, 256, E, 2, dt, vp(ws), ws_bytes, flags, vp(0))

    assert fwd(dt=_lib.MOE_F32) == _lib.MOE_ERR_UNSUPPORTED
    assert fwd(E=6) == _lib.MOE_ERR_INVALID_ARG            # the cache was made for 8 experts
    assert fwd(cache=False) == _lib.MOE_ERR_INVALID_ARG
    assert fwd(w1h=0) == _lib.MOE_ERR_INVALID_ARG
    assert fwd(w1d=0x30_000008) == _lib.MOE_ERR_INVALID_ARG  # misaligned slot bank
    assert fwd(flags=0x8) == _lib.MOE_ERR_INVALID_ARG        # GEMM form flags are not taken here
    assert fwd(ws=0) == _lib.MOE_ERR_WORKSPACE
    assert fwd(ws_bytes=64) == _lib.MOE_ERR_WORKSPACE
    assert st.step == 0


def test_forward_launch_counts(lib):
    # prefill: the down projection is not split, so its epilogue forms y
    assert lib.moe_forward_launches(4096, 4096, 14336, 8, 2, _lib.MOE_BF16) == 5
    assert lib.moe_forward_launches(4096, 4096, 14336, 8, 2, _lib.MOE_FP8_E4M3) == 6
    # one token: router and grouping fused, split down projection whose
    # epilogue still forms y (up to 4 tokens)
    assert lib.moe_forward_launches(1, 4096, 14336, 8, 2, _lib.MOE_BF16) == 4
    assert lib.moe_forward_launches(1, 4096, 14336, 8, 2, _lib.MOE_FP8_E4M3) == 5
    # eight tokens: split down projection, separate combine
    assert lib.moe_forward_launches(8, 4096, 14336, 8, 2, _lib.MOE_BF16) == 5
    # 256 tokens still fuse the router and the grouping, 257 do not
    assert lib.moe_forward_launches(256, 64, 128, 8, 2, _lib.MOE_F32) == 5
    assert lib.moe_forward_launches(257, 64, 128, 8, 2, _lib.MOE_F32) == 6
    # fp32: two SIMT FFN kernels and the combine
    assert lib.moe_forward_launches(64, 64, 128, 8, 2, _lib.MOE_F32) == 5
    assert lib.moe_forward_launches(0, 64, 128, 8, 2, _lib.MOE_BF16) == 0
    assert lib.moe_forward_launches(16, 63, 128, 8, 2, _lib.MOE_BF16) == 0


def test_fp8_weight_bytes(lib):
    # whole 128 x 128 tiles per expert, padding included
    assert lib.moe_fp8_weight_bytes(8, 4096, 14336) == 8 * 4096 * 14336
    assert lib.moe_fp8_weight_bytes(3, 200, 72) == 3 * 2 * 1 * 128 * 128
    assert lib.moe_fp8_weight_bytes(0, 64, 64) == 0
