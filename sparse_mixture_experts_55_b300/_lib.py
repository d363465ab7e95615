"""ctypes loader for libmoe.so (the C ABI of include/moe.h).

The library is built in-tree (``python -m sparse_mixture_experts_55_b300.build``).
There is no fallback: if the shared library is missing or fails to load, every
call raises.
"""
from __future__ import annotations

import ctypes
import pathlib
import threading

LIB_PATH = pathlib.Path(__file__).resolve().parent / "libmoe.so"

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_DEVICE_TIMEOUT = 5
MOE_ERR_NONFINITE = 6
MOE_ERR_DEVICE_BOUNDS = 7

MOE_BF16 = 0
MOE_F32 = 1
MOE_FP8_E4M3 = 2

MOE_ACCUMULATE = 0x1
# stage slots of a stamps array (moe_forward_stamped), in order
MOE_NUM_STAGES = 8
STAGES = ("route", "group", "gather", "gate_up_gemm", "quant_h", "down_gemm", "combine", "rmsnorm")
MOE_DEBUG_CHECKS = 0x2
MOE_DEBUG_FORCE_TIMEOUT = 0x4
MOE_GEMM_PAIR_MMA = 0x8
MOE_GEMM_QUAD = 0x10
MOE_GEMM_MULTICAST_PAIRS = 0x20

# name -> (restype, argtypes), one entry per function declared in include/moe.h
_vp, _i, _sz, _u = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_uint
class ExpertCacheState(ctypes.Structure):
    """Mirror of moe_expert_cache (include/moe.h)."""
    _fields_ = [("E", ctypes.c_int), ("C", ctypes.c_int),
                ("slot_of", ctypes.c_int * 32), ("expert_in", ctypes.c_int * 32),
                ("last_use", ctypes.c_longlong * 32), ("step", ctypes.c_longlong),
                ("hits", ctypes.c_longlong), ("misses", ctypes.c_longlong),
                ("bytes_loaded", ctypes.c_longlong)]


_ip = ctypes.POINTER(ctypes.c_int)
_cp = ctypes.POINTER(ExpertCacheState)

SIGNATURES = {
    "moe_workspace_bytes": (_sz, [_i, _i, _i, _i, _i, _i]),
    "moe_forward_launches": (_i, [_i, _i, _i, _i, _i, _i]),
    "moe_forward": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _sz, _u, _vp]),
    "moe_forward_stamped": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _sz, _u, _vp, _vp]),
    "moe_block_forward": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, ctypes.c_float, _vp, _sz, _u,
                                _vp]),
    "moe_block_forward_stamped": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, ctypes.c_float, _vp, _sz,
                                        _u, _vp, _vp]),
    "moe_quantize_weights_fp8": (_i, [_vp, _i, _i, _i, _vp, _vp, _vp]),
    "moe_fp8_weight_bytes": (_sz, [_i, _i, _i]),
    "moe_forward_fp8": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _sz, _u, _vp]),
    "moe_forward_fp8_stamped": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _sz, _u,
                                     _vp, _vp]),
    "moe_train_workspace_bytes": (_sz, [_i, _i, _i, _i, _i, _i]),
    "moe_forward_train": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _sz, _u, _vp]),
    "moe_backward": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _sz, _u,
                          _vp]),
    "moe_backward_timed": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp,
                                _sz, _u, _vp, _vp]),
    "moe_expert_cache_init": (_i, [_cp, _i, _i]),
    "moe_expert_cache_plan": (_i, [_cp, _ip, _ip, _ip, _ip]),
    "moe_forward_cached": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _cp, _vp, _i, _i, _i, _i, _i, _i, _vp, _sz,
                                _u, _vp]),
    "moe_route": (_i, [_vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_route_noalloc": (_i, [_vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _u, _vp]),
    "moe_route_noalloc_status": (_i, [_vp]),
    "moe_rmsnorm": (_i, [_vp, _vp, _i, _i, ctypes.c_float, _i, _vp]),
    "moe_read_status": (_i, [_vp, _vp]),
    "moe_status_string": (ctypes.c_char_p, [_i]),
    "moe_version": (_i, []),
}

_lock = threading.Lock()
_lib = None


class MoEError(RuntimeError):
    """A libmoe entry point returned a non-zero status."""

    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: status {code} ({status_string(code)})")


def load() -> ctypes.CDLL:
    """Load libmoe.so once and attach the C signatures; raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not LIB_PATH.exists():
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with `python -m sparse_mixture_experts_55_b300.build`")
            lib = ctypes.CDLL(str(LIB_PATH))
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def status_string(code: int) -> str:
    return load().moe_status_string(int(code)).decode()


def check(fn: str, code: int) -> None:
    if code != MOE_OK:
        raise MoEError(fn, code)
