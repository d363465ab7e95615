"""Mixtral-style sparse mixture-of-experts feed-forward layer for NVIDIA B300.

Python binding of libmoe.so (include/moe.h).  These functions only marshal
arguments: they take torch tensors for device memory and streams and pass raw
pointers to the C ABI; every step of the layer runs in the library's CUDA
kernels.  There is no CPU fallback.

    y = moe_forward(x, Wg, W1, W3, W2, K=2)

computes y = sum over the K selected experts of gate * SwiGLU_expert(x), with
x [T, d], Wg [d, E], W1/W3 [E, d, f], W2 [E, f, d] (bf16 or fp32, all on one
CUDA device).
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import (MOE_ACCUMULATE, MOE_BF16, MOE_DEBUG_CHECKS, MOE_DEBUG_FORCE_TIMEOUT, MOE_F32,  # noqa: F401
                   MOE_FP8_E4M3, MOE_GEMM_MULTICAST_PAIRS, MOE_GEMM_PAIR_MMA, MOE_GEMM_QUAD, MoEError,
                   status_string)

__all__ = ["moe_forward", "moe_forward_stamped", "moe_block_forward", "moe_block_forward_stamped", "HostPipeline",
           "quantize_weights_fp8", "moe_forward_fp8", "moe_forward_fp8_stamped", "new_stamps", "stage_spans", "TrainWorkspace", "moe_forward_train", "moe_backward",
           "LayerGrads", "ExpertCache", "moe_forward_host", "moe_route", "moe_rmsnorm", "moe_read_status", "moe_workspace_bytes",
           "Workspace", "MoEError", "MOE_ACCUMULATE", "MOE_DEBUG_CHECKS", "MOE_BF16", "MOE_F32",
           "status_string", "library_path"]

_DTYPES = {torch.bfloat16: MOE_BF16, torch.float32: MOE_F32}
# workspace sizing of the e4m3-weight variant (tokens stay bf16)
_WS_DTYPES = {**_DTYPES, torch.float8_e4m3fn: MOE_FP8_E4M3}


def library_path() -> str:
    return str(_lib.LIB_PATH)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {t.dtype}; use bfloat16 or float32")
    return _DTYPES[t.dtype]


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream_ptr(stream, device) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype=None, device=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def moe_workspace_bytes(T: int, d: int, f: int, E: int, K: int, dtype=torch.bfloat16) -> int:
    code = _WS_DTYPES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    n = _lib.load().moe_workspace_bytes(T, d, f, E, K, code)
    if n == 0:
        raise ValueError(f"unsupported sizes T={T} d={d} f={f} E={E} K={K} dtype={dtype}")
    return int(n)


class Workspace:
    """A reusable device workspace sized by moe_workspace_bytes (a torch uint8 buffer)."""

    def __init__(self, T, d, f, E, K, dtype=torch.bfloat16, device=None):
        self.nbytes = moe_workspace_bytes(T, d, f, E, K, dtype)
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device or "cuda")
        self.key = (T, d, f, E, K, dtype)

    def ptr(self):
        return ctypes.c_void_p(self.buf.data_ptr())


def moe_forward(x, Wg, W1, W3, W2, K: int = 2, y=None, workspace: Workspace | None = None,
                flags: int = 0, stream=None):
    """MoE layer forward on the GPU; returns y [T, d] (written in place if given)."""
    dev = x.device
    dt = x.dtype
    for t, n in ((x, "x"), (Wg, "Wg"), (W1, "W1"), (W3, "W3"), (W2, "W2")):
        _need(t, n, dt, dev)
    T, d = x.shape
    E, d1, f = W1.shape
    if Wg.shape != (d, E) or W3.shape != (E, d, f) or W2.shape != (E, f, d) or d1 != d:
        raise ValueError("shape mismatch: x [T,d], Wg [d,E], W1/W3 [E,d,f], W2 [E,f,d]")
    if y is None:
        y = torch.empty_like(x)
    else:
        _need(y, "y", dt, dev)
    if workspace is None:
        workspace = Workspace(T, d, f, E, K, dt, dev)
    rc = _lib.load().moe_forward(_ptr(x), _ptr(Wg), _ptr(W1), _ptr(W3), _ptr(W2), _ptr(y), T, d, f, E, K,
                                 _dtype_code(x), workspace.ptr(), workspace.nbytes, flags,
                                 _stream_ptr(stream, dev))
    _lib.check("moe_forward", rc)
    return y


def moe_block_forward(h, Wg, W1, W3, W2, K: int = 2, eps: float = 1e-5, workspace: Workspace | None = None,
                      flags: int = 0, stream=None):
    """One pre-norm MoE half-block in place: h <- h + MoE(RMSNorm(h)); returns h."""
    dev = h.device
    dt = h.dtype
    for t, n in ((h, "h"), (Wg, "Wg"), (W1, "W1"), (W3, "W3"), (W2, "W2")):
        _need(t, n, dt, dev)
    T, d = h.shape
    E, d1, f = W1.shape
    if Wg.shape != (d, E) or W3.shape != (E, d, f) or W2.shape != (E, f, d) or d1 != d:
        raise ValueError("shape mismatch: h [T,d], Wg [d,E], W1/W3 [E,d,f], W2 [E,f,d]")
    if workspace is None:
        workspace = Workspace(T, d, f, E, K, dt, dev)
    rc = _lib.load().moe_block_forward(_ptr(h), _ptr(Wg), _ptr(W1), _ptr(W3), _ptr(W2), T, d, f, E, K,
                                       _dtype_code(h), float(eps), workspace.ptr(), workspace.nbytes, flags,
                                       _stream_ptr(stream, dev))
    _lib.check("moe_block_forward", rc)
    return h


def new_stamps(n: int = 1, device=None) -> torch.Tensor:
    """Device buffer for n stamped calls, initialised as the calls expect:
    int64 [n, 2 * MOE_NUM_STAGES], begin slots -1 (all ones as unsigned) and
    end slots 0 (the library treats each row as unsigned 64-bit times)."""
    st = torch.zeros((n, 2 * _lib.MOE_NUM_STAGES), dtype=torch.int64, device=device or "cuda")
    st[:, :_lib.MOE_NUM_STAGES] = -1
    return st


def _stamps_arg(stamps: torch.Tensor, device):
    _need(stamps, "stamps", torch.int64, device)
    if stamps.numel() != 2 * _lib.MOE_NUM_STAGES:
        raise ValueError(f"stamps must hold {2 * _lib.MOE_NUM_STAGES} entries")
    return ctypes.c_void_p(stamps.data_ptr())


def stage_spans(stamps) -> list:
    """Host decoding of stamped calls: for each row of an int64 [n, 16]
    tensor (or one row), a dict stage name -> (begin_ns, end_ns) for the
    stages that ran (end >= begin), in the unsigned global-timer scale."""
    import numpy as np
    a = np.asarray(stamps.cpu() if isinstance(stamps, torch.Tensor) else stamps).astype(np.int64).view(np.uint64)
    a = a.reshape(-1, 2 * _lib.MOE_NUM_STAGES)
    n = _lib.MOE_NUM_STAGES
    out = []
    for row in a:
        out.append({name: (int(row[i]), int(row[n + i])) for i, name in enumerate(_lib.STAGES)
                    if row[n + i] != 0 and row[i] != np.iinfo(np.uint64).max and row[n + i] >= row[i]})
    return out


def moe_forward_stamped(x, Wg, W1, W3, W2, K: int, stamps, y=None, workspace: Workspace | None = None,
                        flags: int = 0, stream=None):
    """moe_forward whose kernels also write their begin/end global-timer
    times into ``stamps`` (one row of new_stamps; decode with stage_spans)."""
    dev = x.device
    T, d = x.shape
    E, _, f = W1.shape
    if y is None:
        y = torch.empty_like(x)
    if workspace is None:
        workspace = Workspace(T, d, f, E, K, x.dtype, dev)
    rc = _lib.load().moe_forward_stamped(_ptr(x), _ptr(Wg), _ptr(W1), _ptr(W3), _ptr(W2), _ptr(y), T, d, f, E, K,
                                         _dtype_code(x), workspace.ptr(), workspace.nbytes, flags,
                                         _stream_ptr(stream, dev), _stamps_arg(stamps, dev))
    _lib.check("moe_forward_stamped", rc)
    return y


def moe_block_forward_stamped(h, Wg, W1, W3, W2, K: int, stamps, eps: float = 1e-5,
                              workspace: Workspace | None = None, flags: int = 0, stream=None):
    """moe_block_forward with stage timestamps (see moe_forward_stamped)."""
    dev = h.device
    T, d = h.shape
    E, _, f = W1.shape
    if workspace is None:
        workspace = Workspace(T, d, f, E, K, h.dtype, dev)
    rc = _lib.load().moe_block_forward_stamped(_ptr(h), _ptr(Wg), _ptr(W1), _ptr(W3), _ptr(W2), T, d, f, E, K,
                                               _dtype_code(h), float(eps), workspace.ptr(), workspace.nbytes, flags,
                                               _stream_ptr(stream, dev), _stamps_arg(stamps, dev))
    _lib.check("moe_block_forward_stamped", rc)
    return h


def moe_forward_host(x_host, y_host, Wg, W1, W3, W2, K: int = 2, x_dev=None, y_dev=None,
                     workspace: Workspace | None = None, stream=None):
    """End-to-end call on host buffers: copy x (pinned host) to the device,
    run the layer, copy y back.  Weights are device-resident."""
    dev = W1.device
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    if x_dev is None:
        x_dev = torch.empty(x_host.shape, dtype=x_host.dtype, device=dev)
    if y_dev is None:
        y_dev = torch.empty_like(x_dev)
    with torch.cuda.stream(s):
        x_dev.copy_(x_host, non_blocking=True)
        moe_forward(x_dev, Wg, W1, W3, W2, K, y=y_dev, workspace=workspace, stream=s)
        y_host.copy_(y_dev, non_blocking=True)
    return y_host


def quantize_weights_fp8(W, stream=None):
    """e4m3 codes of an expert bank: W [E, K, N] bf16 -> (Wq, scales [E, N]
    fp32), one scale per output column (scale = max |column| / 448).  Wq is
    float8_e4m3fn [E, ceil(N/128), ceil(K/128), 128, 128]: 128 x 128 tiles,
    Wq[e, n // 128, k // 128, n % 128, k % 128] = code of W[e, k, n], zero past
    N or K."""
    _need(W, "W", torch.bfloat16)
    E, Kd, N = W.shape
    Wq = torch.empty((E, (N + 127) // 128, (Kd + 127) // 128, 128, 128), dtype=torch.float8_e4m3fn,
                     device=W.device)
    scales = torch.empty((E, N), dtype=torch.float32, device=W.device)
    rc = _lib.load().moe_quantize_weights_fp8(_ptr(W), E, Kd, N, _ptr(Wq), _ptr(scales), _stream_ptr(stream, W.device))
    _lib.check("moe_quantize_weights_fp8", rc)
    return Wq, scales


def _fp8_args(x, Wg, W1q, s1, W3q, s3, W2q, s2, y):
    dev = x.device
    _need(x, "x", torch.bfloat16, dev)
    _need(Wg, "Wg", torch.bfloat16, dev)
    for t, n in ((W1q, "W1q"), (W3q, "W3q"), (W2q, "W2q")):
        _need(t, n, torch.float8_e4m3fn, dev)
    for t, n in ((s1, "s1"), (s3, "s3"), (s2, "s2")):
        _need(t, n, torch.float32, dev)
    T, d = x.shape
    E, f = s1.shape
    tiles = lambda n, k: (E, (n + 127) // 128, (k + 127) // 128, 128, 128)
    if (Wg.shape != (d, E) or W1q.shape != tiles(f, d) or W3q.shape != tiles(f, d) or W2q.shape != tiles(d, f)
            or s3.shape != (E, f) or s2.shape != (E, d)):
        raise ValueError("shape mismatch: x [T,d], Wg [d,E], s1/s3 [E,f], s2 [E,d], W1q/W3q tiles over (f, d), "
                         "W2q tiles over (d, f) (quantize_weights_fp8)")
    if y is None:
        y = torch.empty_like(x)
    else:
        _need(y, "y", torch.bfloat16, dev)
    return T, d, f, E, y


def moe_forward_fp8(x, Wg, W1q, s1, W3q, s3, W2q, s2, K: int = 2, y=None, workspace: Workspace | None = None,
                    flags: int = 0, stream=None):
    """The layer with e4m3 expert weights (codes and scales from
    quantize_weights_fp8); x, Wg, y bf16.  Returns y [T, d]."""
    T, d, f, E, y = _fp8_args(x, Wg, W1q, s1, W3q, s3, W2q, s2, y)
    if workspace is None:
        workspace = Workspace(T, d, f, E, K, torch.float8_e4m3fn, x.device)
    rc = _lib.load().moe_forward_fp8(_ptr(x), _ptr(Wg), _ptr(W1q), _ptr(s1), _ptr(W3q), _ptr(s3), _ptr(W2q), _ptr(s2),
                                     _ptr(y), T, d, f, E, K, workspace.ptr(), workspace.nbytes, flags,
                                     _stream_ptr(stream, x.device))
    _lib.check("moe_forward_fp8", rc)
    return y


def moe_forward_fp8_stamped(x, Wg, W1q, s1, W3q, s3, W2q, s2, K: int, stamps, y=None,
                            workspace: Workspace | None = None, flags: int = 0, stream=None):
    """moe_forward_fp8 with stage timestamps (see moe_forward_stamped)."""
    T, d, f, E, y = _fp8_args(x, Wg, W1q, s1, W3q, s3, W2q, s2, y)
    if workspace is None:
        workspace = Workspace(T, d, f, E, K, torch.float8_e4m3fn, x.device)
    rc = _lib.load().moe_forward_fp8_stamped(_ptr(x), _ptr(Wg), _ptr(W1q), _ptr(s1), _ptr(W3q), _ptr(s3),
                                             _ptr(W2q), _ptr(s2), _ptr(y), T, d, f, E, K, workspace.ptr(),
                                             workspace.nbytes, flags, _stream_ptr(stream, x.device),
                                             _stamps_arg(stamps, x.device))
    _lib.check("moe_forward_fp8_stamped", rc)
    return y


class TrainWorkspace(Workspace):
    """A workspace sized by moe_train_workspace_bytes: the forward's buffers
    plus what moe_forward_train keeps for moe_backward (bf16 only)."""

    def __init__(self, T, d, f, E, K, dtype=torch.bfloat16, device=None):
        self.nbytes = _lib.load().moe_train_workspace_bytes(T, d, f, E, K, _DTYPES.get(dtype, -1))
        if self.nbytes == 0:
            raise ValueError(f"unsupported training sizes T={T} d={d} f={f} E={E} K={K} dtype={dtype} "
                             "(bf16, d and f multiples of 64)")
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device or "cuda")
        self.key = (T, d, f, E, K, dtype)


def _layer_args(x, Wg, W1, W3, W2):
    dev, dt = x.device, x.dtype
    for t, n in ((x, "x"), (Wg, "Wg"), (W1, "W1"), (W3, "W3"), (W2, "W2")):
        _need(t, n, dt, dev)
    T, d = x.shape
    E, d1, f = W1.shape
    if Wg.shape != (d, E) or W3.shape != (E, d, f) or W2.shape != (E, f, d) or d1 != d:
        raise ValueError("shape mismatch: x [T,d], Wg [d,E], W1/W3 [E,d,f], W2 [E,f,d]")
    return T, d, f, E


def moe_forward_train(x, Wg, W1, W3, W2, K: int, workspace: TrainWorkspace, y=None, flags: int = 0, stream=None):
    """moe_forward that keeps in ``workspace`` what moe_backward needs; returns y."""
    T, d, f, E = _layer_args(x, Wg, W1, W3, W2)
    if y is None:
        y = torch.empty_like(x)
    else:
        _need(y, "y", x.dtype, x.device)
    rc = _lib.load().moe_forward_train(_ptr(x), _ptr(Wg), _ptr(W1), _ptr(W3), _ptr(W2), _ptr(y), T, d, f, E, K,
                                       _dtype_code(x), workspace.ptr(), workspace.nbytes, flags,
                                       _stream_ptr(stream, x.device))
    _lib.check("moe_forward_train", rc)
    return y


class LayerGrads(tuple):
    """(dx, dWg, dW1, dW3, dW2), fp32."""
    __slots__ = ()

    def __new__(cls, dx, dWg, dW1, dW3, dW2):
        return super().__new__(cls, (dx, dWg, dW1, dW3, dW2))

    dx = property(lambda s: s[0])
    dWg = property(lambda s: s[1])
    dW1 = property(lambda s: s[2])
    dW3 = property(lambda s: s[3])
    dW2 = property(lambda s: s[4])


def moe_backward(x, Wg, W1, W3, W2, dy, K: int, workspace: TrainWorkspace, grads: LayerGrads | None = None,
                 flags: int = 0, stream=None) -> LayerGrads:
    """Gradients of the layer (fp32) from the state the last moe_forward_train
    on ``workspace`` left; ``grads`` are written (or, with MOE_ACCUMULATE,
    added to) in place if given."""
    T, d, f, E = _layer_args(x, Wg, W1, W3, W2)
    _need(dy, "dy", x.dtype, x.device)
    if dy.shape != x.shape:
        raise ValueError("dy must have the shape of x")
    if grads is None:
        z = dict(dtype=torch.float32, device=x.device)
        grads = LayerGrads(torch.empty(T, d, **z), torch.empty(d, E, **z), torch.empty(E, d, f, **z),
                           torch.empty(E, d, f, **z), torch.empty(E, f, d, **z))
    shapes = ((T, d), (d, E), (E, d, f), (E, d, f), (E, f, d))
    for g, shp, n in zip(grads, shapes, ("dx", "dWg", "dW1", "dW3", "dW2")):
        _need(g, n, torch.float32, x.device)
        if tuple(g.shape) != shp:
            raise ValueError(f"{n} must have shape {shp}")
    rc = _lib.load().moe_backward(_ptr(x), _ptr(Wg), _ptr(W1), _ptr(W3), _ptr(W2), _ptr(dy), *map(_ptr, grads),
                                  T, d, f, E, K, _dtype_code(x), workspace.ptr(), workspace.nbytes, flags,
                                  _stream_ptr(stream, x.device))
    _lib.check("moe_backward", rc)
    return grads


class ExpertCache:
    """Decode-time expert offload: the expert banks in pinned host memory, C
    device slots, least-recently-used replacement (moe_forward_cached).

    ``W1, W3, W2`` are the full banks (any device; copied to pinned host
    memory once).  ``forward`` runs one batch; ``state`` exposes the policy's
    counters (hits, misses, bytes_loaded) and maps."""

    def __init__(self, W1, W3, W2, C: int, device=None):
        if W1.dtype != torch.bfloat16:
            raise TypeError("the expert cache holds bf16 banks")
        E, d, f = W1.shape
        self.E, self.d, self.f, self.C = E, d, f, C
        self.device = torch.device(device) if device is not None else torch.device("cuda")
        self.host = [w.detach().to("cpu").contiguous().pin_memory() for w in (W1, W3, W2)]
        self.slots = [torch.empty((C,) + tuple(w.shape[1:]), dtype=w.dtype, device=self.device)
                      for w in (W1, W3, W2)]
        self.state = _lib.ExpertCacheState()
        _lib.check("moe_expert_cache_init", _lib.load().moe_expert_cache_init(ctypes.byref(self.state), E, C))

    def forward(self, x, Wg, K: int, y=None, workspace: Workspace | None = None, flags: int = 0, stream=None):
        _need(x, "x", torch.bfloat16, self.device)
        _need(Wg, "Wg", torch.bfloat16, self.device)
        T, d = x.shape
        if d != self.d or Wg.shape != (d, self.E):
            raise ValueError("shape mismatch: x [T,d], Wg [d,E]")
        if y is None:
            y = torch.empty_like(x)
        if workspace is None:
            workspace = Workspace(T, d, self.f, self.E, K, torch.bfloat16, self.device)
        rc = _lib.load().moe_forward_cached(_ptr(x), _ptr(Wg), *map(_ptr, self.host), *map(_ptr, self.slots),
                                            ctypes.byref(self.state), _ptr(y), T, d, self.f, self.E, K, MOE_BF16,
                                            workspace.ptr(), workspace.nbytes, flags, _stream_ptr(stream, x.device))
        _lib.check("moe_forward_cached", rc)
        return y


class HostPipeline:
    """moe_forward on batches held in pinned host memory, with the copy of the
    next batch in and of the previous result out overlapping the current
    batch's layer: two device (x, y) buffer pairs, a copy-in stream, a compute
    stream and a copy-out stream ordered by events.  ``submit`` only enqueues;
    ``synchronize`` waits for every submitted batch (read ``y_host`` after it).
    All batches have the shape and dtype given here."""

    def __init__(self, Wg, W1, W3, W2, K: int, T: int, device=None, workspace: Workspace | None = None,
                 fp8_weights=None):
        self.dev = W1.device if device is None else device
        E, d, f = W1.shape
        self.w = (Wg, W1, W3, W2)
        self.q8 = fp8_weights        # (W1q, s1, W3q, s3, W2q, s2): run moe_forward_fp8 instead
        self.K = K
        self.ws = workspace or Workspace(T, d, f, E, K, torch.float8_e4m3fn if fp8_weights else W1.dtype, self.dev)
        self.x = [torch.empty((T, d), dtype=W1.dtype, device=self.dev) for _ in range(2)]
        self.y = [torch.empty((T, d), dtype=W1.dtype, device=self.dev) for _ in range(2)]
        self.s_in = torch.cuda.Stream(self.dev)
        self.s_run = torch.cuda.Stream(self.dev)
        self.s_out = torch.cuda.Stream(self.dev)
        self.in_done = [torch.cuda.Event() for _ in range(2)]
        self.run_done = [torch.cuda.Event() for _ in range(2)]
        self.out_done = [torch.cuda.Event() for _ in range(2)]
        self.n = 0

    def submit(self, x_host, y_host):
        b = self.n & 1
        if self.n >= 2:
            self.s_in.wait_event(self.run_done[b])    # x[b] was read by the layer two batches ago
        with torch.cuda.stream(self.s_in):
            self.x[b].copy_(x_host, non_blocking=True)
            self.in_done[b].record(self.s_in)
        self.s_run.wait_event(self.in_done[b])
        if self.n >= 2:
            self.s_run.wait_event(self.out_done[b])   # y[b] was copied out two batches ago
        if self.q8 is not None:
            moe_forward_fp8(self.x[b], self.w[0], *self.q8, self.K, y=self.y[b], workspace=self.ws, stream=self.s_run)
        else:
            moe_forward(self.x[b], *self.w, self.K, y=self.y[b], workspace=self.ws, stream=self.s_run)
        self.run_done[b].record(self.s_run)
        self.s_out.wait_event(self.run_done[b])
        with torch.cuda.stream(self.s_out):
            y_host.copy_(self.y[b], non_blocking=True)
            self.out_done[b].record(self.s_out)
        self.n += 1

    def synchronize(self):
        for s in (self.s_in, self.s_run, self.s_out):
            s.synchronize()


def moe_route(x, Wg, K: int = 2, workspace: Workspace | None = None, stream=None):
    """Routing only: returns (idx [T,K] int32, gate [T,K] fp32, perm_tok [T*K] int32,
    offsets [E+1] int32, pos [T,K] int32), unpadded grouped order."""
    dev = x.device
    _need(x, "x", None, dev)
    _need(Wg, "Wg", x.dtype, dev)
    T, d = x.shape
    E = Wg.shape[1]
    idx = torch.empty((T, K), dtype=torch.int32, device=dev)
    gate = torch.empty((T, K), dtype=torch.float32, device=dev)
    perm = torch.empty((T * K,), dtype=torch.int32, device=dev)
    offsets = torch.empty((E + 1,), dtype=torch.int32, device=dev)
    pos = torch.empty((T, K), dtype=torch.int32, device=dev)
    f_min = 8 if x.dtype == torch.bfloat16 else 4
    if workspace is None:
        workspace = Workspace(T, d, f_min, E, K, x.dtype, dev)
    rc = _lib.load().moe_route(_ptr(x), _ptr(Wg), T, d, E, K, _dtype_code(x), _ptr(idx), _ptr(gate), _ptr(perm),
                               _ptr(offsets), _ptr(pos), workspace.ptr(), workspace.nbytes,
                               _stream_ptr(stream, dev))
    _lib.check("moe_route", rc)
    return idx, gate, perm, offsets, pos


def moe_rmsnorm(x, eps: float = 1e-5, out=None, stream=None):
    """out = x / sqrt(mean(x^2) + eps) per row (unit gain); in place if out is x."""
    _need(x, "x")
    if out is None:
        out = torch.empty_like(x)
    else:
        _need(out, "out", x.dtype, x.device)
    T, d = x.shape
    rc = _lib.load().moe_rmsnorm(_ptr(x), _ptr(out), T, d, float(eps), _dtype_code(x),
                                 _stream_ptr(stream, x.device))
    _lib.check("moe_rmsnorm", rc)
    return out


def moe_read_status(workspace: Workspace, stream=None) -> int:
    """Synchronise the stream and return the device status word (0 = ok)."""
    return int(_lib.load().moe_read_status(workspace.ptr(), _stream_ptr(stream, workspace.buf.device)))
